// tc_rates.cu -- microbenchmark of the 5th-generation tensor-core operations the decode
// kernels would build on (GB300, sm_103a), one CTA of 16 warps per SM on every SM:
//   mma   : tcgen05.mma kind::f8f6f4 (A e4m3 in tensor memory, B e4m3 in shared memory, fp32
//           accumulators), M x N x 32 per product (M = 128, and M = 64 at N = 16), `iters` back-to-back products per warp and
//           one commit; cycles per product per warp (issue rate) and per SM (throughput);
//   st    : tcgen05.st 32x32b.x32 (a warp's 32 lanes x 32 columns) + wait::st;
//   ld    : tcgen05.ld 32x32b.x16 + wait::ld.
// Prints one JSON object per measurement. Every tensor-memory and shared-memory address stays
// inside the CTA's allocation; the one wait is bounded.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

namespace {

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

constexpr int kCols = 512;

__global__ void rates_kernel(int op, int M, int N, int iters, int nw, long long* out, int* err, float* sink) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint32_t tbase;
  __shared__ __align__(8) uint64_t mbar[16];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < 32768; i += blockDim.x) smem[i] = 0x38;  // e4m3 1.0
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&tbase)), "r"(kCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (threadIdx.x < 16) asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(&mbar[threadIdx.x])), "r"(1));
  asm volatile("fence.mbarrier_init.release.cluster;");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  const uint32_t tb = tbase;
  float acc = 0.f;
  if (warp < nw) {
    long long t0 = clock64(), t1 = t0;
    if (op == 0) {
      // A: columns 0..31 (all lanes), D: 32 + warp * N (nw * N + 32 <= kCols)
      const uint32_t a_tm = tb, d_tm = tb + 32u + (uint32_t)(warp * N);
      const uint32_t idesc = (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
      if (lane == 0) {
        for (int it = 0; it < iters; ++it) {
          const uint64_t bd = smem_desc(su32(smem) + 256u * (it & 3), 128u, 1024u);
          asm volatile(
              "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}" ::"r"(
                  d_tm),
              "r"(a_tm + 8u * (it & 3)), "l"(bd), "r"(idesc), "r"((uint32_t)(it > 0)));
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(&mbar[warp])));
        uint32_t ok = 0;
        const long long w0 = clock64();
        while (!ok) {
          asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}"
                       : "=r"(ok)
                       : "r"(su32(&mbar[warp])), "r"(0));
          if (!ok && clock64() - w0 > 4000000000LL) {
            atomicExch(err, 1);
            break;
          }
        }
      }
      __syncwarp();
      t1 = clock64();
    } else {
      const uint32_t ta = tb + ((uint32_t)(32 * (warp & 3)) << 16) + 32u * (warp >> 2);  // columns < 128
      uint32_t r[32];
      for (int j = 0; j < 32; ++j) r[j] = lane * 7 + j;
      for (int it = 0; it < iters; ++it) {
        if (op == 1) {
          asm volatile(
              "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
              "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(ta),
              "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
              "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
              "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
              "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
              : "memory");
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          r[it & 31] += 1;
        } else {
          uint32_t v[16];
          asm volatile(
              "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
              : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
                "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
              : "r"(ta + 16u * (it & 1))
              : "memory");
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
          for (int j = 0; j < 16; ++j) acc += __uint_as_float(v[j]);
        }
      }
      t1 = clock64();
    }
    if (lane == 0) out[blockIdx.x * 16 + warp] = t1 - t0;
  }
  sink[blockIdx.x * blockDim.x + threadIdx.x] = acc;
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tb), "r"(kCols));
}

}  // namespace

int main() {
  long long* d_out = nullptr;
  int* d_err = nullptr;
  float* d_sink = nullptr;
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  cudaMalloc(&d_out, (size_t)sms * 16 * 8);
  cudaMalloc(&d_err, 4);
  cudaMalloc(&d_sink, (size_t)sms * 512 * 4);
  cudaFuncSetAttribute(rates_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 32768);
  long long* h = new long long[(size_t)sms * 16];
  auto run = [&](const char* name, int op, int M, int N, int iters, int nw) {
    cudaMemset(d_err, 0, 4);
    cudaMemset(d_out, 0, (size_t)sms * 16 * 8);
    rates_kernel<<<sms, 512, 32768>>>(op, M, N, iters, nw, d_out, d_err, d_sink);
    if (cudaDeviceSynchronize() != cudaSuccess) {
      printf("{\"op\": \"%s\", \"error\": \"launch\"}\n", name);
      return false;
    }
    int herr = 0;
    cudaMemcpy(&herr, d_err, 4, cudaMemcpyDeviceToHost);
    cudaMemcpy(h, d_out, (size_t)sms * 16 * 8, cudaMemcpyDeviceToHost);
    double mx = 0;
    for (int b = 0; b < sms; ++b)
      for (int w = 0; w < nw; ++w) mx = (double)h[b * 16 + w] > mx ? (double)h[b * 16 + w] : mx;
    printf("{\"op\": \"%s\", \"M\": %d, \"N\": %d, \"warps_per_sm\": %d, \"cycles_per_op_per_warp\": %.1f, "
           "\"cycles_per_op_per_sm\": %.2f, \"wait_gave_up\": %d}\n",
           name, M, N, nw, mx / iters, mx / iters / nw, herr);
    return true;
  };
  for (int N : {16, 32, 64, 128, 256})
    for (int nw : {1, 4, 16})
      if (32 + nw * N <= kCols && !run("tcgen05.mma f8f6f4 A:tmem B:smem", 0, 128, N, 256, nw)) return 1;
  for (int nw : {1, 4, 16})  // M = 64: the same rows of tensor memory, half of them used
    if (!run("tcgen05.mma f8f6f4 A:tmem B:smem", 0, 64, 16, 256, nw)) return 1;
  for (int nw : {1, 4, 16})
    if (!run("tcgen05.st 32x32b.x32 + wait", 1, 0, 0, 1000, nw)) return 1;
  for (int nw : {1, 4, 16})
    if (!run("tcgen05.ld 32x32b.x16 + wait", 2, 0, 0, 1000, nw)) return 1;
  delete[] h;
  return 0;
}
