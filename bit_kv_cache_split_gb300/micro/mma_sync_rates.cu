// mma_sync_rates.cu -- microbenchmark of the warp-level tensor-core products (mma.sync) on this
// GPU, one CTA per SM on every SM with 4, 8 or 16 warps, each warp issuing 8 independent
// accumulator chains for `iters` rounds:
//   f16  : m16n8k16, fp16 A and B, fp32 accumulators (the decode kernel's product);
//   e4m3 : m16n8k32, e4m3 A and B, fp32 accumulators;
//   u8s8 : m16n8k32, unsigned 8-bit A, signed 8-bit B, int32 accumulators.
// The A operands change every round (an XOR with the round index), so that no conversion of
// them can be hoisted out of the loop. Prints one JSON object per measurement: SM cycles per
// product (all warps of the SM together) and per k-element of a product's 16 x 8 tile.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

namespace {

constexpr int kChains = 8;

template <int KIND>
__global__ void mma_rates_kernel(const uint32_t* in, float* out, int iters) {
  const int t = threadIdx.x;
  uint32_t a0 = in[t & 127], a1 = in[(t + 32) & 127], a2 = in[(t + 64) & 127], a3 = in[(t + 96) & 127];
  const uint32_t b0 = in[(t + 5) & 127], b1 = in[(t + 7) & 127];
  float cf[kChains][4];
  int ci[kChains][4];
#pragma unroll
  for (int j = 0; j < kChains; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) cf[j][e] = 0.f, ci[j][e] = 0;
  for (int i = 0; i < iters; ++i) {
    const uint32_t v = (uint32_t)i & 0x01010101u;
#pragma unroll
    for (int j = 0; j < kChains; ++j) {
      const uint32_t x0 = a0 ^ (v << j), x1 = a1 ^ (v << j);
      if (KIND == 0) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(cf[j][0]), "+f"(cf[j][1]), "+f"(cf[j][2]), "+f"(cf[j][3])
            : "r"(x0), "r"(x1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
      } else if (KIND == 1) {
        asm volatile(
            "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(cf[j][0]), "+f"(cf[j][1]), "+f"(cf[j][2]), "+f"(cf[j][3])
            : "r"(x0), "r"(x1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
      } else {
        asm volatile(
            "mma.sync.aligned.m16n8k32.row.col.s32.u8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+r"(ci[j][0]), "+r"(ci[j][1]), "+r"(ci[j][2]), "+r"(ci[j][3])
            : "r"(x0), "r"(x1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
      }
    }
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < kChains; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) s += cf[j][e] + (float)ci[j][e];
  out[(size_t)blockIdx.x * blockDim.x + t] = s;  // keeps the products live
}

}  // namespace

int main() {
  int sms = 0, clk_khz = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  cudaDeviceGetAttribute(&clk_khz, cudaDevAttrClockRate, 0);
  uint32_t* d_in = nullptr;
  float* d_out = nullptr;
  if (cudaMalloc(&d_in, 128 * sizeof(uint32_t)) != cudaSuccess ||
      cudaMalloc(&d_out, (size_t)sms * 512 * sizeof(float)) != cudaSuccess) {
    printf("{\"error\": \"allocation\"}\n");
    return 1;
  }
  cudaMemset(d_in, 0x11, 128 * sizeof(uint32_t));  // fp16 / e4m3 / 8-bit values of moderate size
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  const int iters = 4096;
  const char* names[3] = {"f16_m16n8k16", "e4m3_m16n8k32", "u8s8_m16n8k32"};
  const int kdim[3] = {16, 32, 32};
  int rc = 0;
  for (int kind = 0; kind < 3; ++kind) {
    for (int warps = 4; warps <= 16; warps *= 2) {
      float ms = 0.f;
      for (int rep = 0; rep < 2; ++rep) {  // the first launch warms up
        cudaEventRecord(e0);
        if (kind == 0)
          mma_rates_kernel<0><<<sms, warps * 32>>>(d_in, d_out, iters);
        else if (kind == 1)
          mma_rates_kernel<1><<<sms, warps * 32>>>(d_in, d_out, iters);
        else
          mma_rates_kernel<2><<<sms, warps * 32>>>(d_in, d_out, iters);
        cudaEventRecord(e1);
        cudaEventSynchronize(e1);
        cudaEventElapsedTime(&ms, e0, e1);
      }
      if (cudaGetLastError() != cudaSuccess) {
        printf("{\"op\": \"%s\", \"error\": \"launch\"}\n", names[kind]);
        rc = 1;
        continue;
      }
      const double products_per_sm = (double)warps * iters * kChains;
      const double cycles = (double)ms * 1e-3 * (double)clk_khz * 1e3;
      const double per_product = cycles / products_per_sm;
      printf("{\"op\": \"mma.sync %s\", \"warps_per_sm\": %d, \"ms\": %.3f, \"sm_cycles_per_product\": %.2f, "
             "\"sm_cycles_per_k_element\": %.3f}\n",
             names[kind], warps, ms, per_product, per_product / kdim[kind]);
    }
  }
  return rc;
}
