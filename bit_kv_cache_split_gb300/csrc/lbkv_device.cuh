// lbkv_device.cuh -- sm_103a building blocks: mbarriers with bounded waits, bulk
// copies into shared memory, the fp16 tensor-core product and the bit tricks that
// turn packed 2-/4-bit codes into exact fp16 operands.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lbkv {

// Device status codes written to the workspace status word instead of hanging.
enum : int32_t {
  kStatusConsumerTimeout = 1,  // a warp waited ~1 s for its own bulk copies
  kStatusDrainTimeout = 3,     // after that, the copies still in flight did not land
  kStatusAppendFull = 4,       // an appended token did not fit (capacity or window state)
  kStatusBadPage = 5,          // a page-table entry outside the page pool (read as page 0)
};

// Normalized Hadamard rotation of a 128-channel row held by a warp, 4 channels per lane
// (lane l: channels 4l .. 4l + 3), in place. The butterflies run in stages of span 1, 2,
// 4, ..., 64; in each, the lower channel of a pair takes a + b and the upper a - b (a the
// lower's value, b the upper's); then every channel is scaled by fp32(1/sqrt(128)). Each
// step is one IEEE single-precision operation, so the result is the same bits whatever the
// hardware. The matrix is symmetric and orthogonal: applying it twice gives the row back.
__device__ __forceinline__ void hadamard128(float (&v)[4], int lane) {
  float a, b;
  a = v[0], b = v[1], v[0] = __fadd_rn(a, b), v[1] = __fsub_rn(a, b);  // span 1
  a = v[2], b = v[3], v[2] = __fadd_rn(a, b), v[3] = __fsub_rn(a, b);
  a = v[0], b = v[2], v[0] = __fadd_rn(a, b), v[2] = __fsub_rn(a, b);  // span 2
  a = v[1], b = v[3], v[1] = __fadd_rn(a, b), v[3] = __fsub_rn(a, b);
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {  // span 4m: the partner channel is in lane l ^ m
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float o = __shfl_xor_sync(0xffffffffu, v[u], m);
      v[u] = upper ? __fsub_rn(o, v[u]) : __fadd_rn(v[u], o);
    }
  }
  const float c = __uint_as_float(0x3db504f3u);  // 1/sqrt(128) rounded to fp32
#pragma unroll
  for (int u = 0; u < 4; ++u) v[u] = __fmul_rn(v[u], c);
}

// Channels 4 lane .. 4 lane + 3 of a bf16 row, as fp32.
__device__ __forceinline__ void load_row4(const __nv_bfloat16* row, int lane, float (&v)[4]) {
  const uint2 raw = reinterpret_cast<const uint2*>(row)[lane];
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
  const float2 a = __bfloat1622float2(h[0]), c = __bfloat1622float2(h[1]);
  v[0] = a.x, v[1] = a.y, v[2] = c.x, v[3] = c.y;
}

// The same four channels rounded to bf16 (nearest, ties to even) into a bf16 row.
__device__ __forceinline__ void store_row4(__nv_bfloat16* row, int lane, const float (&v)[4]) {
  __nv_bfloat162 h[2];
  h[0] = __floats2bfloat162_rn(v[0], v[1]);
  h[1] = __floats2bfloat162_rn(v[2], v[3]);
  reinterpret_cast<uint2*>(row)[lane] = *reinterpret_cast<const uint2*>(h);
}

// Where token t of KV head kvh (cache unit `unit` = b * hkv + kvh) is stored: its row of
// codes (and of token-wise scales) and its block of channel-wise scales (one block per
// `g` tokens). Contiguous cache (page_tokens == 0): [B][Hkv][T_cap] rows. Paged cache:
// row t mod page_tokens of `page`, the page-table entry of t, in a pool of
// [num_pages][Hkv][page_tokens] rows.
struct KvAddr {
  size_t row, block;
};
__device__ __forceinline__ KvAddr kv_addr(int page_tokens, int page, size_t unit, int kvh, int hkv, int T_cap, int g,
                                          size_t t) {
  KvAddr a;
  if (page_tokens == 0) {
    a.row = unit * T_cap + t;
    a.block = unit * (size_t)(T_cap / g) + t / g;
  } else {
    const size_t pu = (size_t)page * hkv + kvh, off = t % (size_t)page_tokens;
    a.row = pu * page_tokens + off;
    a.block = pu * (size_t)(page_tokens / g) + off / g;
  }
  return a;
}

// The page-table entry of token t of sequence b (table [B][max_pages]), or -1 when it
// lies outside the pool of num_pages pages.
__device__ __forceinline__ int kv_page(const int32_t* table, int max_pages, int num_pages, int page_tokens, int b,
                                       size_t t) {
  const int page = __ldg(table + (size_t)b * max_pages + t / page_tokens);
  return (page < 0 || page >= num_pages) ? -1 : page;
}

// A bounded wait gives up after this many nanoseconds of wall time.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Slow path of a bounded wait: polls until the phase completes or `limit_ns` of wall
// time has passed; then records `code` in the status word and returns false.
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, int32_t* status, int32_t code,
                                                   uint64_t limit_ns) {
  const uint64_t t0 = global_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) {
      atomicExch(status, code);
      return false;
    }
  }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int32_t* status, int32_t code,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, status, code, limit_ns);
}

// Bulk (non-tensor) copy global -> shared, completing on an mbarrier.
// Both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// L2 policy for data read exactly once (the streamed cache).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Orders this thread's earlier generic-proxy shared-memory accesses before its later
// async-proxy ones (a bulk copy refilling a buffer that was just read).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------- tensor-core product
// D[16x8] += A[16x16] * B[16x8], fp16 inputs, fp32 accumulators.
// Fragments (lane = 4*g + c): A reg0 row g k 2c,2c+1; reg1 row g+8 k 2c,2c+1;
// reg2 row g k 2c+8,2c+9; reg3 row g+8 k 2c+8,2c+9 (low half = lower k);
// B reg0 k 2c,2c+1 col g; reg1 k 2c+8,2c+9 col g; D d0,d1 row g cols 2c,2c+1,
// d2,d3 row g+8 cols 2c,2c+1.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A * B + C with a separate starting value C (the first product of a chain).
__device__ __forceinline__ void mma_f16_c(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1, float c0, float c1, float c2, float c3) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2), "f"(c3));
}

// e4m3 image of x (round to nearest even, saturating to +-448) in the low byte, and
// the value of an e4m3 byte.
__device__ __forceinline__ uint32_t e4m3_rn(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.f), "f"(x));
  return r & 0xffu;
}
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)b));
  return __half2float(__ushort_as_half((unsigned short)(r & 0xffffu)));
}

__device__ __forceinline__ uint32_t f16x2_from(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ------------------------------------------------------------ conversions
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Programmatic dependent launch: a grid lets its dependent grid start launching
// (launch_dependents), and a dependent grid's thread waits until its prerequisite grid has
// completed with its memory visible (wait; it returns at once when the grid was launched
// without a prerequisite).
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Thread-block clusters: this CTA's rank, the cluster's CTA count and its index, the
// shared-memory address of the same variable in CTA `rank` of the cluster, loads from it,
// and the cluster-wide barrier (release / acquire: the shared-memory writes before it are
// seen by every CTA after it).
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 2^e for integer e in [-126, 127], exactly.
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((e + 127) << 23); }

// floor(log2(x)) for a positive normal float.
__device__ __forceinline__ int ilog2f(float x) { return ((__float_as_int(x) >> 23) & 0xff) - 127; }

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace lbkv
