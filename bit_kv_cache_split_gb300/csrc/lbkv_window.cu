// lbkv_window.cu -- attention of each (sequence, KV head) pair's queries over its
// full-precision bf16 window (the most recent tokens, kept unquantized after the
// cached ones), written as one partial (m, l, O) per pair; the decode kernel merges
// it with the cached tokens' partials. A rotated cache keeps its window rotated too, so
// the partial is in the same (rotated) basis as the cached tokens' partials.
#include "lbkv_internal.h"

namespace lbkv {

// One CTA per pair. The window's K rows go to shared memory (rows padded by one word, so
// that the 32 rows a warp reads at once sit in 32 different banks); then every (query,
// token) score is one thread's dot product, each query's softmax one warp's reduction, and
// every output channel of a query one thread's weighted sum over the V rows. The V rows
// are loaded into registers at the start (their latency overlaps the scores) and moved into
// the K rows' shared memory once the scores are done.
constexpr int kWinThreads = 32 * kWinWarps;
constexpr int kWinKStride = kHeadDim + 2;  // bf16 per shared K row

__global__ void __launch_bounds__(kWinThreads, 1) window_partial_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int D = kHeadDim;
  constexpr unsigned FULLMASK = 0xffffffffu;
  __shared__ __align__(16) __nv_bfloat16 sK[kWinMax * kWinKStride];
  __shared__ float sQ[kMaxHq * D];
  __shared__ float sS[kMaxHq * kWinMax];  // scores (log2 units), then weights
  __shared__ float sM[kMaxHq], sL[kMaxHq];

  // the decode kernel may start launching now: it waits for this grid only where it reads
  // the window partials
  grid_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kvh = blockIdx.x, b = blockIdx.y;
  const int hq = p.hq;
  const int u = b * p.Hkv + kvh;
  const int W = min(max(p.win_lens[b], 0), p.win_cap);
  const size_t wbase = (size_t)(u >> p.kv_shift) * p.win_cap;  // the pair's cached KV head
  for (int idx = threadIdx.x; idx < hq * D; idx += kWinThreads)
    sQ[idx] = __bfloat162float(p.q[((size_t)b * p.Hq + kvh * hq) * D + idx]);
  for (int e = threadIdx.x; e < W * (D / 2); e += kWinThreads) {
    const int t = e / (D / 2), d2 = e % (D / 2);
    reinterpret_cast<uint32_t*>(sK + t * kWinKStride)[d2] =
        reinterpret_cast<const uint32_t*>(p.k_win + (wbase + t) * D)[d2];
  }
  constexpr int kVWords = kWinMax * (D / 2) / kWinThreads;  // V words (two channels) per thread
  uint32_t vreg[kVWords];
#pragma unroll
  for (int j = 0; j < kVWords; ++j) {
    const int e = threadIdx.x + j * kWinThreads, t = e / (D / 2), d2 = e % (D / 2);
    vreg[j] = (t < W) ? reinterpret_cast<const uint32_t*>(p.v_win + (wbase + t) * D)[d2] : 0u;
  }
  __syncthreads();
  if (p.rotation & 1) {  // window keys stored rotated like the cache's: the scores take H q
    for (int i = warp; i < hq; i += kWinWarps) {
      float v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = sQ[i * D + 4 * lane + e];
      hadamard128(v, lane);
#pragma unroll
      for (int e = 0; e < 4; ++e) sQ[i * D + 4 * lane + e] = v[e];
    }
    __syncthreads();
  }

  // scores: thread per (query i, token t)
  for (int e = threadIdx.x; e < hq * W; e += kWinThreads) {
    const int i = e / W, t = e % W;
    const uint32_t* krow = reinterpret_cast<const uint32_t*>(sK + t * kWinKStride);
    const float* qrow = sQ + i * D;
    float acc = 0.f;
#pragma unroll 8
    for (int d2 = 0; d2 < D / 2; ++d2) {
      const float2 k2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(krow + d2));
      acc = fmaf(qrow[2 * d2], k2.x, acc);
      acc = fmaf(qrow[2 * d2 + 1], k2.y, acc);
    }
    sS[i * kWinMax + t] = acc * p.sl2;
  }
  __syncthreads();  // the K rows are read: the V rows take their place
#pragma unroll
  for (int j = 0; j < kVWords; ++j) {
    const int e = threadIdx.x + j * kWinThreads, t = e / (D / 2), d2 = e % (D / 2);
    if (t < W) reinterpret_cast<uint32_t*>(sK + t * kWinKStride)[d2] = vreg[j];
  }

  // per query: maximum, weights 2^(s - m), their sum (warp i)
  for (int i = warp; i < hq; i += kWinWarps) {
    float m = -INFINITY;
    for (int t = lane; t < W; t += 32) m = fmaxf(m, sS[i * kWinMax + t]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULLMASK, m, o));
    float l = 0.f;
    for (int t = lane; t < W; t += 32) {
      const float w = fast_exp2(sS[i * kWinMax + t] - m);
      sS[i * kWinMax + t] = w;
      l += w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(FULLMASK, l, o);
    if (lane == 0) {
      sM[i] = m;
      sL[i] = l;
    }
  }
  __syncthreads();

  // unnormalised output: thread per (query i, channel d)
  for (int e = threadIdx.x; e < hq * D; e += kWinThreads) {
    const int i = e / D, d = e % D;
    const float* w = sS + i * kWinMax;
    const __nv_bfloat16* vcol = sK + d;  // the V rows, same padded stride
    float acc = 0.f;
#pragma unroll 8
    for (int t = 0; t < W; ++t) acc = fmaf(w[t], __bfloat162float(vcol[t * kWinKStride]), acc);
    const size_t prow = (size_t)u * hq + i;
    p.win_o[prow * D + d] = acc;
    if (d == 0) p.win_ml[prow] = make_float2(sM[i], sL[i]);
  }
}

int launch_window_partial(const DecodeParams& p, cudaStream_t stream) {
  dim3 grid((unsigned)p.Hkv, (unsigned)p.B);
  window_partial_kernel<<<grid, kWinThreads, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace lbkv
