// lbkv_window.cu -- attention of each (sequence, KV head) pair's queries over its
// full-precision bf16 window (the most recent tokens, kept unquantized after the
// cached ones), written as one partial (m, l, O) per pair; the decode kernel merges
// it with the cached tokens' partials. A rotated cache keeps its window rotated too, so
// the partial is in the same (rotated) basis as the cached tokens' partials.
#include "lbkv_internal.h"

namespace lbkv {

__global__ void __launch_bounds__(32 * kWinWarps, 1) window_partial_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int D = kHeadDim;
  constexpr unsigned FULLMASK = 0xffffffffu;
  __shared__ float sQ[kMaxHq * D];
  __shared__ float sM[kWinWarps][kMaxHq];
  __shared__ float sL[kWinWarps][kMaxHq];
  __shared__ float sO[kWinWarps][kMaxHq][D];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kvh = blockIdx.x, b = blockIdx.y;
  const int hq = p.hq;
  const int u = b * p.Hkv + kvh;
  for (int idx = threadIdx.x; idx < hq * D; idx += 32 * kWinWarps)
    sQ[idx] = __bfloat162float(p.q[((size_t)b * p.Hq + kvh * hq) * D + idx]);
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

  // warp w scores tokens w, w + W, ...; lane holds channels 4 lane .. 4 lane + 3
  const int W = min(max(p.win_lens[b], 0), p.win_cap);
  float m[kMaxHq], l[kMaxHq], o[kMaxHq][4];
#pragma unroll
  for (int i = 0; i < kMaxHq; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
    o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  }
  const size_t wbase = (size_t)(u >> p.kv_shift) * p.win_cap;  // the pair's cached KV head
  for (int t = warp; t < W; t += kWinWarps) {
    const uint2 kr = reinterpret_cast<const uint2*>(p.k_win + (wbase + t) * D)[lane];
    const uint2 vr = reinterpret_cast<const uint2*>(p.v_win + (wbase + t) * D)[lane];
    const __nv_bfloat162* kh = reinterpret_cast<const __nv_bfloat162*>(&kr);
    const __nv_bfloat162* vh = reinterpret_cast<const __nv_bfloat162*>(&vr);
    const float2 k01 = __bfloat1622float2(kh[0]), k23 = __bfloat1622float2(kh[1]);
    const float2 v01 = __bfloat1622float2(vh[0]), v23 = __bfloat1622float2(vh[1]);
#pragma unroll
    for (int i = 0; i < kMaxHq; ++i) {
      if (i >= hq) break;
      const float* qrow = sQ + i * D + 4 * lane;
      float d = qrow[0] * k01.x + qrow[1] * k01.y + qrow[2] * k23.x + qrow[3] * k23.y;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(FULLMASK, d, off);
      const float s = d * p.sl2;  // log2 units
      const float mn = fmaxf(m[i], s);
      const float a = fast_exp2(m[i] - mn);
      const float pr = fast_exp2(s - mn);
      m[i] = mn;
      l[i] = l[i] * a + pr;
      o[i][0] = o[i][0] * a + pr * v01.x;
      o[i][1] = o[i][1] * a + pr * v01.y;
      o[i][2] = o[i][2] * a + pr * v23.x;
      o[i][3] = o[i][3] * a + pr * v23.y;
    }
  }
#pragma unroll
  for (int i = 0; i < kMaxHq; ++i) {
    if (i >= hq) break;
    if (lane == 0) {
      sM[warp][i] = m[i];
      sL[warp][i] = l[i];
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) sO[warp][i][4 * lane + k] = o[i][k];
  }
  __syncthreads();

  // merge the warps into the window slot of the pair
  for (int idx = threadIdx.x; idx < hq * D; idx += 32 * kWinWarps) {
    const int i = idx / D, ch = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWinWarps; ++w) M = fmaxf(M, sM[w][i]);
    float acc = 0.f, lt = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWinWarps; ++w) {
        const float sc = (sM[w][i] == -INFINITY) ? 0.f : fast_exp2(sM[w][i] - M);
        acc = fmaf(sc, sO[w][i][ch], acc);
        lt = fmaf(sc, sL[w][i], lt);
      }
    }
    const size_t prow = (size_t)u * hq + i;
    p.win_o[prow * D + ch] = acc;
    if (ch == 0) p.win_ml[prow] = make_float2(M, lt);
  }
}

int launch_window_partial(const DecodeParams& p, cudaStream_t stream) {
  dim3 grid((unsigned)p.Hkv, (unsigned)p.B);
  window_partial_kernel<<<grid, 32 * kWinWarps, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace lbkv
