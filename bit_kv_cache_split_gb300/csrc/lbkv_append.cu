// lbkv_append.cu -- quantize-on-append: after a decode step, the new token's K and V
// go into the packed cache, quantized by the same arithmetic as the pack kernel
// (lbkv_quant.cuh). Serving needs this step before every decode call ("FOSCAR:
// Accelerating Decode Attention over 2- and 4-Bit KV Caches through Affine Folding",
// abstract: the SGLang integration); the append scheme below is this library's reading.
//
// Token-wise groups span channels of one token, so a new token is quantized at once
// and stored at position L_b. Channel-wise groups span g tokens of one channel, so the
// token waits in the bf16 window (attended like any window token) until g tokens have
// gathered; they are then quantized as one group at positions L_b .. L_b + g - 1 and the
// window empties. When either side is channel-wise, both sides take the window route,
// so that the cache and the window always hold the same tokens for K and V. A side
// stored rotated (lbkv_rotate) is rotated on the way in: the window holds it rotated too.
#include "lbkv_internal.h"
#include "lbkv_quant.cuh"

namespace lbkv {

// The new token row rotated by H and rounded to bf16, as stored (channels 4 lane .. +3).
__device__ __forceinline__ void rotate_bf16(float (&v)[4], int lane) {
  hadamard128(v, lane);
#pragma unroll
  for (int e = 0; e < 4; ++e) v[e] = __bfloat162float(__float2bfloat16_rn(v[e]));
}

constexpr int kAppendThreads = 512;  // 16 warps: the 2 Hkv rows of a token at once (Hkv <= 8)
constexpr int kAppendWarps = kAppendThreads / 32;

// Storage row and channel-group block of position L of KV head kvh of sequence b
// (`page`: the page-table entry of L in a paged cache).
__device__ __forceinline__ KvAddr append_addr(const AppendArgs& a, int page, int b, int kvh, int L) {
  return kv_addr(a.pg.page_tokens, page, (size_t)b * a.Hkv + kvh, kvh, a.Hkv, a.T_cap, a.group, L);
}

// One side (K or V) of the g window tokens of sequence b, all KV heads, into the cache
// at positions L .. L + g - 1 (one group: never split over two pages).
template <int BITS>
__device__ void flush_side(const AppendArgs& a, const __nv_bfloat16* win, int layout, uint8_t* codes, __half* scale,
                           __half* off, int b, int L, int page) {
  constexpr int RB = kHeadDim * BITS / 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = a.group;
  if (layout == 0) {
    // g token rows per KV head, one warp each
    for (int job = warp; job < a.Hkv * g; job += kAppendWarps) {
      const int kvh = job / g, t = job % g;
      const size_t unit = (size_t)b * a.Hkv + kvh;
      const size_t row = append_addr(a, page, b, kvh, L).row + t;
      const size_t si = row * (kHeadDim / g);
      quantize_token_row<BITS>(win + (unit * a.win_cap + t) * kHeadDim, g, codes + row * RB, scale + si, off + si,
                               lane);
    }
  } else {
    // one group per KV head: 128 threads, one channel each (4 KV heads at a time)
    for (int kvh = threadIdx.x / kHeadDim; kvh < a.Hkv; kvh += kAppendThreads / kHeadDim) {
      const int d = threadIdx.x % kHeadDim;
      const size_t unit = (size_t)b * a.Hkv + kvh;
      const KvAddr ad = append_addr(a, page, b, kvh, L);
      const size_t row0 = ad.row;
      const size_t si = ad.block * kHeadDim + d;
      quantize_channel_group<BITS>(win + unit * a.win_cap * kHeadDim, g, g, codes + row0 * RB, scale + si, off + si,
                                   d);
    }
  }
}

// One block per sequence b.
template <int BITS>
__global__ void __launch_bounds__(kAppendThreads) append_kernel(const __grid_constant__ AppendArgs a) {
  constexpr int RB = kHeadDim * BITS / 8;
  __shared__ int s_L, s_W, s_ok, s_flush, s_page;
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool windowed = a.k_layout == 1 || a.v_layout == 1;
  if (threadIdx.x == 0) {
    const int L = min(max(a.seq_lens[b], 0), a.T_cap);
    const int W = windowed ? min(max(a.win_lens[b], 0), a.win_cap) : 0;
    int ok, flush = 0;
    if (!windowed) {
      ok = L < a.T_cap;
    } else {
      flush = (W + 1 == a.group);
      ok = W < a.group && (!flush || (L % a.group == 0 && L + a.group <= a.T_cap));
    }
    if (!ok && a.status) atomicExch(a.status, kStatusAppendFull);
    // a paged cache: the page of position L (a token-wise store or a group flush)
    int page = 0;
    if (ok && a.pg.page_table && (!windowed || flush)) {
      page = kv_page(a.pg.page_table, a.pg.max_pages, a.pg.num_pages, a.pg.page_tokens, b, L);
      if (page < 0) {
        ok = 0;
        if (a.status) atomicExch(a.status, kStatusBadPage);
      }
    }
    s_L = L;
    s_W = W;
    s_ok = ok;
    s_flush = flush;
    s_page = page;
  }
  __syncthreads();
  if (!s_ok) return;  // nothing is written for this sequence
  const int L = s_L, W = s_W, page = s_page;

  if (!windowed) {
    // 2 Hkv token rows: (KV head, side); warp w takes rows w, w + 16, ...
    for (int row = warp; row < 2 * a.Hkv; row += kAppendWarps) {
      const int kvh = row >> 1, side = row & 1;
      const size_t unit = (size_t)b * a.Hkv + kvh;
      const size_t crow = append_addr(a, page, b, kvh, L).row;
      const size_t si = crow * (kHeadDim / a.group);
      float v[4];
      load_row4((side ? a.v_new : a.k_new) + unit * kHeadDim, lane, v);
      if (a.rotation & (1 << side)) rotate_bf16(v, lane);
      if (side)
        quantize_token_vals<BITS>(v, a.group, a.v_codes + crow * RB, a.v_scale + si, a.v_off + si, lane);
      else
        quantize_token_vals<BITS>(v, a.group, a.k_codes + crow * RB, a.k_scale + si, a.k_off + si, lane);
    }
    __syncthreads();
    if (threadIdx.x == 0) a.seq_lens[b] = L + 1;
    return;
  }

  // the token into window slot W (both sides), 8 bf16 per thread and step; a side stored
  // rotated goes in rotated (one warp per row)
  if (a.rotation) {
    for (int row = warp; row < 2 * a.Hkv; row += kAppendWarps) {
      const int kvh = row >> 1, side = row & 1;
      const size_t unit = (size_t)b * a.Hkv + kvh;
      float v[4];
      load_row4((side ? a.v_new : a.k_new) + unit * kHeadDim, lane, v);
      if (a.rotation & (1 << side)) hadamard128(v, lane);
      store_row4((side ? a.v_win : a.k_win) + (unit * a.win_cap + W) * kHeadDim, lane, v);
    }
  } else {
    for (int idx = threadIdx.x; idx < 2 * a.Hkv * (kHeadDim / 8); idx += kAppendThreads) {
      const int side = idx / (a.Hkv * (kHeadDim / 8));
      const int rem = idx - side * a.Hkv * (kHeadDim / 8);
      const int kvh = rem / (kHeadDim / 8), k8 = rem % (kHeadDim / 8);
      const size_t unit = (size_t)b * a.Hkv + kvh;
      const uint4 v = reinterpret_cast<const uint4*>((side ? a.v_new : a.k_new) + unit * kHeadDim)[k8];
      reinterpret_cast<uint4*>((side ? a.v_win : a.k_win) + (unit * a.win_cap + W) * kHeadDim)[k8] = v;
    }
  }
  if (!s_flush) {
    __syncthreads();
    if (threadIdx.x == 0) a.win_lens[b] = W + 1;
    return;
  }
  __syncthreads();  // the window's g tokens are in place
  flush_side<BITS>(a, a.k_win, a.k_layout, a.k_codes, a.k_scale, a.k_off, b, L, page);
  flush_side<BITS>(a, a.v_win, a.v_layout, a.v_codes, a.v_scale, a.v_off, b, L, page);
  __syncthreads();
  if (threadIdx.x == 0) {
    a.seq_lens[b] = L + a.group;
    a.win_lens[b] = 0;
  }
}

int launch_append(const AppendArgs& a, cudaStream_t stream) {
  if (a.B == 0) return 0;
  if (a.bits == 2)
    append_kernel<2><<<(unsigned)a.B, kAppendThreads, 0, stream>>>(a);
  else
    append_kernel<4><<<(unsigned)a.B, kAppendThreads, 0, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace lbkv
