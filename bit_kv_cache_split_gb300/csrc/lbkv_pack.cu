// lbkv_pack.cu -- quantizer of a bf16 cache side into packed 2-/4-bit codes
// with one fp16 scale and offset per group, stored contiguously or in the pages of a
// paged cache. The arithmetic is the quantizer of lbkv_quant.cuh (min/max per group,
// s = fp16((max - min) / (2^b - 1)), z = fp16(min), q = clamp(rint(fl((x - z) / s)))),
// bit-exact, with a faster route to the same codes:
//
// Bracketed quotient. With inv = fl(1/s), inv_lo = fl(inv (1 - 2^-21)) and
// inv_hi = fl(inv (1 + 2^-21)), every d satisfies d inv_lo <= fl(d / s) <= d inv_hi
// for d >= 0 (fl(d / s) is within 2^-24 of d / s, inv within 2^-24 of 1 / s). One fused
// multiply-add per bound, fma(d, inv, 1.5 * 2^23), rounds the exact product to an integer
// (ties to even) in the low bits of its result; rint is monotone, so where the two bounds
// round to the same integer, that integer is rint(fl(d / s)). Where they differ (d / s
// within about 2^-20 d / s of a half-integer; with bf16 inputs these are nearly always
// exact ties, about 6e-4 of the values) the correctly rounded division decides: a thread
// notes the code words that hold such a value and recomputes them after all its words,
// so that the lanes of a warp that need a fix-up do it in one pass instead of each
// stopping the warp at its own word.
// A group takes this route when z equals its minimum exactly (a bf16 minimum inside the
// fp16 normal range) and s is a normal fp16, or zero: then 0 <= d / s < qmax + 0.01, so
// the codes need no clamp; any other group (and any value that is not finite) takes the
// division for every value.
#include "lbkv_internal.h"
#include "lbkv_quant.cuh"

namespace lbkv {

namespace {

constexpr int kPackRows = 64;     // token rows per CTA of the token-wise kernel (divides the 128-token slot)
constexpr int kPackStride = 272;  // their shared-memory stride: 256 bytes + 16 keeps 16-byte reads conflict-free
constexpr float kRintMagic = 12582912.f;  // 1.5 * 2^23: x + this has rint(x) in its low bits, |x| < 2^22

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Scale and offset of a group from its extremes, as lbkv_quant.cuh forms them, and the
// constants of the bracketed quotient. fast: the group may take the bracketed route.
struct GroupQ {
  __half sh, zh;
  float sf, zf, inv, inv_lo, inv_hi;
  bool fast;
};
template <int BITS>
__device__ __forceinline__ GroupQ group_params(float mn, float mx, bool has_nan) {
  constexpr int qmax = (1 << BITS) - 1;
  GroupQ g;
  mn = __fadd_rn(mn, 0.f);  // a -0 extreme is read as +0
  mx = __fadd_rn(mx, 0.f);
  g.sh = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), (float)qmax));
  g.zh = __float2half_rn(mn);
  g.sf = __half2float(g.sh);
  g.zf = __half2float(g.zh);
  g.inv = __frcp_rn(g.sf);
  g.inv_lo = __fmul_rn(g.inv, 1.f - 4.76837158203125e-07f);  // 1 - 2^-21
  g.inv_hi = __fmul_rn(g.inv, 1.f + 4.76837158203125e-07f);  // 1 + 2^-21
  // z = min and s normal; or s = 0 (a constant group: every code 0, as the bounds 0 give)
  // (a NaN value, which the extremes skip, would break the packing: division route)
  g.fast = !has_nan && (g.zf == mn) && ((g.sf >= 6.103515625e-05f && g.sf <= 65504.f) || g.sf == 0.f);
  if (g.sf == 0.f) g.inv_lo = g.inv_hi = 0.f;
  return g;
}

// Bracketed code of x (see the file comment): the integer in the low bits of the result;
// diff collects the bits in which the two bounds differ (zero where they agree).
__device__ __forceinline__ uint32_t bracket_code(float x, const GroupQ& g, uint32_t& diff) {
  const float d = __fsub_rn(x, g.zf);
  const uint32_t a = __float_as_uint(__fmaf_rn(d, g.inv_lo, kRintMagic));
  const uint32_t b = __float_as_uint(__fmaf_rn(d, g.inv_hi, kRintMagic));
  diff |= a ^ b;
  return a;
}
// The code of x in a group that takes the bracketed route, by the correctly rounded
// division (no clamp needed there).
__device__ __forceinline__ uint32_t exact_code(float x, const GroupQ& g) {
  if (g.sf == 0.f) return 0u;
  return (uint32_t)rintf(__fdiv_rn(__fsub_rn(x, g.zf), g.sf));
}

// Packs 16 (INT2) or 8 (INT4) bracketed codes (low bits of each word, anything above bit
// 21) into one word, code i at bits BITS i: shift-and-add pairs, whose garbage stays above
// bit 21, then one byte permute for the last level.
template <int BITS>
__device__ __forceinline__ uint32_t pack_word(const uint32_t* c) {
  constexpr int N = 32 / BITS;
  uint32_t u[N / 2];
#pragma unroll
  for (int i = 0; i < N / 2; ++i) u[i] = (c[2 * i + 1] << BITS) + c[2 * i];
  int n = N / 2, sh = 2 * BITS;
#pragma unroll
  for (; n > 2; n >>= 1, sh <<= 1)
#pragma unroll
    for (int i = 0; i < n / 2; ++i) u[i] = (u[2 * i + 1] << sh) + u[2 * i];
  return __byte_perm(u[0], u[1], 0x5410);  // low 16 bits of each
}

template <int GW>
__device__ __forceinline__ void store_words(uint32_t* dst, const uint32_t (&out)[GW]) {
  if constexpr (GW % 4 == 0) {
#pragma unroll
    for (int j = 0; j < GW; j += 4)
      *reinterpret_cast<uint4*>(dst + j) = make_uint4(out[j], out[j + 1], out[j + 2], out[j + 3]);
  } else {
#pragma unroll
    for (int j = 0; j < GW; j += 2) *reinterpret_cast<uint2*>(dst + j) = make_uint2(out[j], out[j + 1]);
  }
}

// Codes of the token-wise group of G bf16 values at x (shared memory, 16-byte aligned) into
// the code words dst[0 .. G * BITS / 32 - 1], its scale and offset into sh, zh, its
// quotient constants into g. Two passes over x: extremes, then codes (fewer registers
// than holding the group, so more CTAs share an SM). Returns the mask of the words that
// hold a value whose bounds differ (to be recomputed by fix_word).
template <int BITS, int G>
__device__ __forceinline__ uint32_t quantize_group_smem(const uint4* x, uint32_t* dst, __half& sh, __half& zh,
                                                        GroupQ& g) {
  constexpr int qmax = (1 << BITS) - 1, PER = 32 / BITS, GW = G * BITS / 32;
  constexpr int CPW = PER / 8;  // 16-byte chunks (8 values) per code word: 2 at INT2, 1 at INT4
  __nv_bfloat162 mn2, mx2, nan2;
#pragma unroll
  for (int k = 0; k < G / 8; ++k) {
    const uint4 v = x[k];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
      if (k == 0 && i == 0) {
        mn2 = mx2 = nan2 = b;
      } else {
        mn2 = __hmin2(mn2, b);
        mx2 = __hmax2(mx2, b);
        nan2 = __hmin2_nan(nan2, b);  // NaN if any value is
      }
    }
  }
  const float mn = fminf(__low2float(mn2), __high2float(mn2));
  const float mx = fmaxf(__low2float(mx2), __high2float(mx2));
  const float nn = __low2float(nan2) + __high2float(nan2);
  g = group_params<BITS>(mn, mx, nn != nn);
  sh = g.sh;
  zh = g.zh;
  uint32_t bad = 0u, out[GW];
#pragma unroll
  for (int j = 0; j < GW; ++j) {
    uint32_t w[PER / 2];
#pragma unroll
    for (int cc = 0; cc < CPW; ++cc) {
      const uint4 v = x[j * CPW + cc];
      w[4 * cc] = v.x, w[4 * cc + 1] = v.y, w[4 * cc + 2] = v.z, w[4 * cc + 3] = v.w;
    }
    if (g.fast) {
      uint32_t c[PER], diff = 0u;
#pragma unroll
      for (int i = 0; i < PER / 2; ++i) {
        c[2 * i] = bracket_code(bf16_lo(w[i]), g, diff);
        c[2 * i + 1] = bracket_code(bf16_hi(w[i]), g, diff);
      }
      out[j] = pack_word<BITS>(c);
      bad |= (diff != 0u ? 1u : 0u) << j;
    } else {  // the correctly rounded division for every value of the group
      uint32_t word = 0u;
#pragma unroll
      for (int i = 0; i < PER / 2; ++i) {
        word |= (uint32_t)quantize_one(bf16_lo(w[i]), g.zf, g.sf, g.inv, qmax) << (BITS * 2 * i);
        word |= (uint32_t)quantize_one(bf16_hi(w[i]), g.zf, g.sf, g.inv, qmax) << (BITS * (2 * i + 1));
      }
      out[j] = word;
    }
  }
  store_words<GW>(dst, out);
  return bad;
}

// Code word j of a bracketed group recomputed by the division, from the group's bf16
// values x[0 .. G-1].
template <int BITS>
__device__ __forceinline__ uint32_t fix_word(const __nv_bfloat16* x, int j, const GroupQ& g) {
  constexpr int PER = 32 / BITS;
  uint32_t word = 0u;
#pragma unroll
  for (int i = 0; i < PER; ++i) word |= exact_code(__bfloat162float(x[j * PER + i]), g) << (BITS * i);
  return word;
}

// The storage row and channel-group block of token t of cache unit `unit` (= b * Hkv +
// kvh), or false when the token lies in no page of the pool (recorded as status 5).
__device__ __forceinline__ bool pack_addr(const PackArgs& a, size_t unit, int t, KvAddr* ad) {
  int page = 0;
  const int b = (int)(unit / a.Hkv), kvh = (int)(unit % a.Hkv);
  if (a.pg.page_table) {
    page = kv_page(a.pg.page_table, a.pg.max_pages, a.pg.num_pages, a.pg.page_tokens, b, t);
    if (page < 0) {
      if (a.status) atomicExch(a.status, kStatusBadPage);
      return false;
    }
  }
  *ad = kv_addr(a.pg.page_tokens, page, unit, kvh, a.Hkv, a.T_cap, a.group, t);
  return true;
}

// Token-wise groups: a CTA takes kPackRows consecutive token rows of one cache unit
// (T_cap is a multiple of 128), stages them in shared memory with coalesced 16-byte loads,
// and thread (row, group) quantizes one group of G channels. The contiguous cache has the
// codes of positions t >= L_b cleared; the paged cache stores positions t < L_b only.
template <int BITS, int G>
__global__ void __launch_bounds__(kPackRows * (kHeadDim / G), 13 * kPackRows / (kPackRows * (kHeadDim / G)))
    pack_tokenwise_kernel(const __grid_constant__ PackArgs a) {
  constexpr int TPR = kHeadDim / G, NT = kPackRows * TPR;
  constexpr int RB = kHeadDim * BITS / 8, GW = G * BITS / 32;  // code bytes per row, code words per group
  __shared__ __align__(16) uint8_t tile[kPackRows * kPackStride];
  const size_t row0 = (size_t)blockIdx.x * kPackRows;
  const size_t unit = row0 / (size_t)a.T_cap;
  const int t0 = (int)(row0 - unit * (size_t)a.T_cap);
  const int L = a.seq_lens[unit / a.Hkv];
  const int nvalid = min(max(L - t0, 0), kPackRows);
  if (nvalid == 0 && a.pg.page_table) return;
  const uint4* src = reinterpret_cast<const uint4*>(a.x + row0 * kHeadDim);
  for (int i = threadIdx.x; i < nvalid * 16; i += NT)
    *reinterpret_cast<uint4*>(tile + (i >> 4) * kPackStride + (i & 15) * 16) = __ldcs(src + i);
  __syncthreads();
  const int r = threadIdx.x / TPR, gi = threadIdx.x % TPR;
  const bool valid = r < nvalid;
  if (!valid && a.pg.page_table) return;
  KvAddr ad;
  if (!pack_addr(a, unit, t0 + r, &ad)) return;
  uint32_t* dst = reinterpret_cast<uint32_t*>(a.codes + ad.row * RB) + gi * GW;
  if (valid) {
    const uint4* row = reinterpret_cast<const uint4*>(tile + r * kPackStride + gi * G * 2);
    __half sh, zh;
    GroupQ g;
    uint32_t bad = quantize_group_smem<BITS, G>(row, dst, sh, zh, g);
    const size_t si = ad.row * (kHeadDim / G) + gi;
    a.scale[si] = sh;
    a.off[si] = zh;
    const __nv_bfloat16* xg = reinterpret_cast<const __nv_bfloat16*>(tile + r * kPackStride + gi * G * 2);
    while (bad) {  // rare: words with a value on a rounding boundary, after the plain stores
      const int j = __ffs(bad) - 1;
      bad &= bad - 1u;
      dst[j] = fix_word<BITS>(xg, j, g);
    }
  } else {
    uint32_t out[GW];
#pragma unroll
    for (int j = 0; j < GW; ++j) out[j] = 0u;
    store_words<GW>(dst, out);
  }
}

// Channel-wise groups: one CTA of kCwWarps warps per (unit, token group tau). Warp w takes
// the group's tokens w G/kCwWarps .. (w+1) G/kCwWarps - 1, lane p the channels 4p .. 4p+3
// (one INT2 code byte, two INT4 code bytes, per token); a warp reads each token row whole
// (256 bytes). A thread loads all its values at once and holds them in registers for both
// passes (no shared-memory tile). Pass 1: per-warp extremes per channel; thread d < 128
// combines them for channel d and forms the group's scale, offset and quotient constants.
// Pass 2: the codes. Full groups (the common case) take a path without per-token tests.
// The paged cache stores the groups that hold a position t < L_b only.
constexpr int kCwWarps = 8;

template <int BITS, int TW, bool FULL>
__device__ __forceinline__ void cw_codes(const uint2 (&xv)[TW], int nv, const float (&zf)[4], const float (&lo)[4],
                                         const float (&hi)[4], bool fast4, const GroupQ* gq, int lane, uint8_t* crow,
                                         uint32_t& bad) {
  constexpr int qmax = (1 << BITS) - 1, RB = kHeadDim * BITS / 8;
#pragma unroll
  for (int k = 0; k < TW; ++k) {
    uint32_t word = 0u;  // codes of channels 4 lane .. 4 lane + 3 at bits BITS u
    if (FULL || k < nv) {
      const float x[4] = {bf16_lo(xv[k].x), bf16_hi(xv[k].x), bf16_lo(xv[k].y), bf16_hi(xv[k].y)};
      if (fast4) {
        uint32_t c[4], diff = 0u;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float d = __fsub_rn(x[u], zf[u]);
          c[u] = __float_as_uint(__fmaf_rn(d, lo[u], kRintMagic));
          diff |= c[u] ^ __float_as_uint(__fmaf_rn(d, hi[u], kRintMagic));
        }
        word = ((((c[3] << BITS) + c[2]) << (2 * BITS)) + (c[1] << BITS) + c[0]) & ((1u << (4 * BITS)) - 1u);
        bad |= (diff != 0u ? 1u : 0u) << k;
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const GroupQ& g = gq[4 * lane + u];
          word |= (uint32_t)quantize_one(x[u], g.zf, g.sf, g.inv, qmax) << (BITS * u);
        }
      }
    }
    uint8_t* cr = crow + k * RB;
    if (BITS == 2)
      *cr = (uint8_t)word;
    else
      *reinterpret_cast<uint16_t*>(cr) = (uint16_t)word;
  }
}

template <int BITS, int G>
__global__ void __launch_bounds__(32 * kCwWarps) pack_channelwise_kernel(const __grid_constant__ PackArgs a) {
  constexpr int RB = kHeadDim * BITS / 8, TW = G / kCwWarps;  // tokens per warp
  __shared__ float2 part[kCwWarps][kHeadDim];
  __shared__ uint32_t part_nan[kCwWarps][kHeadDim / 4];  // per warp and lane: a NaN among its values
  __shared__ GroupQ gq[kHeadDim];
  const int unit = blockIdx.x, tau = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = a.seq_lens[unit / a.Hkv];
  const int t0 = tau * G;
  const int nvalid = max(0, min(G, L - t0));
  if (nvalid == 0 && a.pg.page_table) return;
  KvAddr ad;
  if (!pack_addr(a, (size_t)unit, t0, &ad)) return;
  // this lane's 4 channels of the warp's first token (rows of 32 uint2)
  const int tw0 = warp * TW;
  const uint2* src = reinterpret_cast<const uint2*>(a.x + ((size_t)unit * a.T_cap + t0 + tw0) * kHeadDim) + lane;
  const int nv = min(max(nvalid - tw0, 0), TW);  // this warp's valid tokens
  const bool full = nvalid == G;
  uint2 xv[TW];
  if (full) {
#pragma unroll
    for (int k = 0; k < TW; ++k) xv[k] = __ldcs(src + k * 32);
  } else {
#pragma unroll
    for (int k = 0; k < TW; ++k) xv[k] = (k < nv) ? __ldcs(src + k * 32) : make_uint2(0u, 0u);
  }
  if (nv > 0) {
    __nv_bfloat162 mnA = *reinterpret_cast<__nv_bfloat162*>(&xv[0].x), mxA = mnA, nA = mnA;
    __nv_bfloat162 mnB = *reinterpret_cast<__nv_bfloat162*>(&xv[0].y), mxB = mnB, nB = mnB;
#pragma unroll
    for (int k = 1; k < TW; ++k) {
      if (!full && k >= nv) break;
      const __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&xv[k].x);
      const __nv_bfloat162 y = *reinterpret_cast<__nv_bfloat162*>(&xv[k].y);
      mnA = __hmin2(mnA, x), mxA = __hmax2(mxA, x), nA = __hmin2_nan(nA, x);
      mnB = __hmin2(mnB, y), mxB = __hmax2(mxB, y), nB = __hmin2_nan(nB, y);
    }
    const float nn = __low2float(nA) + __high2float(nA) + __low2float(nB) + __high2float(nB);
    part_nan[warp][lane] = nn != nn ? 1u : 0u;
    part[warp][4 * lane] = make_float2(__low2float(mnA), __low2float(mxA));
    part[warp][4 * lane + 1] = make_float2(__high2float(mnA), __high2float(mxA));
    part[warp][4 * lane + 2] = make_float2(__low2float(mnB), __low2float(mxB));
    part[warp][4 * lane + 3] = make_float2(__high2float(mnB), __high2float(mxB));
  }
  __syncthreads();
  if (nvalid > 0 && threadIdx.x < kHeadDim) {
    const int d = threadIdx.x;
    float2 e = part[0][d];
    bool has_nan = part_nan[0][d / 4] != 0u;
    for (int w = 1; w < kCwWarps && w * TW < nvalid; ++w) {
      const float2 f = part[w][d];
      e.x = fminf(e.x, f.x);
      e.y = fmaxf(e.y, f.y);
      has_nan = has_nan || part_nan[w][d / 4] != 0u;
    }
    const GroupQ g = group_params<BITS>(e.x, e.y, has_nan);
    gq[d] = g;
    const size_t si = ad.block * kHeadDim + d;
    a.scale[si] = g.sh;
    a.off[si] = g.zh;
  }
  __syncthreads();
  float zf[4] = {0.f, 0.f, 0.f, 0.f}, lo[4] = {0.f, 0.f, 0.f, 0.f}, hi[4] = {0.f, 0.f, 0.f, 0.f};
  bool fast4 = true;
  if (nvalid > 0) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const GroupQ& g = gq[4 * lane + u];
      zf[u] = g.zf, lo[u] = g.inv_lo, hi[u] = g.inv_hi;
      fast4 = fast4 && g.fast;
    }
  }
  uint8_t* crow = a.codes + (ad.row + tw0) * RB + (BITS / 2) * lane;  // this lane's code byte(s), token tw0
  uint32_t bad = 0u;  // tokens whose codes are recomputed by the division
  if (full)
    cw_codes<BITS, TW, true>(xv, nv, zf, lo, hi, fast4, gq, lane, crow, bad);
  else
    cw_codes<BITS, TW, false>(xv, nv, zf, lo, hi, fast4, gq, lane, crow, bad);
  while (bad) {  // rare: tokens with a value on a rounding boundary, after the plain stores
    const int k = __ffs(bad) - 1;
    bad &= bad - 1u;
    const uint2 v = src[k * 32];
    const float x[4] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y)};
    uint32_t word = 0u;
#pragma unroll
    for (int u = 0; u < 4; ++u) word |= exact_code(x[u], gq[4 * lane + u]) << (BITS * u);
    uint8_t* cr = crow + k * RB;
    if (BITS == 2)
      *cr = (uint8_t)word;
    else
      *reinterpret_cast<uint16_t*>(cr) = (uint16_t)word;
  }
}

template <int BITS>
void launch_pack_bits(const PackArgs& a, cudaStream_t stream) {
  if (a.layout == 0) {
    const long long rows = (long long)a.B * a.Hkv * a.T_cap;
    const unsigned blocks = (unsigned)(rows / kPackRows);  // T_cap is a multiple of kPackRows
    if (a.group == 128)
      pack_tokenwise_kernel<BITS, 128><<<blocks, kPackRows, 0, stream>>>(a);
    else if (a.group == 64)
      pack_tokenwise_kernel<BITS, 64><<<blocks, kPackRows * 2, 0, stream>>>(a);
    else
      pack_tokenwise_kernel<BITS, 32><<<blocks, kPackRows * 4, 0, stream>>>(a);
  } else {
    dim3 grid((unsigned)(a.B * a.Hkv), (unsigned)(a.T_cap / a.group));
    if (a.group == 128)
      pack_channelwise_kernel<BITS, 128><<<grid, 32 * kCwWarps, 0, stream>>>(a);
    else if (a.group == 64)
      pack_channelwise_kernel<BITS, 64><<<grid, 32 * kCwWarps, 0, stream>>>(a);
    else
      pack_channelwise_kernel<BITS, 32><<<grid, 32 * kCwWarps, 0, stream>>>(a);
  }
}

}  // namespace

int launch_pack(const PackArgs& a, cudaStream_t stream) {
  static_assert(kSlotTokens % kPackRows == 0, "a CTA's rows lie in one cache unit");
  if (a.bits == 2)
    launch_pack_bits<2>(a, stream);
  else
    launch_pack_bits<4>(a, stream);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace lbkv
