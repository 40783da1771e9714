// lbkv_quant.cuh -- the quantizer of one token row (token-wise groups) and of one
// channel over a token group (channel-wise groups), shared by the pack and append
// kernels so that both produce the same bits.
//
// Value model s * q + z with unsigned b-bit codes: explainer "FOSCAR speeds up
// 2-bit KV decode -- Affine folding of KV dequantization", quantization-format
// paragraph. The quantizer (min/max per group, round-half-even) is this
// library's reading; every step is one IEEE single-precision operation rounded
// on its own (no contraction), so the result is bit-exact:
//   s = fp16((max - min) / (2^b - 1)),  z = fp16(min),
//   q = clamp(rint((x - z) / s), 0, 2^b - 1),  q = 0 when s == 0.
#pragma once

#include "lbkv_decode.cuh"

namespace lbkv {

// q = clamp(rint(fl((x - z) / s)), 0, qmax), with fl the correctly rounded fp32 division;
// inv = fl(1 / s). The division is done only where it can change the result: the product
// r = fl(d * inv) differs from fl(d / s) by at most 3 * 2^-24 |d / s| (three roundings),
// i.e. by less than 3 * 2^-18 (< 2^-16) for |r| < 64, so wherever r is at least 2^-16 away
// from a half-integer (the only places where rint changes) both round to the same integer,
// and the clamp sees the same value (r - floor(r) is exact for r >= 0 and off by at most
// 2^-24 below). Near a half-integer (ties to even among them), for |r| >= 64 and for
// non-finite values the correctly rounded division decides.
__device__ __forceinline__ int quantize_one(float x, float zf, float sf, float inv, int qmax) {
  if (sf == 0.f) return 0;
  const float d = __fsub_rn(x, zf);
  float v = __fmul_rn(d, inv);
  const float fr = __fsub_rn(v, floorf(v));
  if (!(fabsf(v) < 64.f) || fabsf(__fsub_rn(fr, 0.5f)) < 1.52587890625e-05f) v = __fdiv_rn(d, sf);
  const float r = rintf(v);
  return r < 0.f ? 0 : (r > (float)qmax ? qmax : (int)r);
}

// One warp quantizes one token row with token-wise groups of `group` channels, given as
// the fp32 values of channels 4 lane .. 4 lane + 3 in v: codes into crow[D * BITS / 8],
// the group's scale and offset into srow/zrow[D / group]. A group is group/4 consecutive lanes.
template <int BITS>
__device__ __forceinline__ void quantize_token_vals(const float (&v)[4], int group, uint8_t* crow, __half* srow,
                                                    __half* zrow, int lane) {
  float mn = fminf(fminf(v[0], v[1]), fminf(v[2], v[3]));
  float mx = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
  const int lanes = group / 4;
  for (int o = 1; o < lanes; o <<= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  constexpr int qmax = (1 << BITS) - 1;
  mn = __fadd_rn(mn, 0.f);  // a -0 extreme is read as +0
  mx = __fadd_rn(mx, 0.f);
  const __half sh = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), (float)qmax));
  const __half zh = __float2half_rn(mn);
  const float sf = __half2float(sh), zf = __half2float(zh);
  const float inv = __frcp_rn(sf);
  uint32_t packed = 0;
#pragma unroll
  for (int u = 0; u < 4; ++u) packed |= (uint32_t)quantize_one(v[u], zf, sf, inv, qmax) << (BITS * u);
  if (BITS == 2)
    crow[lane] = (uint8_t)packed;
  else
    reinterpret_cast<uint16_t*>(crow)[lane] = (uint16_t)packed;
  if (lane % lanes == 0) {
    srow[lane / lanes] = sh;
    zrow[lane / lanes] = zh;
  }
}

// The same for the bf16 token row x[D].
template <int BITS>
__device__ __forceinline__ void quantize_token_row(const __nv_bfloat16* __restrict__ x, int group, uint8_t* crow,
                                                   __half* srow, __half* zrow, int lane) {
  float v[4];
  load_row4(x, lane, v);
  quantize_token_vals<BITS>(v, group, crow, srow, zrow, lane);
}

// Thread d of 128 (channel d) quantizes channel d over one channel-wise token group:
// tokens x[t * D + d], t < nvalid (rows with t >= nvalid, up to `group`, get code 0);
// codes into crows[t * D * BITS / 8 + ...], the group's scale and offset into *s / *z.
// Threads d and d^1 (and d^2, d^3 at INT2) share code bytes: all 128 threads take part.
template <int BITS>
__device__ __forceinline__ void quantize_channel_group(const __nv_bfloat16* __restrict__ x, int nvalid, int group,
                                                       uint8_t* crows, __half* s, __half* z, int d) {
  constexpr int RB = kHeadDim * BITS / 8;
  constexpr int per_byte = 8 / BITS;
  constexpr int qmax = (1 << BITS) - 1;
  float sf = 0.f, zf = 0.f, inv = 0.f;
  if (nvalid > 0) {
    float mn = __bfloat162float(x[d]), mx = mn;
    for (int t = 1; t < nvalid; ++t) {
      const float v = __bfloat162float(x[(size_t)t * kHeadDim + d]);
      mn = fminf(mn, v);
      mx = fmaxf(mx, v);
    }
    mn = __fadd_rn(mn, 0.f);  // a -0 extreme is read as +0
    mx = __fadd_rn(mx, 0.f);
    const __half sh = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), (float)qmax));
    const __half zh = __float2half_rn(mn);
    *s = sh;
    *z = zh;
    sf = __half2float(sh);
    zf = __half2float(zh);
    inv = __frcp_rn(sf);
  }
  for (int t = 0; t < group; ++t) {
    int q = 0;
    if (t < nvalid) q = quantize_one(__bfloat162float(x[(size_t)t * kHeadDim + d]), zf, sf, inv, qmax);
    // gather the codes of the channels sharing this byte (adjacent lanes)
    uint32_t bits = (uint32_t)q << (BITS * (d % per_byte));
#pragma unroll
    for (int o = 1; o < per_byte; o <<= 1) bits |= __shfl_xor_sync(0xffffffffu, bits, o);
    if (d % per_byte == 0) crows[(size_t)t * RB + d / per_byte] = (uint8_t)bits;
  }
}

}  // namespace lbkv
