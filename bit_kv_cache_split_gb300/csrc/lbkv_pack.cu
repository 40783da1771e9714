// lbkv_pack.cu -- quantizer of a bf16 cache side into packed 2-/4-bit codes
// with one fp16 scale and offset per group.
//
// Value model s * q + z with unsigned b-bit codes: explainer "FOSCAR speeds up
// 2-bit KV decode -- Affine folding of KV dequantization", quantization-format
// paragraph. The quantizer (min/max per group, round-half-even) is this
// library's reading; every step is one IEEE single-precision operation rounded
// on its own (no contraction), so the result is bit-exact:
//   s = fp16((max - min) / (2^b - 1)),  z = fp16(min),
//   q = clamp(rint((x - z) / s), 0, 2^b - 1),  q = 0 when s == 0.
#include "lbkv_internal.h"

namespace lbkv {

__device__ __forceinline__ int quantize_one(float x, float zf, float sf, int qmax) {
  if (sf == 0.f) return 0;
  const float v = __fdiv_rn(__fsub_rn(x, zf), sf);
  const float r = rintf(v);
  return r < 0.f ? 0 : (r > (float)qmax ? qmax : (int)r);
}

// One warp per token row; lane l holds channels 4l..4l+3. A group is g
// consecutive channels = g/4 consecutive lanes.
template <int BITS>
__global__ void __launch_bounds__(256) pack_tokenwise_kernel(const __nv_bfloat16* __restrict__ x,
                                                             const int32_t* __restrict__ seq_lens, int Hkv,
                                                             int T_cap, int group, long long rows,
                                                             uint8_t* __restrict__ codes, __half* __restrict__ scale,
                                                             __half* __restrict__ off) {
  constexpr int RB = kHeadDim * BITS / 8;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int t = (int)(row % T_cap);
  const int b = (int)(row / T_cap / Hkv);
  uint8_t* crow = codes + row * RB;
  if (t >= seq_lens[b]) {
    if (BITS == 2)
      crow[lane] = 0;
    else
      reinterpret_cast<uint16_t*>(crow)[lane] = 0;
    return;
  }
  const uint2 raw = reinterpret_cast<const uint2*>(x + row * kHeadDim)[lane];
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
  const float2 a = __bfloat1622float2(h[0]), c = __bfloat1622float2(h[1]);
  const float v[4] = {a.x, a.y, c.x, c.y};
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
  uint32_t packed = 0;
#pragma unroll
  for (int u = 0; u < 4; ++u) packed |= (uint32_t)quantize_one(v[u], zf, sf, qmax) << (BITS * u);
  if (BITS == 2)
    crow[lane] = (uint8_t)packed;
  else
    reinterpret_cast<uint16_t*>(crow)[lane] = (uint16_t)packed;
  if (lane % lanes == 0) {
    const long long si = row * (kHeadDim / group) + lane / lanes;
    scale[si] = sh;
    off[si] = zh;
  }
}

// One block of 128 threads per (unit, token group): thread d owns channel d.
template <int BITS>
__global__ void __launch_bounds__(128) pack_channelwise_kernel(const __nv_bfloat16* __restrict__ x,
                                                               const int32_t* __restrict__ seq_lens, int Hkv,
                                                               int T_cap, int group, uint8_t* __restrict__ codes,
                                                               __half* __restrict__ scale,
                                                               __half* __restrict__ off) {
  constexpr int RB = kHeadDim * BITS / 8;
  constexpr int per_byte = 8 / BITS;
  const int unit = blockIdx.x, tau = blockIdx.y, d = threadIdx.x;
  const int b = unit / Hkv;
  const int L = seq_lens[b];
  const int t0 = tau * group;
  const int nvalid = max(0, min(group, L - t0));
  const size_t rowbase = (size_t)unit * T_cap + t0;
  constexpr int qmax = (1 << BITS) - 1;
  float sf = 0.f, zf = 0.f;
  if (nvalid > 0) {
    float mn = __bfloat162float(x[rowbase * kHeadDim + d]), mx = mn;
    for (int t = 1; t < nvalid; ++t) {
      const float v = __bfloat162float(x[(rowbase + t) * kHeadDim + d]);
      mn = fminf(mn, v);
      mx = fmaxf(mx, v);
    }
    mn = __fadd_rn(mn, 0.f);  // a -0 extreme is read as +0
    mx = __fadd_rn(mx, 0.f);
    const __half sh = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), (float)qmax));
    const __half zh = __float2half_rn(mn);
    const size_t si = ((size_t)unit * (T_cap / group) + tau) * kHeadDim + d;
    scale[si] = sh;
    off[si] = zh;
    sf = __half2float(sh);
    zf = __half2float(zh);
  }
  for (int t = 0; t < group; ++t) {
    int q = 0;
    if (t < nvalid) q = quantize_one(__bfloat162float(x[(rowbase + t) * kHeadDim + d]), zf, sf, qmax);
    // gather the codes of the channels sharing this byte (adjacent lanes)
    uint32_t bits = (uint32_t)q << (BITS * (d % per_byte));
#pragma unroll
    for (int o = 1; o < per_byte; o <<= 1) bits |= __shfl_xor_sync(0xffffffffu, bits, o);
    if (d % per_byte == 0) codes[(rowbase + t) * RB + d / per_byte] = (uint8_t)bits;
  }
}

int launch_pack(const PackArgs& a, cudaStream_t stream) {
  if (a.layout == 0) {
    const long long rows = (long long)a.B * a.Hkv * a.T_cap;
    const unsigned blocks = (unsigned)((rows + 7) / 8);
    if (a.bits == 2)
      pack_tokenwise_kernel<2><<<blocks, 256, 0, stream>>>(a.x, a.seq_lens, a.Hkv, a.T_cap, a.group, rows, a.codes,
                                                           a.scale, a.off);
    else
      pack_tokenwise_kernel<4><<<blocks, 256, 0, stream>>>(a.x, a.seq_lens, a.Hkv, a.T_cap, a.group, rows, a.codes,
                                                           a.scale, a.off);
  } else {
    dim3 grid((unsigned)(a.B * a.Hkv), (unsigned)(a.T_cap / a.group));
    if (a.bits == 2)
      pack_channelwise_kernel<2><<<grid, 128, 0, stream>>>(a.x, a.seq_lens, a.Hkv, a.T_cap, a.group, a.codes, a.scale,
                                                           a.off);
    else
      pack_channelwise_kernel<4><<<grid, 128, 0, stream>>>(a.x, a.seq_lens, a.Hkv, a.T_cap, a.group, a.codes, a.scale,
                                                           a.off);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace lbkv
