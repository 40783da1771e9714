// lbkv_pack.cu -- quantizer of a bf16 cache side into packed 2-/4-bit codes
// with one fp16 scale and offset per group (the arithmetic is in lbkv_quant.cuh).
#include "lbkv_internal.h"
#include "lbkv_quant.cuh"

namespace lbkv {

// One warp per token row.
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
  const long long si = row * (kHeadDim / group);
  quantize_token_row<BITS>(x + row * kHeadDim, group, crow, scale + si, off + si, lane);
}

// One block of 128 threads per (unit, token group): thread d owns channel d.
template <int BITS>
__global__ void __launch_bounds__(128) pack_channelwise_kernel(const __nv_bfloat16* __restrict__ x,
                                                               const int32_t* __restrict__ seq_lens, int Hkv,
                                                               int T_cap, int group, uint8_t* __restrict__ codes,
                                                               __half* __restrict__ scale,
                                                               __half* __restrict__ off) {
  constexpr int RB = kHeadDim * BITS / 8;
  const int unit = blockIdx.x, tau = blockIdx.y, d = threadIdx.x;
  const int b = unit / Hkv;
  const int L = seq_lens[b];
  const int t0 = tau * group;
  const int nvalid = max(0, min(group, L - t0));
  const size_t rowbase = (size_t)unit * T_cap + t0;
  const size_t si = ((size_t)unit * (T_cap / group) + tau) * kHeadDim + d;
  quantize_channel_group<BITS>(x + rowbase * kHeadDim, nvalid, group, codes + rowbase * RB, scale + si, off + si, d);
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
