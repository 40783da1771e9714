// lbkv_pack.cu -- quantizer of a bf16 cache side into packed 2-/4-bit codes
// with one fp16 scale and offset per group (the arithmetic is in lbkv_quant.cuh), stored
// contiguously or in the pages of a paged cache.
#include "lbkv_internal.h"
#include "lbkv_quant.cuh"

namespace lbkv {

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

// One warp per token row. The contiguous cache has the codes of positions t >= L_b
// cleared; the paged cache stores positions t < L_b only.
template <int BITS>
__global__ void __launch_bounds__(256) pack_tokenwise_kernel(const __grid_constant__ PackArgs a) {
  constexpr int RB = kHeadDim * BITS / 8;
  const long long rows = (long long)a.B * a.Hkv * a.T_cap;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int t = (int)(row % a.T_cap);
  const size_t unit = (size_t)(row / a.T_cap);
  const bool valid = t < a.seq_lens[unit / a.Hkv];
  if (!valid && a.pg.page_table) return;
  KvAddr ad;
  if (!pack_addr(a, unit, t, &ad)) return;
  uint8_t* crow = a.codes + ad.row * RB;
  if (!valid) {
    if (BITS == 2)
      crow[lane] = 0;
    else
      reinterpret_cast<uint16_t*>(crow)[lane] = 0;
    return;
  }
  const size_t si = ad.row * (kHeadDim / a.group);
  quantize_token_row<BITS>(a.x + row * kHeadDim, a.group, crow, a.scale + si, a.off + si, lane);
}

// One block of 128 threads per (unit, token group): thread d owns channel d. The paged
// cache stores the groups that hold a position t < L_b only.
template <int BITS>
__global__ void __launch_bounds__(128) pack_channelwise_kernel(const __grid_constant__ PackArgs a) {
  constexpr int RB = kHeadDim * BITS / 8;
  const int unit = blockIdx.x, tau = blockIdx.y, d = threadIdx.x;
  const int L = a.seq_lens[unit / a.Hkv];
  const int t0 = tau * a.group;
  const int nvalid = max(0, min(a.group, L - t0));
  if (nvalid == 0 && a.pg.page_table) return;
  KvAddr ad;
  if (!pack_addr(a, (size_t)unit, t0, &ad)) return;
  const size_t xrow = (size_t)unit * a.T_cap + t0;
  const size_t si = ad.block * kHeadDim + d;
  quantize_channel_group<BITS>(a.x + xrow * kHeadDim, nvalid, a.group, a.codes + ad.row * RB, a.scale + si,
                               a.off + si, d);
}

int launch_pack(const PackArgs& a, cudaStream_t stream) {
  if (a.layout == 0) {
    const long long rows = (long long)a.B * a.Hkv * a.T_cap;
    const unsigned blocks = (unsigned)((rows + 7) / 8);
    if (a.bits == 2)
      pack_tokenwise_kernel<2><<<blocks, 256, 0, stream>>>(a);
    else
      pack_tokenwise_kernel<4><<<blocks, 256, 0, stream>>>(a);
  } else {
    dim3 grid((unsigned)(a.B * a.Hkv), (unsigned)(a.T_cap / a.group));
    if (a.bits == 2)
      pack_channelwise_kernel<2><<<grid, 128, 0, stream>>>(a);
    else
      pack_channelwise_kernel<4><<<grid, 128, 0, stream>>>(a);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace lbkv
