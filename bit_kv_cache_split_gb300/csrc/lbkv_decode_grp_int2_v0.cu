// lbkv_decode_grp_int2_v0.cu -- instantiations of the group decode kernel (QK^T on the
// tensor cores, one product per 128-token item) for 2-bit codes with a token-wise K side
// and a token-wise V side.
#include "lbkv_decode_grp.cuh"
#include "lbkv_internal.h"

#ifndef LBKV_PAGED
#define LBKV_PAGED false  // the contiguous cache (lbkv_decode_grp_*_paged.cu: the paged one)
#endif

namespace lbkv {

template <>
DecodeKernel decode_kernel_grp<2, 0, LBKV_PAGED>(int mode, int log2g) {
#define LBKV_PICK(M, LG)                                                           \
  if (mode == M && log2g == LG) {                                                  \
    using C = Cfg<2, 0, 0, M, LG>;                                                   \
    if constexpr (GrpShape<C>::OK) return &grp_decode_kernel<C, LBKV_PAGED>;       \
    return nullptr;                                                                \
  }
  LBKV_PICK(kModeDup, 7)
  LBKV_PICK(kModePair, 7)
  LBKV_PICK(kModeDup, 6)
  LBKV_PICK(kModePair, 6)
  LBKV_PICK(kModeDup, 5)
  LBKV_PICK(kModePair, 5)
  LBKV_PICK(kModeWide, 6)
  LBKV_PICK(kModeWide, 5)
#undef LBKV_PICK
  return nullptr;
}

}  // namespace lbkv
