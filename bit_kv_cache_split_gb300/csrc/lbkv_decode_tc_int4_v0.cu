// lbkv_decode_tc_int4_v0.cu -- instantiations of the tensor-core QK^T decode kernel for
// 4-bit codes with a token-wise K side and a token-wise V side.
#include "lbkv_decode_tc.cuh"
#include "lbkv_internal.h"

#ifndef LBKV_PAGED
#define LBKV_PAGED false  // the contiguous cache (lbkv_decode_tc_*_paged.cu: the paged one)
#endif

namespace lbkv {

template <>
TcKernelInfo tc_kernel<4, 0, LBKV_PAGED>(int mode, int log2g) {
#define LBKV_PICK(M, LG)                                                                       \
  if (mode == M && log2g == LG) {                                                              \
    using C = TcCfg<4, 0, M, LG>;                                                              \
    return TcKernelInfo{&tc_decode_kernel<C, LBKV_PAGED>, C::MERGE_OFF, C::E.bytes, C::WARPS, C::MAX_RING}; \
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
  return TcKernelInfo{nullptr, 0, 0, 0, 0};
}

}  // namespace lbkv
