// lbkv_decode_int2_k0_v1.cu -- instantiations of the split-decode kernel for
// 2-bit codes with a token-wise K side and a channel-wise V side.
#include "lbkv_internal.h"

#ifndef LBKV_PAGED
#define LBKV_PAGED false  // the contiguous cache (lbkv_decode_*_paged.cu: the paged one)
#endif

namespace lbkv {

template <>
DecodeKernel decode_kernel<2, 0, 1, LBKV_PAGED>(int mode, int log2g, bool cluster) {
#define LBKV_PICK(M, LG) \
  if (mode == M && log2g == LG)                                                            \
    return cluster ? &split_decode_kernel<Cfg<2, 0, 1, M, LG>, LBKV_PAGED, true> \
                   : &split_decode_kernel<Cfg<2, 0, 1, M, LG>, LBKV_PAGED, false>;
  LBKV_PICK(kModeDup, 7)
  LBKV_PICK(kModePair, 7)
  LBKV_PICK(kModeDup, 6)
  LBKV_PICK(kModePair, 6)
  LBKV_PICK(kModeDup, 5)
  LBKV_PICK(kModePair, 5)
#undef LBKV_PICK
  return nullptr;
}

}  // namespace lbkv
