// lbkv_decode_int4_k0.cu -- instantiations of the split-decode kernel for 4-bit
// codes with a token-wise K side.
#include "lbkv_internal.h"

namespace lbkv {

DecodeKernel decode_kernel_int4_k0(int vl, int nt, int log2g) {
#define LBKV_PICK(VL, NT, LG) \
  if (vl == VL && nt == NT && log2g == LG) return &split_decode_kernel<Cfg<4, 0, VL, NT, LG>>;
  LBKV_PICK(0, 1, 7)
  LBKV_PICK(0, 2, 7)
  LBKV_PICK(0, 1, 6)
  LBKV_PICK(1, 1, 7)
  LBKV_PICK(1, 2, 7)
  LBKV_PICK(1, 1, 6)
  LBKV_PICK(1, 2, 6)
  LBKV_PICK(1, 1, 5)
  LBKV_PICK(1, 2, 5)
#undef LBKV_PICK
  return nullptr;
}

}  // namespace lbkv
