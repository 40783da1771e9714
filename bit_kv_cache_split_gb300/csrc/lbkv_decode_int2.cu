// lbkv_decode_int2.cu -- instantiations of the split-decode kernel for 2-bit codes.
#include "lbkv_internal.h"

namespace lbkv {

DecodeKernel decode_kernel_int2(int kl, int vl, int nt, int gv) {
#define LBKV_PICK(KL, VL, NT, GV) \
  if (kl == KL && vl == VL && nt == NT && gv == GV) return &split_decode_kernel<2, KL, VL, NT, GV>;
  LBKV_PICK(0, 0, 1, 1)
  LBKV_PICK(0, 0, 2, 1)
  LBKV_PICK(0, 0, 1, 2)
  LBKV_PICK(1, 0, 1, 1)
  LBKV_PICK(1, 0, 2, 1)
  LBKV_PICK(1, 0, 1, 2)
  LBKV_PICK(0, 1, 1, 1)
  LBKV_PICK(0, 1, 2, 1)
  LBKV_PICK(1, 1, 1, 1)
  LBKV_PICK(1, 1, 2, 1)
#undef LBKV_PICK
  return nullptr;
}

}  // namespace lbkv
