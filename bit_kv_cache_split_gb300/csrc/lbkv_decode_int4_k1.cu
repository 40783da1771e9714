// lbkv_decode_int4_k1.cu -- instantiations of the split-decode kernel for 4-bit
// codes with a channel-wise K side.
#include "lbkv_internal.h"

namespace lbkv {

DecodeKernel decode_kernel_int4_k1(int vl, int ntv, int log2g) {
#define LBKV_PICK(VL, NTV, LG) \
  if (vl == VL && ntv == NTV && log2g == LG) return &split_decode_kernel<Cfg<4, 1, VL, NTV, LG>>;
  LBKV_PICK(0, 1, 7)
  LBKV_PICK(0, 1, 6)
  LBKV_PICK(0, 2, 6)
  LBKV_PICK(0, 1, 5)
  LBKV_PICK(0, 2, 5)
  LBKV_PICK(1, 1, 7)
  LBKV_PICK(1, 1, 6)
  LBKV_PICK(1, 1, 5)
#undef LBKV_PICK
  return nullptr;
}

}  // namespace lbkv
