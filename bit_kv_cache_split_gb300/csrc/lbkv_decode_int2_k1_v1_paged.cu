// lbkv_decode_int2_k1_v1_paged.cu -- instantiations of the split-decode kernel for
// 2-bit codes with a channel-wise K side and a channel-wise V side, over a paged cache.
#define LBKV_PAGED true
#include "lbkv_decode_int2_k1_v1.cu"
