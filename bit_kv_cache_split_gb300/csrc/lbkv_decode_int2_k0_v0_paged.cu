// lbkv_decode_int2_k0_v0_paged.cu -- instantiations of the split-decode kernel for
// 2-bit codes with a token-wise K side and a token-wise V side, over a paged cache.
#define LBKV_PAGED true
#include "lbkv_decode_int2_k0_v0.cu"
