// lbkv_decode_int4_k1_v0_paged.cu -- instantiations of the split-decode kernel for
// 4-bit codes with a channel-wise K side and a token-wise V side, over a paged cache.
#define LBKV_PAGED true
#include "lbkv_decode_int4_k1_v0.cu"
