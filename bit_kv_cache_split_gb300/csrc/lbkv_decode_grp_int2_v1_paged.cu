// lbkv_decode_grp_int2_v1_paged.cu -- instantiations of the group decode kernel for
// 2-bit codes with a token-wise K side and a channel-wise V side, over a paged cache.
#define LBKV_PAGED true
#include "lbkv_decode_grp_int2_v1.cu"
