// lbkv_internal.h -- declarations shared by the library's translation units
// (not part of the public interface in include/lbkv.h).
#pragma once

#include "lbkv_decode.cuh"

namespace lbkv {

struct PackArgs {
  const __nv_bfloat16* x;
  const int32_t* seq_lens;
  int B, Hkv, T_cap, bits, layout, group;
  uint8_t* codes;
  __half* scale;
  __half* off;
};

int launch_pack(const PackArgs& a, cudaStream_t stream);

using DecodeKernel = void (*)(const DecodeParams);

// Instantiated kernel for (v_layout, PV n-tiles, log2 group) of one bit width and
// K layout, or nullptr when that combination is not built.
DecodeKernel decode_kernel_int2_k0(int vl, int ntv, int log2g);
DecodeKernel decode_kernel_int2_k1(int vl, int ntv, int log2g);
DecodeKernel decode_kernel_int4_k0(int vl, int ntv, int log2g);
DecodeKernel decode_kernel_int4_k1(int vl, int ntv, int log2g);

}  // namespace lbkv
