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

// Instantiated kernel for (bits, k_layout, v_layout, n-tiles, V groups), or nullptr.
DecodeKernel decode_kernel_int2(int kl, int vl, int nt, int gv);
DecodeKernel decode_kernel_int4(int kl, int vl, int nt, int gv);

}  // namespace lbkv
