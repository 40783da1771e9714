// lbkv_internal.h -- declarations shared by the library's translation units
// (not part of the public interface in include/lbkv.h).
#pragma once

#include <cuda.h>  // CUtensorMap (the driver is reached through the runtime's entry points)

#include "lbkv.h"
#include "lbkv_decode.cuh"

namespace lbkv {

// A paged cache (page_table != nullptr): token t of sequence b lives in page
// page_table[b * max_pages + t / page_tokens] of a pool of num_pages pages.
struct PagedArgs {
  const int32_t* page_table;
  int page_tokens, max_pages, num_pages;
};

struct PackArgs {
  const __nv_bfloat16* x;
  const int32_t* seq_lens;
  int B, Hkv, T_cap, bits, layout, group;
  uint8_t* codes;
  __half* scale;
  __half* off;
  PagedArgs pg;
  int32_t* status;  // status word, or nullptr
};

int launch_pack(const PackArgs& a, cudaStream_t stream);

struct AppendArgs {
  const __nv_bfloat16* k_new;  // [B][Hkv][D]
  const __nv_bfloat16* v_new;
  int32_t* seq_lens;           // [B], advanced in place
  __nv_bfloat16* k_win;        // [B][Hkv][win_cap][D] (channel-wise sides only)
  __nv_bfloat16* v_win;
  int32_t* win_lens;           // [B], advanced / reset in place
  int32_t* status;             // status word, or nullptr
  int B, Hkv, T_cap, win_cap, bits, k_layout, v_layout, group;
  uint8_t* k_codes;
  __half* k_scale;
  __half* k_off;
  uint8_t* v_codes;
  __half* v_scale;
  __half* v_off;
  PagedArgs pg;
  int rotation;  // bit 0: store the new K rotated, bit 1: the new V
};

int launch_append(const AppendArgs& a, cudaStream_t stream);

// y[r] = bf16(H x[r]) for rows of 128 channels (H: the normalized Hadamard matrix).
int launch_rotate(const __nv_bfloat16* x, __nv_bfloat16* y, long long rows, cudaStream_t stream);

// BF16 comparator: tokens per chunk (one CTA each), and the arguments of its two kernels.
constexpr int kBfChunk = 512;
struct Bf16Params {
  CUtensorMap tm_k;        // K and V as 2-D tensors [B*Hkv*T_cap rows][128 channels] bf16,
  CUtensorMap tm_v;        //   64 x 64 boxes with the 128-byte swizzle
  const __nv_bfloat16* q;  // [B][Hq][D]
  const __nv_bfloat16* k;  // [B][Hkv][T_cap][D]
  const __nv_bfloat16* v;
  const int32_t* seq_lens;
  float2* part_ml;         // [B*Hkv*max_chunks][hq] chunk partials (max in log2 units, denominator)
  float* part_o;           // [B*Hkv*max_chunks][hq][D]
  int32_t* status;
  __nv_bfloat16* out;      // [B][Hq][D]
  int B, Hq, Hkv, hq, T_cap, max_chunks;
  float sl2;               // softmax scale times log2(e)
};
const void* bf16_split_kernel_fn();
int bf16_split_smem_bytes();
int launch_bf16(const Bf16Params& p, cudaStream_t stream);

// Workspace layout of one lbkv_decode_attn call, from the same plan the call uses: the
// total size (0 when the arguments are invalid or unsupported) and, in *zero_bytes, the
// length of its head (status word and per-pair split counters) that must read zero when
// the call starts.
size_t decode_workspace_plan(const lbkv_desc* desc, int bits, int k_layout, int v_layout, int group,
                             size_t* zero_bytes);

using DecodeKernel = void (*)(const DecodeParams);

// Window partials (one per sequence and KV head) into the last partial slot of each
// pair; launched before the decode kernel when a bf16 window is present.
constexpr int kWinMax = 128;  // window capacity limit (tokens)
int launch_window_partial(const DecodeParams& p, cudaStream_t stream);

// Instantiated kernel for (column mode, log2 group) of one bit width, K/V layout
// pair and cache kind (contiguous or paged), in its cluster mode (one thread-block
// cluster per pair, merged in distributed shared memory) or not, or nullptr when that
// combination is not built. One translation unit per specialisation.
template <int BITS, int KL, int VL, bool PAGED>
DecodeKernel decode_kernel(int mode, int log2g, bool cluster);
#define LBKV_DECLARE_DECODE(B, K, V)                                  \
  template <> DecodeKernel decode_kernel<B, K, V, false>(int, int, bool); \
  template <> DecodeKernel decode_kernel<B, K, V, true>(int, int, bool);
LBKV_DECLARE_DECODE(2, 0, 0)
LBKV_DECLARE_DECODE(2, 0, 1)
LBKV_DECLARE_DECODE(2, 1, 0)
LBKV_DECLARE_DECODE(2, 1, 1)
LBKV_DECLARE_DECODE(4, 0, 0)
LBKV_DECLARE_DECODE(4, 0, 1)
LBKV_DECLARE_DECODE(4, 1, 0)
LBKV_DECLARE_DECODE(4, 1, 1)
#undef LBKV_DECLARE_DECODE


// The tensor-core decode kernel (token-wise K side; QK^T on tcgen05, one product per
// 128-token item shared by a group of four warps) for (column mode, log2 group), or nullptr
// when it does not fit that shape.
template <int BITS, int VL, bool PAGED>
DecodeKernel decode_kernel_grp(int mode, int log2g);
#define LBKV_DECLARE_GRP(B, V)                                        \
  template <> DecodeKernel decode_kernel_grp<B, V, false>(int, int); \
  template <> DecodeKernel decode_kernel_grp<B, V, true>(int, int);
LBKV_DECLARE_GRP(2, 0)
LBKV_DECLARE_GRP(2, 1)
LBKV_DECLARE_GRP(4, 0)
LBKV_DECLARE_GRP(4, 1)
#undef LBKV_DECLARE_GRP

}  // namespace lbkv
