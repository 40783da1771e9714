// lbkv_rotate.cu -- the normalized Hadamard rotation of bf16 rows of 128 channels, the
// step that stores a cache rotated (an accuracy recipe for 2-bit caches: OSCAR's
// rotations, accuracy paragraph of the explainer "FOSCAR speeds up 2-bit KV decode --
// Affine folding of KV dequantization"; the related explainer "KVarN -- Hadamard-rotated
// 2-bit KV cache"). Decode folds the rotation into the query and the output.
#include "lbkv_internal.h"

namespace lbkv {

// One warp per row: y[r] = bf16(H x[r]) (x and y may be the same array).
__global__ void __launch_bounds__(256) rotate_rows_kernel(const __nv_bfloat16* x, __nv_bfloat16* y, long long rows) {
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;  // the whole warp leaves together
  float v[4];
  load_row4(x + row * kHeadDim, lane, v);
  hadamard128(v, lane);
  store_row4(y + row * kHeadDim, lane, v);
}

int launch_rotate(const __nv_bfloat16* x, __nv_bfloat16* y, long long rows, cudaStream_t stream) {
  if (rows == 0) return 0;
  const unsigned blocks = (unsigned)((rows + 7) / 8);
  rotate_rows_kernel<<<blocks, 256, 0, stream>>>(x, y, rows);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace lbkv
