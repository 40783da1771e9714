// lbkv_rotate.cu -- the normalized Hadamard rotation of bf16 rows of 128 channels, the
// step that stores a cache rotated (an accuracy recipe for 2-bit caches: OSCAR's
// rotations, accuracy paragraph of the explainer "FOSCAR speeds up 2-bit KV decode --
// Affine folding of KV dequantization"; the related explainer "KVarN -- Hadamard-rotated
// 2-bit KV cache"). Decode folds the rotation into the query and the output.
#include "lbkv_internal.h"

namespace lbkv {

constexpr int kRotRows = 4;  // rows per warp: their loads are all in flight before the first butterfly

// Each warp rotates rows r0 .. r0 + kRotRows - 1: y[r] = bf16(H x[r]) (x and y may be the
// same array: a row is read whole before it is written, by the same warp).
__global__ void __launch_bounds__(256) rotate_rows_kernel(const __nv_bfloat16* x, __nv_bfloat16* y, long long rows) {
  const long long r0 = ((long long)blockIdx.x * 8 + (threadIdx.x >> 5)) * kRotRows;
  const int lane = threadIdx.x & 31;
  float v[kRotRows][4];
#pragma unroll
  for (int k = 0; k < kRotRows; ++k)
    if (r0 + k < rows) load_row4(x + (r0 + k) * kHeadDim, lane, v[k]);  // the whole warp takes a row or not
#pragma unroll
  for (int k = 0; k < kRotRows; ++k) {
    if (r0 + k >= rows) break;
    hadamard128(v[k], lane);
    store_row4(y + (r0 + k) * kHeadDim, lane, v[k]);
  }
}

int launch_rotate(const __nv_bfloat16* x, __nv_bfloat16* y, long long rows, cudaStream_t stream) {
  if (rows == 0) return 0;
  const unsigned blocks = (unsigned)((rows + 8 * kRotRows - 1) / (8 * kRotRows));
  rotate_rows_kernel<<<blocks, 256, 0, stream>>>(x, y, rows);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace lbkv
