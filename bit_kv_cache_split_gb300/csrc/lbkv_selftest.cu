// lbkv_selftest.cu -- a self-test of the bounded waits: one warp waits on an mbarrier
// that nothing completes and must give up after the given time, recording the status
// code in the status word, so that the context stays usable.
#include "lbkv.h"
#include "lbkv_internal.h"

namespace lbkv {

__global__ void __launch_bounds__(32, 1) wait_timeout_selftest_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_addr(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);  // one arrival expected; none comes
    mbar_init_fence();
  }
  __syncwarp();
  // phase 0 never completes: the wait runs out after limit_ns
  if (!mbar_wait(b, 0, status, kStatusConsumerTimeout, limit_ns) && threadIdx.x == 0)
    atomicAdd(status + 1, 1);  // the kernel went on past the failed wait
}

}  // namespace lbkv

extern "C" {

int lbkv_selftest_wait_timeout(void* status, uint64_t limit_ns, lbkv_stream_t stream) {
  if (!status || limit_ns == 0 || limit_ns > lbkv::kWaitLimitNs) return LBKV_EINVAL;
  if (reinterpret_cast<uintptr_t>(status) & 15u) return LBKV_EALIGN;
  lbkv::wait_timeout_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<int32_t*>(status), limit_ns);
  return cudaGetLastError() == cudaSuccess ? LBKV_OK : LBKV_ECUDA;
}

}  // extern "C"
