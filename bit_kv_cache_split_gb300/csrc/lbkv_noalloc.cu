// lbkv_noalloc.cu -- a decode entry point for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc at decode time: code that runs inside an
// inference engine whose allocator owns every byte of device memory, plugins
// that are handed only input and output buffers, and real-time loops where an
// allocation (and its possible implicit synchronization) is not allowed. For
// them the split-KV scratch lives in one fixed array in this library's device
// memory, so the call needs nothing besides its inputs and output.
//
// Cost of that convenience: every GPU that loads the library keeps
// kNoallocScratchBytes of device memory until the process exits, and all calls
// on one device share the array, so calls that overlap on the GPU (two streams,
// two threads) race and corrupt each other's results.
#include <mutex>

#include "lbkv.h"
#include "lbkv_internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = size_t(16) << 20;  // 16 MiB per device
constexpr int kNoallocMaxDevices = 64;

}  // namespace

// The shared scratch. In host code this name is only a stand-in for the symbol,
// never a device address: the address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

namespace {

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoallocMaxDevices];  // device address per device, filled on first use

// Device address of the scratch on the current device (looked up once per device,
// with that device current).
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LBKV_ECUDA;
  if (dev < 0 || dev >= kNoallocMaxDevices) return LBKV_ECUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return LBKV_ECUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return LBKV_OK;
}

}  // namespace

extern "C" {

size_t lbkv_noalloc_scratch_bytes(void) { return kNoallocScratchBytes; }

int lbkv_decode_attn_noalloc(const lbkv_desc* desc, const void* q, const uint8_t* k_codes, const void* k_scale,
                             const void* k_off, const uint8_t* v_codes, const void* v_scale, const void* v_off,
                             const int32_t* seq_lens, int bits, int k_layout, int v_layout, int group, void* out,
                             lbkv_stream_t stream) {
  if (!desc) return LBKV_EINVAL;
  lbkv_desc d = *desc;
  d.workspace = nullptr;
  d.workspace_bytes = 0;
  size_t head = 0;
  const size_t need = lbkv::decode_workspace_plan(&d, bits, k_layout, v_layout, group, &head);
  if (need == 0) {
    // invalid or unsupported arguments: let the regular entry point name the reason
    return lbkv_decode_attn(&d, q, k_codes, k_scale, k_off, v_codes, v_scale, v_off, seq_lens, bits, k_layout,
                            v_layout, group, out, stream);
  }
  if (need > kNoallocScratchBytes) return LBKV_ESCRATCH;
  void* scratch = nullptr;
  const int st = noalloc_scratch(&scratch);
  if (st != LBKV_OK) return st;
  // The status word and the split counters (one per pair of the plan, which splits a KV
  // head into two pairs when it has 32 (query, V group) columns) must start at zero: the
  // plan gives the length of that head of the layout.
  if (cudaMemsetAsync(scratch, 0, head < need ? head : need, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return LBKV_ECUDA;
  d.workspace = scratch;
  d.workspace_bytes = kNoallocScratchBytes;
  return lbkv_decode_attn(&d, q, k_codes, k_scale, k_off, v_codes, v_scale, v_off, seq_lens, bits, k_layout,
                          v_layout, group, out, stream);
}

}  // extern "C"
