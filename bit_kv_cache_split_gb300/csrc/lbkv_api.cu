// lbkv_api.cu -- the C ABI (include/lbkv.h): argument validation, split-KV
// planning, workspace layout and kernel launches. Nothing here allocates,
// frees or synchronizes (except lbkv_device_status, documented as such).
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "lbkv.h"
#include "lbkv_internal.h"

using namespace lbkv;

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int> g_smem_optin[kMaxDevices];

int current_device_props(int* sms, int* smem_optin) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LBKV_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return LBKV_ECUDA;
  int s = g_sm_count[dev].load(std::memory_order_relaxed);
  int m = g_smem_optin[dev].load(std::memory_order_relaxed);
  if (s <= 0 || m <= 0) {
    if (cudaDeviceGetAttribute(&s, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return LBKV_ECUDA;
    if (cudaDeviceGetAttribute(&m, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return LBKV_ECUDA;
    g_sm_count[dev].store(s, std::memory_order_relaxed);
    g_smem_optin[dev].store(m, std::memory_order_relaxed);
  }
  *sms = s;
  *smem_optin = m;
  return LBKV_OK;
}

// Opt-in shared memory is set once per (device, kernel): later calls skip the driver call.
std::mutex g_attr_mu;
std::unordered_map<uint64_t, int> g_attr_smem;

int ensure_smem_attr(const void* fn, int bytes, bool big_clusters = false) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LBKV_ECUDA;
  const uint64_t key = ((reinterpret_cast<uint64_t>(fn) << 6) ^ (uint64_t)dev) ^ (big_clusters ? 1ull << 63 : 0ull);
  std::lock_guard<std::mutex> lock(g_attr_mu);
  auto it = g_attr_smem.find(key);
  if (it != g_attr_smem.end() && it->second >= bytes) return LBKV_OK;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return LBKV_ECUDA;
  // clusters of more than 8 CTAs (a non-portable size)
  if (big_clusters && cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    return LBKV_ECUDA;
  g_attr_smem[key] = bytes;
  return LBKV_OK;
}

// Clusters of `cpp` CTAs of kernel fn (with its block size and shared memory) that the
// device holds at once, cached per (device, kernel, cluster size, block size, shared memory).
struct ClusterKey {
  const void* fn;
  int dev, cpp, threads, smem;
  bool operator==(const ClusterKey& o) const {
    return fn == o.fn && dev == o.dev && cpp == o.cpp && threads == o.threads && smem == o.smem;
  }
};
struct ClusterKeyHash {
  size_t operator()(const ClusterKey& k) const {
    uint64_t h = reinterpret_cast<uint64_t>(k.fn);
    for (int v : {k.dev, k.cpp, k.threads, k.smem}) h = h * 0x9E3779B97F4A7C15ull ^ (uint64_t)(uint32_t)v;
    return (size_t)h;
  }
};
std::unordered_map<ClusterKey, int, ClusterKeyHash> g_max_clusters;

int max_active_clusters(const void* fn, int cpp, int threads, int smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const ClusterKey key{fn, dev, cpp, threads, smem};
  {
    std::lock_guard<std::mutex> lock(g_attr_mu);
    auto it = g_max_clusters.find(key);
    if (it != g_max_clusters.end()) return it->second;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cpp);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cpp;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  std::lock_guard<std::mutex> lock(g_attr_mu);
  g_max_clusters[key] = n;
  return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t x, size_t m) { return (x + m - 1) / m * m; }

// A paged cache (page_table given): pages of a power of two of at least 128 tokens (whole
// 128-token slots, so that no kernel item straddles two pages), a non-empty pool and a
// table row with room for max_seq_len tokens.
int paged_check(const lbkv_desc* d) {
  if (!d->page_table) return LBKV_OK;
  if (d->page_tokens < kSlotTokens || (d->page_tokens & (d->page_tokens - 1))) return LBKV_EINVAL;
  if (d->max_pages <= 0 || d->num_pages <= 0) return LBKV_EINVAL;
  if ((long long)d->max_pages * d->page_tokens < d->max_seq_len) return LBKV_EINVAL;
  if ((long long)d->batch * d->max_pages >= (1ll << 31)) return LBKV_EINVAL;
  if (reinterpret_cast<uintptr_t>(d->page_table) & 3u) return LBKV_EALIGN;
  return LBKV_OK;
}

PagedArgs paged_args(const lbkv_desc* d) {
  if (!d->page_table) return PagedArgs{nullptr, 0, 0, 0};
  return PagedArgs{d->page_table, d->page_tokens, d->max_pages, d->num_pages};
}

// Work split: a pair boundary (the segment's prologue, the wait for its slowest warp and
// the merges) costs about as much CTA time as this many cached tokens (16 items of 128
// tokens, 32 of 64). Measured on ragged batches (16 sequences of 1K-64K tokens, INT2
// token-wise): 81.5 us against 100.8 us without the boundary cost.
constexpr int kSplitBoundaryTokens = 2048;

// Shared memory the decode kernels declare statically (the split scan and a few words),
// kept free below the opt-in limit when the rings are sized.
constexpr int kStaticSmemReserve = 2048;

struct Plan {
  int hq, hkv, kv_shift, mode, gv, win;
  int unit_tokens, n_cta;
  int ring_off, ring_per_warp, entry_bytes, smem_bytes, threads;
  size_t off_done, off_ml, off_o, off_wml, off_wo, ws_bytes;
  DecodeKernel tc_fn;  // the tensor-core kernel when it takes the call, else nullptr
  bool grp;            // the tensor-core kernel (rings per group of four warps)
  int cluster_ctas;    // cluster mode: CTAs per pair (one thread-block cluster each), else 0
  int sms;             // SMs of the device
};

// LBKV_DECODE_KERNEL=tc in the environment (read at every call) makes a token-wise K side
// take the tensor-core decode kernel (lbkv_decode_grp.cuh) where it is built for the shape;
// by default every call takes the mma.sync split-decode kernel, which is faster on GB300
// (measured: 164 us against 288 us at batch 32, 32K context, INT2 token-wise g128).
bool tc_kernel_requested() {
  const char* e = std::getenv("LBKV_DECODE_KERNEL");
  return e != nullptr && std::strcmp(e, "tc") == 0;
}

template <bool PAGED>
DecodeKernel pick_grp_of(int bits, int vl, int mode, int lg) {
  if (bits == 2) return vl ? decode_kernel_grp<2, 1, PAGED>(mode, lg) : decode_kernel_grp<2, 0, PAGED>(mode, lg);
  return vl ? decode_kernel_grp<4, 1, PAGED>(mode, lg) : decode_kernel_grp<4, 0, PAGED>(mode, lg);
}


// Validates shapes and format, then fixes the persistent grid and the rings.
int make_plan(const lbkv_desc* d, int bits, int kl, int vl, int group, Plan* pl) {
  if (!d) return LBKV_EINVAL;
  if (d->batch < 0 || d->num_q_heads <= 0 || d->num_kv_heads <= 0) return LBKV_EINVAL;
  if (d->num_q_heads % d->num_kv_heads) return LBKV_EINVAL;
  if (d->head_dim != kHeadDim) return LBKV_EUNSUPPORTED;
  if (d->max_seq_len <= 0 || d->max_seq_len % kSlotTokens) return LBKV_EINVAL;
  if (bits != 2 && bits != 4) return LBKV_EINVAL;
  if ((kl != LBKV_TOKENWISE && kl != LBKV_CHANNELWISE) || (vl != LBKV_TOKENWISE && vl != LBKV_CHANNELWISE))
    return LBKV_EINVAL;
  if (group != 32 && group != 64 && group != 128) return LBKV_EUNSUPPORTED;
  const int hq = d->num_q_heads / d->num_kv_heads;
  if (hq != 1 && hq != 2 && hq != 4 && hq != 8) return LBKV_EUNSUPPORTED;
  const bool win = d->k_win != nullptr;
  if (win != (d->v_win != nullptr) || win != (d->win_lens != nullptr)) return LBKV_EINVAL;
  if (win && (d->win_cap <= 0 || d->win_cap > kWinMax)) return LBKV_EINVAL;
  if (int st = paged_check(d)) return st;
  if (d->rotation & ~(LBKV_ROTATE_K | LBKV_ROTATE_V)) return LBKV_EINVAL;
  // PV columns are (query, V channel group) pairs: a token-wise V side with G channel
  // groups feeds G separately scaled copies of the weights (operand-fold); the kernel
  // holds at most two PV n-tiles of 8 columns.
  const int groups_v = (vl == LBKV_TOKENWISE) ? kHeadDim / group : 1;
  pl->gv = groups_v;
  // 32 pairs (token-wise V with 4 groups, 8 queries per KV head): each KV head is split in
  // two halves of its queries that read the same cached data (16 pairs each)
  pl->kv_shift = (hq * groups_v > 16) ? 1 : 0;
  pl->hq = hq >> pl->kv_shift;
  pl->hkv = d->num_kv_heads << pl->kv_shift;
  pl->mode = decode_mode(pl->hq * groups_v);
  if (pl->mode < 0) return LBKV_EUNSUPPORTED;

  int sms = 0, smem_optin = 0;
  int st = current_device_props(&sms, &smem_optin);
  if (st) return st;

  const int lg = group == 128 ? 7 : group == 64 ? 6 : 5;
  // With LBKV_DECODE_KERNEL=tc a token-wise K side takes the tensor-core kernel (items of 128
  // tokens, a ring per group of four warps with at least two entries) where it is built for
  // the shape; every other call takes the split-decode kernel.
  const int warps = decode_warps(bits, pl->mode, pl->gv);
  pl->tc_fn = nullptr;
  pl->grp = false;
  if (kl == LBKV_TOKENWISE && tc_kernel_requested()) {
    DecodeKernel fn = d->page_table ? pick_grp_of<true>(bits, vl, pl->mode, lg) : pick_grp_of<false>(bits, vl, pl->mode, lg);
    if (fn) {
      const int groups = warps / 4;
      const EntryLayout el = entry_layout(bits, kl, vl, 128, group);
      const int ring_off = (int)round_up((size_t)kGrpMergeOffset + merge_bytes(pl->hq, warps), 128);
      int r = (smem_optin - kStaticSmemReserve - ring_off) / (groups * el.bytes);
      if (r > 12) r = 12;
      if (r >= 2) {
        pl->tc_fn = fn;
        pl->grp = true;
        pl->unit_tokens = 128;
        pl->entry_bytes = el.bytes;
        pl->threads = 32 * warps;
        pl->ring_off = ring_off;
        pl->ring_per_warp = r;
        pl->smem_bytes = ring_off + groups * r * el.bytes;
      }
    }
  }
  if (!pl->grp) {
    // ring entry: one item of `ut` tokens, K half then V half
    const int ut = kChunk * unit_chunks(bits, pl->mode, lg);
    const EntryLayout el = entry_layout(bits, kl, vl, ut, group);
    pl->unit_tokens = ut;
    pl->entry_bytes = el.bytes;
    pl->threads = 32 * warps;
    pl->ring_off = kPrologueBytes + merge_bytes(pl->hq, warps);
    const int budget = smem_optin - kStaticSmemReserve - pl->ring_off;
    int r_w = budget / (warps * pl->entry_bytes);
    if (r_w > kMaxRing / (2 * warps)) r_w = kMaxRing / (2 * warps);  // two mbarriers per entry
    if (r_w < 1) return LBKV_EUNSUPPORTED;
    pl->ring_per_warp = r_w;
    pl->smem_bytes = pl->ring_off + warps * r_w * pl->entry_bytes;
  }
  const int ut = pl->unit_tokens;

  // Persistent grid, one CTA per SM: the kernel splits the items of all pairs (from the
  // device lengths) over the CTAs, evenly once each pair boundary is counted as
  // kSplitBoundaryTokens of work. A CTA holds partials of at most two pairs.
  const long long units = (long long)d->batch * pl->hkv;  // pairs
  pl->win = win ? 1 : 0;
  // Small problems: about one item per warp at most (from the capacity, the host's bound on
  // the device lengths), so that a pair is split over fewer CTAs and their partials merge
  // sooner. Measured on batch 8 at 4K context: 18.3 us against 24.7 us with every SM.
  {
    const long long max_items = units * (((long long)d->max_seq_len + ut - 1) / ut);
    const int units_per_cta = pl->grp ? warps / 4 : warps;  // warps, or groups of four
    const long long want = (max_items + units_per_cta - 1) / units_per_cta;
    pl->n_cta = (int)(want < sms ? (want > 0 ? want : 1) : sms);
    pl->sms = sms;
    // With a window and few pairs, the window kernel's CTAs (one per pair, launched first)
    // hold their SMs while the decode kernel starts: the grid leaves those SMs out, so that
    // no decode CTA waits for one of them to finish.
    if (win && units * 16 <= sms && pl->n_cta > sms - units) pl->n_cta = (int)(sms - units);
  }
  // Cluster mode: with few pairs (at most half as many as SMs), one thread-block cluster of
  // up to cluster_ctas CTAs per pair (a power of two from 2 to 16: no more than about one item
  // per warp from the capacity, but at least 4 where the pairs allow it, and all CTAs in one
  // wave; the launch lowers it until the GPU holds all clusters at once and takes the mode only
  // where it costs a warp at most one item more); its CTAs merge their partials in
  // distributed shared memory instead of through the workspace, with no length scan.
  pl->cluster_ctas = 0;
  if (!pl->grp && units * 2 <= sms) {
    const long long items_pair = ((long long)d->max_seq_len + ut - 1) / ut;
    int cpp = 16;
    while (cpp > 4 && (long long)(cpp / 2) * warps >= items_pair) cpp >>= 1;  // short pairs
    while (cpp > 2 && units * cpp > sms) cpp >>= 1;                           // one wave
    pl->cluster_ctas = cpp;
  }

  // workspace: status word | per-pair counters | CTA partials (m, l) | CTA partials O |
  // window partials (m, l) | window partials O
  const size_t rows = (size_t)pl->n_cta * 2 * pl->hq, wrows = pl->win ? (size_t)units * pl->hq : 0;
  pl->off_done = 256;
  pl->off_ml = round_up(pl->off_done + (size_t)units * sizeof(int32_t), 256);
  pl->off_o = round_up(pl->off_ml + rows * sizeof(float2), 256);
  pl->off_wml = round_up(pl->off_o + rows * kHeadDim * sizeof(float), 256);
  pl->off_wo = round_up(pl->off_wml + wrows * sizeof(float2), 256);
  pl->ws_bytes = round_up(pl->off_wo + wrows * kHeadDim * sizeof(float), 256);
  return LBKV_OK;
}

template <bool PAGED>
DecodeKernel pick_kernel_of(int bits, int kl, int vl, int mode, int lg, bool cl) {
  if (bits == 2) {
    if (kl == 0)
      return vl ? decode_kernel<2, 0, 1, PAGED>(mode, lg, cl) : decode_kernel<2, 0, 0, PAGED>(mode, lg, cl);
    return vl ? decode_kernel<2, 1, 1, PAGED>(mode, lg, cl) : decode_kernel<2, 1, 0, PAGED>(mode, lg, cl);
  }
  if (kl == 0) return vl ? decode_kernel<4, 0, 1, PAGED>(mode, lg, cl) : decode_kernel<4, 0, 0, PAGED>(mode, lg, cl);
  return vl ? decode_kernel<4, 1, 1, PAGED>(mode, lg, cl) : decode_kernel<4, 1, 0, PAGED>(mode, lg, cl);
}

DecodeKernel pick_kernel(int bits, int kl, int vl, int mode, int group, bool paged, bool cluster = false) {
  const int lg = group == 128 ? 7 : group == 64 ? 6 : 5;
  return paged ? pick_kernel_of<true>(bits, kl, vl, mode, lg, cluster)
               : pick_kernel_of<false>(bits, kl, vl, mode, lg, cluster);
}

}  // namespace

namespace lbkv {

size_t decode_workspace_plan(const lbkv_desc* desc, int bits, int k_layout, int v_layout, int group,
                             size_t* zero_bytes) {
  Plan pl;
  if (make_plan(desc, bits, k_layout, v_layout, group, &pl) != LBKV_OK) return 0;
  if (zero_bytes) *zero_bytes = pl.off_ml;
  return pl.ws_bytes;
}

}  // namespace lbkv

// Cluster mode: the kernel, CTAs per cluster and clusters per pair a call takes, or no kernel
// (the split-decode grid). A device that cannot hold the clusters takes the split-decode grid.
struct ClusterChoice {
  DecodeKernel fn = nullptr;
  int cpp = 0, split = 1;
};
ClusterChoice choose_clusters(const lbkv_desc* desc, const Plan& pl, int bits, int k_layout, int v_layout,
                              int group) {
  ClusterChoice ch;
  if (pl.cluster_ctas <= 0 || pl.tc_fn) return ch;
  DecodeKernel kc = pick_kernel(bits, k_layout, v_layout, pl.mode, group, desc->page_table != nullptr, true);
  if (!kc || ensure_smem_attr(reinterpret_cast<const void*>(kc), pl.smem_bytes, true) != LBKV_OK) return ch;
  const long long units = (long long)desc->batch * pl.hkv;
  // the largest cluster size (down to 2) whose clusters, one per pair, the device holds at once
  int cpp = pl.cluster_ctas;
  while (cpp >= 2 && max_active_clusters(reinterpret_cast<const void*>(kc), cpp, pl.threads, pl.smem_bytes) < units)
    cpp >>= 1;
  // Taken only when it gives a warp at most one item more than the split-decode grid (an
  // item costs a warp about 4.6 us among 16, the cluster merge saves about 6 us of fixed
  // costs). Measured (graph replay, INT2): batch 8 at 16K 32.1 -> 26.8 us and at 32K 47.9 ->
  // 44.7 us with clusters of 2, but at 64K 77.9 -> 80.5 us and at 128K 140.4 -> 152.4 us (two
  // and more items more per warp). Clusters of 16 CTAs of this size fit 7 at a time, of 8
  // CTAs 15, of 4 CTAs 36.
  const long long wpc = pl.threads / 32;  // warps per CTA
  const long long items_pair = ((long long)desc->max_seq_len + pl.unit_tokens - 1) / pl.unit_tokens;
  const long long ipw_split = (units * items_pair + (long long)pl.n_cta * wpc - 1) / ((long long)pl.n_cta * wpc);
  const long long ipw_cluster = (items_pair + (long long)cpp * wpc - 1) / ((long long)cpp * wpc);
  bool take = cpp >= 2 && ipw_cluster <= ipw_split + 1;
  // Two levels: several clusters per pair (each merges its CTAs in distributed shared memory
  // and writes one partial; the pair's last cluster merges those), where that gives a warp
  // fewer items than one cluster per pair and no more than the split-decode grid. The
  // partials take CTA-partial rows of the workspace (2 per CTA of the split-decode grid).
  int split = 1;
  long long best = take ? ipw_cluster : ipw_split + 1;
  for (int c2 = 16; c2 >= 2; c2 >>= 1) {  // (larger clusters first: fewer partials per pair)
    for (int s2 = 2; s2 <= 16; ++s2) {
      if (units * c2 * s2 > pl.sms || units * s2 > 2LL * pl.n_cta) continue;
      const long long ipw2 = (items_pair + (long long)c2 * s2 * wpc - 1) / ((long long)c2 * s2 * wpc);
      if (ipw2 >= best || ipw2 > ipw_split) continue;
      if (max_active_clusters(reinterpret_cast<const void*>(kc), c2, pl.threads, pl.smem_bytes) < units * s2)
        continue;
      best = ipw2;
      cpp = c2;
      split = s2;
      take = true;
    }
  }
  if (take) {
    ch.fn = kc;
    ch.cpp = cpp;
    ch.split = split;
  }
  return ch;
}

extern "C" {

size_t lbkv_workspace_bytes(const lbkv_desc* desc, int bits, int k_layout, int v_layout, int group) {
  Plan pl;
  if (make_plan(desc, bits, k_layout, v_layout, group, &pl) != LBKV_OK) return 0;
  return pl.ws_bytes;
}

int lbkv_decode_attn(const lbkv_desc* desc, const void* q, const uint8_t* k_codes, const void* k_scale,
                     const void* k_off, const uint8_t* v_codes, const void* v_scale, const void* v_off,
                     const int32_t* seq_lens, int bits, int k_layout, int v_layout, int group, void* out,
                     lbkv_stream_t stream) {
  Plan pl;
  int st = make_plan(desc, bits, k_layout, v_layout, group, &pl);
  if (st) return st;
  if (desc->batch == 0) return LBKV_OK;
  const void* ptrs[] = {q, k_codes, k_scale, k_off, v_codes, v_scale, v_off, seq_lens, out};
  for (const void* p : ptrs)
    if (!p) return LBKV_EINVAL;
  for (const void* p : ptrs)
    if (!aligned16(p)) return LBKV_EALIGN;
  if (desc->k_win && (!aligned16(desc->k_win) || !aligned16(desc->v_win))) return LBKV_EALIGN;
  if (!desc->workspace || desc->workspace_bytes < pl.ws_bytes) return LBKV_EWORKSPACE;
  if (reinterpret_cast<uintptr_t>(desc->workspace) & 255u) return LBKV_EALIGN;
  DecodeKernel kern = pl.tc_fn ? pl.tc_fn
                               : pick_kernel(bits, k_layout, v_layout, pl.mode, group, desc->page_table != nullptr);
  if (!kern) return LBKV_EUNSUPPORTED;

  uint8_t* ws = static_cast<uint8_t*>(desc->workspace);
  DecodeParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k_codes = k_codes;
  p.k_scale = static_cast<const __half*>(k_scale);
  p.k_off = static_cast<const __half*>(k_off);
  p.v_codes = v_codes;
  p.v_scale = static_cast<const __half*>(v_scale);
  p.v_off = static_cast<const __half*>(v_off);
  p.seq_lens = seq_lens;
  p.k_win = static_cast<const __nv_bfloat16*>(desc->k_win);
  p.v_win = static_cast<const __nv_bfloat16*>(desc->v_win);
  p.win_lens = desc->win_lens;
  p.part_ml = reinterpret_cast<float2*>(ws + pl.off_ml);
  p.part_o = reinterpret_cast<float*>(ws + pl.off_o);
  p.win_ml = reinterpret_cast<float2*>(ws + pl.off_wml);
  p.win_o = reinterpret_cast<float*>(ws + pl.off_wo);
  p.status = reinterpret_cast<int32_t*>(ws);
  p.done = reinterpret_cast<int32_t*>(ws + pl.off_done);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.B = desc->batch;
  p.Hq = desc->num_q_heads;
  p.Hkv = pl.hkv;
  p.hq = pl.hq;
  p.kv_shift = pl.kv_shift;
  p.T_cap = desc->max_seq_len;
  p.win_cap = desc->k_win ? desc->win_cap : 0;
  const float sigma = desc->sm_scale > 0.f ? desc->sm_scale : 1.f / std::sqrt((float)desc->head_dim);
  p.sl2 = sigma * 1.4426950408889634f;
  p.n_cta = pl.n_cta;
  p.split_w = kSplitBoundaryTokens / pl.unit_tokens;
  p.cluster_split = 1;
  p.has_win = pl.win;
  p.ring_off = pl.ring_off;
  p.ring_per_warp = pl.ring_per_warp;
  p.rotation = desc->rotation;
  p.page_table = desc->page_table;
  if (desc->page_table) {
    p.log2_page = 0;
    while ((1 << p.log2_page) < desc->page_tokens) ++p.log2_page;
    p.max_pages = desc->max_pages;
    p.num_pages = desc->num_pages;
  }

  if (ensure_smem_attr(reinterpret_cast<const void*>(kern), pl.smem_bytes) != LBKV_OK) return LBKV_ECUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (pl.win && launch_window_partial(p, s) != 0) return LBKV_ECUDA;
  // With a window the decode kernel is a programmatic dependent of the window kernel: it
  // starts while the window is scored and waits for it only where it reads its partials.
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3((unsigned)pl.threads);
  cfg.dynamicSmemBytes = (size_t)pl.smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  const ClusterChoice cc = choose_clusters(desc, pl, bits, k_layout, v_layout, group);
  if (cc.fn) {  // cluster mode (if the launch fails, the split-decode grid takes the call)
    const int n = (int)((long long)desc->batch * pl.hkv * cc.cpp * cc.split);
    DecodeParams pc = p;
    pc.n_cta = n;
    pc.cluster_split = cc.split;
    cfg.gridDim = dim3((unsigned)n);
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)cc.cpp;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    if (pl.win) {
      cfg.numAttrs = 2;
    } else {
      attr[0] = attr[1];
      cfg.numAttrs = 1;
    }
    if (cudaLaunchKernelEx(&cfg, cc.fn, pc) == cudaSuccess && cudaGetLastError() == cudaSuccess) return LBKV_OK;
    (void)cudaGetLastError();
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
  }
  cfg.gridDim = dim3((unsigned)pl.n_cta);
  cfg.numAttrs = pl.win ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return LBKV_ECUDA;
  if (cudaGetLastError() != cudaSuccess) return LBKV_ECUDA;
  return LBKV_OK;
}

int lbkv_decode_launch_info(const lbkv_desc* desc, int bits, int k_layout, int v_layout, int group, int* grid,
                            int* cluster, int* split) {
  if (!grid || !cluster || !split) return LBKV_EINVAL;
  Plan pl;
  int st = make_plan(desc, bits, k_layout, v_layout, group, &pl);
  if (st) return st;
  *grid = pl.n_cta;
  *cluster = 0;
  *split = 1;
  if (desc->batch == 0) {
    *grid = 0;
    return LBKV_OK;
  }
  const ClusterChoice cc = choose_clusters(desc, pl, bits, k_layout, v_layout, group);
  if (cc.fn) {
    *grid = (int)((long long)desc->batch * pl.hkv * cc.cpp * cc.split);
    *cluster = cc.cpp;
    *split = cc.split;
  }
  return LBKV_OK;
}

int lbkv_pack(const lbkv_desc* desc, const void* x, const int32_t* seq_lens, int bits, int layout, int group,
              uint8_t* codes, void* scale, void* off, lbkv_stream_t stream) {
  if (!desc) return LBKV_EINVAL;
  if (desc->batch < 0 || desc->num_kv_heads <= 0) return LBKV_EINVAL;
  if (desc->head_dim != kHeadDim) return LBKV_EUNSUPPORTED;
  if (desc->max_seq_len <= 0 || desc->max_seq_len % kSlotTokens) return LBKV_EINVAL;
  if (bits != 2 && bits != 4) return LBKV_EINVAL;
  if (layout != LBKV_TOKENWISE && layout != LBKV_CHANNELWISE) return LBKV_EINVAL;
  if (group != 32 && group != 64 && group != 128) return LBKV_EUNSUPPORTED;
  if (int st = paged_check(desc)) return st;
  if (desc->batch == 0) return LBKV_OK;
  const void* ptrs[] = {x, seq_lens, codes, scale, off};
  for (const void* p : ptrs)
    if (!p) return LBKV_EINVAL;
  for (const void* p : ptrs)
    if (!aligned16(p)) return LBKV_EALIGN;
  if (desc->workspace && (reinterpret_cast<uintptr_t>(desc->workspace) & 255u)) return LBKV_EALIGN;
  PackArgs a{static_cast<const __nv_bfloat16*>(x), seq_lens, desc->batch, desc->num_kv_heads, desc->max_seq_len,
             bits, layout, group, codes, static_cast<__half*>(scale), static_cast<__half*>(off), paged_args(desc),
             desc->workspace ? static_cast<int32_t*>(desc->workspace) : nullptr};
  if (launch_pack(a, reinterpret_cast<cudaStream_t>(stream)) != 0) return LBKV_ECUDA;
  return LBKV_OK;
}

int lbkv_append(const lbkv_desc* desc, const void* k_new, const void* v_new, int32_t* seq_lens, int bits,
                int k_layout, int v_layout, int group, uint8_t* k_codes, void* k_scale, void* k_off,
                uint8_t* v_codes, void* v_scale, void* v_off, lbkv_stream_t stream) {
  if (!desc) return LBKV_EINVAL;
  if (desc->batch < 0 || desc->num_kv_heads <= 0) return LBKV_EINVAL;
  if (desc->head_dim != kHeadDim) return LBKV_EUNSUPPORTED;
  if (desc->max_seq_len <= 0 || desc->max_seq_len % kSlotTokens) return LBKV_EINVAL;
  if (bits != 2 && bits != 4) return LBKV_EINVAL;
  if ((k_layout != LBKV_TOKENWISE && k_layout != LBKV_CHANNELWISE) ||
      (v_layout != LBKV_TOKENWISE && v_layout != LBKV_CHANNELWISE))
    return LBKV_EINVAL;
  if (group != 32 && group != 64 && group != 128) return LBKV_EUNSUPPORTED;
  const bool windowed = k_layout == LBKV_CHANNELWISE || v_layout == LBKV_CHANNELWISE;
  const bool win = desc->k_win != nullptr;
  if (win != (desc->v_win != nullptr) || win != (desc->win_lens != nullptr)) return LBKV_EINVAL;
  if (windowed && (!win || desc->win_cap < group || desc->win_cap > kWinMax)) return LBKV_EINVAL;
  if (int st = paged_check(desc)) return st;
  if (desc->rotation & ~(LBKV_ROTATE_K | LBKV_ROTATE_V)) return LBKV_EINVAL;
  if (desc->batch == 0) return LBKV_OK;
  const void* ptrs[] = {k_new, v_new, seq_lens, k_codes, k_scale, k_off, v_codes, v_scale, v_off};
  for (const void* p : ptrs)
    if (!p) return LBKV_EINVAL;
  for (const void* p : ptrs)
    if (!aligned16(p)) return LBKV_EALIGN;
  if (windowed && (!aligned16(desc->k_win) || !aligned16(desc->v_win) || !aligned16(desc->win_lens)))
    return LBKV_EALIGN;
  if (desc->workspace && (reinterpret_cast<uintptr_t>(desc->workspace) & 255u)) return LBKV_EALIGN;
  AppendArgs a{};
  a.k_new = static_cast<const __nv_bfloat16*>(k_new);
  a.v_new = static_cast<const __nv_bfloat16*>(v_new);
  a.seq_lens = seq_lens;
  a.k_win = windowed ? static_cast<__nv_bfloat16*>(const_cast<void*>(desc->k_win)) : nullptr;
  a.v_win = windowed ? static_cast<__nv_bfloat16*>(const_cast<void*>(desc->v_win)) : nullptr;
  a.win_lens = windowed ? const_cast<int32_t*>(desc->win_lens) : nullptr;
  a.status = desc->workspace ? static_cast<int32_t*>(desc->workspace) : nullptr;
  a.B = desc->batch;
  a.Hkv = desc->num_kv_heads;
  a.T_cap = desc->max_seq_len;
  a.win_cap = windowed ? desc->win_cap : 0;
  a.bits = bits;
  a.k_layout = k_layout;
  a.v_layout = v_layout;
  a.group = group;
  a.k_codes = k_codes;
  a.k_scale = static_cast<__half*>(k_scale);
  a.k_off = static_cast<__half*>(k_off);
  a.v_codes = v_codes;
  a.v_scale = static_cast<__half*>(v_scale);
  a.v_off = static_cast<__half*>(v_off);
  a.pg = paged_args(desc);
  a.rotation = desc->rotation;
  if (launch_append(a, reinterpret_cast<cudaStream_t>(stream)) != 0) return LBKV_ECUDA;
  return LBKV_OK;
}

// BF16 comparator: its K/V tensor maps, encoded through the driver entry point that the
// runtime hands out (no link against the driver library).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
static EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}
static bool kv_tensor_map(CUtensorMap* m, const void* base, uint64_t rows) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// BF16 comparator: status word | chunk partials (m, l) | chunk partials O.
static int bf16_layout(const lbkv_desc* d, size_t* off_ml, size_t* off_o, size_t* bytes, int* max_chunks) {
  if (!d) return LBKV_EINVAL;
  if (d->batch < 0 || d->num_q_heads <= 0 || d->num_kv_heads <= 0) return LBKV_EINVAL;
  if (d->num_q_heads % d->num_kv_heads) return LBKV_EINVAL;
  if (d->head_dim != kHeadDim) return LBKV_EUNSUPPORTED;
  if (d->max_seq_len <= 0 || d->max_seq_len % kSlotTokens) return LBKV_EINVAL;
  const int hq = d->num_q_heads / d->num_kv_heads;
  if (hq > kMaxHq) return LBKV_EUNSUPPORTED;
  if (d->k_win || d->v_win || d->win_lens) return LBKV_EUNSUPPORTED;  // the comparator has no window
  if (d->page_table || d->rotation) return LBKV_EUNSUPPORTED;          // nor a paged or rotated cache
  if ((long long)d->batch * d->num_kv_heads * d->max_seq_len >= (1ll << 31)) return LBKV_EUNSUPPORTED;  // TMA rows
  *max_chunks = (d->max_seq_len + kBfChunk - 1) / kBfChunk;
  const size_t rows = (size_t)d->batch * d->num_kv_heads * (size_t)*max_chunks * hq;
  *off_ml = 256;
  *off_o = round_up(*off_ml + rows * sizeof(float2), 256);
  *bytes = round_up(*off_o + rows * kHeadDim * sizeof(float), 256);
  return LBKV_OK;
}

int lbkv_rotate(const void* x, void* y, int64_t rows, int head_dim, lbkv_stream_t stream) {
  if (head_dim != kHeadDim) return LBKV_EUNSUPPORTED;
  if (rows < 0 || rows > (int64_t)0x7fffffff * 8) return LBKV_EINVAL;
  if (rows == 0) return LBKV_OK;
  if (!x || !y) return LBKV_EINVAL;
  if (!aligned16(x) || !aligned16(y)) return LBKV_EALIGN;
  if (launch_rotate(static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y), (long long)rows,
                    reinterpret_cast<cudaStream_t>(stream)) != 0)
    return LBKV_ECUDA;
  return LBKV_OK;
}

size_t lbkv_bf16_workspace_bytes(const lbkv_desc* desc) {
  size_t a, b, n;
  int mc;
  return bf16_layout(desc, &a, &b, &n, &mc) == LBKV_OK ? n : 0;
}

int lbkv_decode_bf16(const lbkv_desc* desc, const void* q, const void* k, const void* v, const int32_t* seq_lens,
                     void* out, lbkv_stream_t stream) {
  size_t off_ml, off_o, bytes;
  int max_chunks;
  int st = bf16_layout(desc, &off_ml, &off_o, &bytes, &max_chunks);
  if (st) return st;
  if (desc->batch == 0) return LBKV_OK;
  const void* ptrs[] = {q, k, v, seq_lens, out};
  for (const void* p : ptrs)
    if (!p) return LBKV_EINVAL;
  for (const void* p : ptrs)
    if (!aligned16(p)) return LBKV_EALIGN;
  if (!desc->workspace || desc->workspace_bytes < bytes) return LBKV_EWORKSPACE;
  if (reinterpret_cast<uintptr_t>(desc->workspace) & 255u) return LBKV_EALIGN;
  if (ensure_smem_attr(bf16_split_kernel_fn(), bf16_split_smem_bytes()) != LBKV_OK) return LBKV_ECUDA;
  uint8_t* ws = static_cast<uint8_t*>(desc->workspace);
  Bf16Params p{};
  const uint64_t rows = (uint64_t)desc->batch * desc->num_kv_heads * desc->max_seq_len;
  if (!kv_tensor_map(&p.tm_k, k, rows) || !kv_tensor_map(&p.tm_v, v, rows)) return LBKV_ECUDA;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.seq_lens = seq_lens;
  p.part_ml = reinterpret_cast<float2*>(ws + off_ml);
  p.part_o = reinterpret_cast<float*>(ws + off_o);
  p.status = reinterpret_cast<int32_t*>(ws);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.B = desc->batch;
  p.Hq = desc->num_q_heads;
  p.Hkv = desc->num_kv_heads;
  p.hq = desc->num_q_heads / desc->num_kv_heads;
  p.T_cap = desc->max_seq_len;
  p.max_chunks = max_chunks;
  const float sigma = desc->sm_scale > 0.f ? desc->sm_scale : 1.f / std::sqrt((float)desc->head_dim);
  p.sl2 = sigma * 1.4426950408889634f;
  if (launch_bf16(p, reinterpret_cast<cudaStream_t>(stream)) != 0) return LBKV_ECUDA;
  return LBKV_OK;
}

int lbkv_device_status(const lbkv_desc* desc, lbkv_stream_t stream, int32_t* code) {
  if (!desc) return LBKV_EINVAL;
  if (!desc->workspace || desc->workspace_bytes < 256) return LBKV_EWORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t host = 0;
  if (cudaMemcpyAsync(&host, desc->workspace, sizeof(host), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return LBKV_ECUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return LBKV_ECUDA;
  if (code) *code = host;
  if (host != 0) {
    if (cudaMemsetAsync(desc->workspace, 0, sizeof(int32_t), s) != cudaSuccess) return LBKV_ECUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return LBKV_ECUDA;
    return LBKV_EDEVICE;
  }
  return LBKV_OK;
}

const char* lbkv_strerror(int status) {
  switch (status) {
    case LBKV_OK: return "success";
    case LBKV_EINVAL: return "invalid argument (null pointer, size or range)";
    case LBKV_EALIGN: return "pointer not aligned (16 bytes; workspace 256 bytes)";
    case LBKV_EUNSUPPORTED: return "valid but unsupported combination of shape and format";
    case LBKV_EWORKSPACE: return "workspace missing or smaller than lbkv_workspace_bytes";
    case LBKV_ECUDA: return "CUDA launch or runtime error";
    case LBKV_EDEVICE: return "a kernel reported a device-side error (a bounded wait ran out, or an appended token did not fit)";
    case LBKV_ESCRATCH: return "the call needs more scratch than the fixed no-allocation array holds";
    default: return "unknown status";
  }
}

}  // extern "C"
