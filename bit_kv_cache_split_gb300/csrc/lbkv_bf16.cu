// lbkv_bf16.cu -- the BF16 comparator: the same split-KV decode attention over a bf16
// cache (no quantization), on the same GPU and pipeline, so that the speedup the pages
// report over a BF16 decode kernel ("FOSCAR: Accelerating Decode Attention over 2- and
// 4-Bit KV Caches through Affine Folding", abstract: the comparison with FlashInfer BF16)
// can be measured here.
//
// Each CTA takes a chunk of kBfChunk tokens of one (sequence, KV head) pair and streams
// it in 64-token tiles through a 3-stage shared-memory ring: per tile four 2-D TMA boxes
// (K and V, channels 0-63 and 64-127, 64 rows of 128 bytes each) with the 128-byte swizzle,
// which the fragment loads undo, so that they are free of bank conflicts. A warp owns 16
// tokens of each tile:
//   S^T = Q K^T on mma.sync m16n8k16 bf16 (rows = queries, padded to 16; K as the B
//   operand, read straight from its rows), online softmax in fp32 (exp2, sigma log2 e
//   folded), O += P V with P reused from registers as the A operand and V loaded
//   transposed by ldmatrix.
// The warps merge into one partial per chunk; a small kernel merges the chunks.
#include "lbkv_internal.h"

namespace lbkv {

constexpr int kBfTile = 64;                       // tokens per stage
constexpr int kBfStages = 3;
constexpr int kBfWarps = 4;                       // 16 tokens of each tile per warp
constexpr int kBfHalfBytes = kBfTile * 128;       // one box: 64 rows x 64 channels (bf16)
constexpr int kBfStageBytes = 4 * kBfHalfBytes;   // K channels 0-63, K 64-127, V 0-63, V 64-127
constexpr int kBfSmem = kBfStages * kBfStageBytes;

// Byte offset of (row r, channel ch) in one side (K or V) of a stage: the half of ch, then
// the row, then its 16-byte chunk j placed at j ^ (r mod 8) (the TMA 128-byte swizzle).
__device__ __forceinline__ int swz(int r, int ch) {
  const int cc = ch & 63;
  return (ch >> 6) * kBfHalfBytes + r * 128 + ((((cc >> 3) ^ (r & 7))) << 4) + ((cc & 7) << 1);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint32_t bf16x2_from(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__global__ void __launch_bounds__(32 * kBfWarps, 2) bf16_split_kernel(const __grid_constant__ Bf16Params p) {
  constexpr int D = kHeadDim;
  constexpr unsigned FULLMASK = 0xffffffffu;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) uint64_t s_full[kBfStages], s_empty[kBfStages];
  __shared__ int s_fail;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int pair = blockIdx.x / p.max_chunks, chunk = blockIdx.x % p.max_chunks;
  const int b = pair / p.Hkv, kvh = pair % p.Hkv;
  const int hq = p.hq;
  const int L = min(max(__ldg(p.seq_lens + b), 0), p.T_cap);
  const int t0 = chunk * kBfChunk;
  if (t0 >= L) return;  // the combine kernel reads only chunks that hold tokens
  const int t1 = min(L, t0 + kBfChunk);
  const int ntiles = (t1 - t0 + kBfTile - 1) / kBfTile;
  const size_t kvrow0 = ((size_t)b * p.Hkv + kvh) * p.T_cap;  // the pair's first cache row

  const uint32_t full0 = smem_addr(&s_full[0]), empty0 = smem_addr(&s_empty[0]);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kBfStages; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, kBfWarps);
    }
    s_fail = 0;
    mbar_init_fence();
  }
  __syncthreads();

  // warp 0 (lane 0): the 64 rows of tile k into stage k % kBfStages, four 2-D TMA boxes
  // (rows past the pair's tokens are read too and masked; past the tensor they are zero)
  auto issue = [&](int k) {
    if (lane != 0) return;
    const int st = k % kBfStages;
    const int y = (int)(kvrow0 + t0 + k * kBfTile);
    const uint32_t bar = full0 + 8u * st, dst = smem_addr(smem + st * kBfStageBytes);
    const uint64_t pol = l2_evict_first_policy();
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, (uint32_t)kBfStageBytes);
    tma_load_2d(dst, &p.tm_k, 0, y, bar, pol);
    tma_load_2d(dst + kBfHalfBytes, &p.tm_k, 64, y, bar, pol);
    tma_load_2d(dst + 2 * kBfHalfBytes, &p.tm_v, 0, y, bar, pol);
    tma_load_2d(dst + 3 * kBfHalfBytes, &p.tm_v, 64, y, bar, pol);
  };
  int n_issued = 0, n_waited = 0;  // tiles issued / waited for (warp 0)
  if (warp == 0)
    for (; n_issued < min(kBfStages, ntiles); ++n_issued) issue(n_issued);

  // Q as the A operand: rows g (queries; rows g + 8 stay zero), k-step ks
  uint32_t qa[8][2];
  {
    const bool live = g < hq;
    const __nv_bfloat16* qrow = p.q + ((size_t)b * p.Hq + kvh * hq + (live ? g : 0)) * D;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qa[ks][0] = live ? *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * c) : 0u;
      qa[ks][1] = live ? *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * c + 8) : 0u;
    }
  }
  float o[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;
  bool failed = false;

  for (int k = 0; k < ntiles; ++k) {
    const int st = k % kBfStages;
    if (!mbar_wait(full0 + 8u * st, (k / kBfStages) & 1, p.status, kStatusConsumerTimeout)) {
      failed = true;
      break;
    }
    n_waited = k + 1;
    uint8_t* kst = smem + st * kBfStageBytes;
    uint8_t* vst = kst + 2 * kBfHalfBytes;
    const int r0 = t0 + k * kBfTile, nrows = min(kBfTile, t1 - r0);
    const int w0 = 16 * warp;  // this warp's first row of the tile
    if (w0 < nrows) {
      // rows past the last token may hold anything: their V rows are zeroed (P is 0 there)
      if (w0 + 16 > nrows) {
        for (int idx = lane; idx < 16 * (D / 8); idx += 32) {
          const int r = w0 + idx / (D / 8), j = idx % (D / 8);  // both halves, 8 chunks each
          if (r >= nrows)
            *reinterpret_cast<uint4*>(vst + (j >> 3) * kBfHalfBytes + r * 128 + ((j & 7) << 4)) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();  // before a later bulk copy into the stage
        __syncwarp();
      }
      // S^T for tokens w0 + 8 j + (2c, 2c + 1), rows g
      float s[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
        const int kr = w0 + 8 * j + g;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t b0 = *reinterpret_cast<const uint32_t*>(kst + swz(kr, 16 * ks + 2 * c));
          const uint32_t b1 = *reinterpret_cast<const uint32_t*>(kst + swz(kr, 16 * ks + 2 * c + 8));
          const uint32_t a[4] = {qa[ks][0], 0u, qa[ks][1], 0u};
          mma_bf16(s[j], a, b0, b1);
        }
      }
      float mt = -INFINITY;
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int r = w0 + 8 * j + 2 * c + e;
          s[j][e] = (r < nrows) ? s[j][e] * p.sl2 : -INFINITY;
          mt = fmaxf(mt, s[j][e]);
        }
      mt = fmaxf(mt, __shfl_xor_sync(FULLMASK, mt, 1));
      mt = fmaxf(mt, __shfl_xor_sync(FULLMASK, mt, 2));
      const float m_new = fmaxf(m_run, mt);
      const float alpha = (m_run == -INFINITY) ? 0.f : fast_exp2(m_run - m_new);
      float pv[2][2];
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) pv[j][e] = (s[j][e] == -INFINITY) ? 0.f : fast_exp2(s[j][e] - m_new);
      l_run = alpha * l_run + ((pv[0][0] + pv[0][1]) + (pv[1][0] + pv[1][1]));
      m_run = m_new;
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        o[n][0] *= alpha;
        o[n][1] *= alpha;
      }
      const uint32_t pa[4] = {bf16x2_from(pv[0][0], pv[0][1]), 0u, bf16x2_from(pv[1][0], pv[1][1]), 0u};
      // O += P V: V^T fragments of channel tiles 2 nn, 2 nn + 1 by one transposed ldmatrix
      const int mi = lane >> 3, vr = w0 + (mi & 1) * 8 + (lane & 7);
      const uint32_t vbase = smem_addr(vst);
#pragma unroll
      for (int nn = 0; nn < 8; ++nn) {
        uint32_t v0, v1, v2, v3;
        ldmatrix_x4_trans(vbase + swz(vr, 16 * nn + 8 * (mi >> 1)), v0, v1, v2, v3);
        mma_bf16(o[2 * nn], pa, v0, v1);
        mma_bf16(o[2 * nn + 1], pa, v2, v3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8u * st);
    if (warp == 0 && k + kBfStages < ntiles) {
      // every warp is done with the stage: refill it with tile k + kBfStages
      if (!mbar_wait(empty0 + 8u * st, (k / kBfStages) & 1, p.status, kStatusConsumerTimeout)) {
        failed = true;
        break;
      }
      issue(k + kBfStages);
      ++n_issued;
    }
  }
  if (failed) s_fail = 1;
  __syncthreads();
  if (s_fail) {
    // every copy issued must have landed before shared memory is freed: wait (bounded)
    if (threadIdx.x == 0)
      for (int k = n_waited; k < n_issued; ++k)
        if (!mbar_wait(full0 + 8u * (k % kBfStages), (k / kBfStages) & 1, p.status, kStatusDrainTimeout)) break;
    return;
  }

  // ---------------------------------------------------- the chunk's partial from the warps
  // per warp: (m, l) per query, O [hq][D]; in the idle ring
  float* sm_ml = reinterpret_cast<float*>(smem);            // [kBfWarps][kMaxHq][2]
  float* sm_o = sm_ml + kBfWarps * kMaxHq * 2;              // [kBfWarps][hq][D]
  float lsum = l_run;
  lsum += __shfl_xor_sync(FULLMASK, lsum, 1);
  lsum += __shfl_xor_sync(FULLMASK, lsum, 2);
  if (g < hq) {
    if (c == 0) {
      sm_ml[(warp * kMaxHq + g) * 2] = m_run;
      sm_ml[(warp * kMaxHq + g) * 2 + 1] = lsum;
    }
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      sm_o[(warp * hq + g) * D + 8 * n + 2 * c] = o[n][0];
      sm_o[(warp * hq + g) * D + 8 * n + 2 * c + 1] = o[n][1];
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < hq * D; idx += 32 * kBfWarps) {
    const int i = idx / D, ch = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kBfWarps; ++w) M = fmaxf(M, sm_ml[(w * kMaxHq + i) * 2]);
    float acc = 0.f, lt = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kBfWarps; ++w) {
        const float mw = sm_ml[(w * kMaxHq + i) * 2];
        const float sc = (mw == -INFINITY) ? 0.f : fast_exp2(mw - M);
        acc = fmaf(sc, sm_o[(w * hq + i) * D + ch], acc);
        lt = fmaf(sc, sm_ml[(w * kMaxHq + i) * 2 + 1], lt);
      }
    }
    const size_t row = (size_t)blockIdx.x * hq + i;
    p.part_o[row * D + ch] = acc;
    if (ch == 0) p.part_ml[row] = make_float2(M, lt);
  }
}

// One CTA per pair, one warp per query: the chunks' partials into the bf16 output
// (out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s, zero without tokens).
__global__ void __launch_bounds__(256) bf16_combine_kernel(const __grid_constant__ Bf16Params p) {
  constexpr int D = kHeadDim;
  constexpr unsigned FULLMASK = 0xffffffffu;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = blockIdx.x, b = pair / p.Hkv, kvh = pair % p.Hkv, hq = p.hq;
  const int L = min(max(__ldg(p.seq_lens + b), 0), p.T_cap);
  const int n = (L + kBfChunk - 1) / kBfChunk;
  for (int i = warp; i < hq; i += 8) {
    float M = -INFINITY;
    for (int k = lane; k < n; k += 32) M = fmaxf(M, __ldcg(&p.part_ml[((size_t)pair * p.max_chunks + k) * hq + i]).x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(FULLMASK, M, o));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float lt = 0.f;
    if (M != -INFINITY) {
      for (int k0 = 0; k0 < n; k0 += 32) {
        float sc = 0.f;  // scale of chunk k0 + lane
        if (k0 + lane < n) {
          const float2 ml = __ldcg(&p.part_ml[((size_t)pair * p.max_chunks + k0 + lane) * hq + i]);
          if (ml.x != -INFINITY) {
            sc = fast_exp2(ml.x - M);
            lt = fmaf(sc, ml.y, lt);
          }
        }
        const int kn = min(32, n - k0);
#pragma unroll 8
        for (int kk = 0; kk < kn; ++kk) {
          const float sk = __shfl_sync(FULLMASK, sc, kk);
          const size_t row = ((size_t)pair * p.max_chunks + k0 + kk) * hq + i;
          if (sk != 0.f) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(p.part_o + row * D) + lane);
            acc.x = fmaf(sk, v.x, acc.x);
            acc.y = fmaf(sk, v.y, acc.y);
            acc.z = fmaf(sk, v.z, acc.z);
            acc.w = fmaf(sk, v.w, acc.w);
          }
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lt += __shfl_xor_sync(FULLMASK, lt, o);
    const bool any = lt > 0.f;
    const __nv_bfloat162 lo = __floats2bfloat162_rn(any ? acc.x / lt : 0.f, any ? acc.y / lt : 0.f);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(any ? acc.z / lt : 0.f, any ? acc.w / lt : 0.f);
    uint2 w;
    w.x = *reinterpret_cast<const uint32_t*>(&lo);
    w.y = *reinterpret_cast<const uint32_t*>(&hi);
    reinterpret_cast<uint2*>(p.out + ((size_t)b * p.Hq + kvh * hq + i) * D)[lane] = w;
  }
}

const void* bf16_split_kernel_fn() { return reinterpret_cast<const void*>(bf16_split_kernel); }
int bf16_split_smem_bytes() { return kBfSmem; }

int launch_bf16(const Bf16Params& p, cudaStream_t stream) {
  const long long pairs = (long long)p.B * p.Hkv;
  if (pairs == 0) return 0;
  bf16_split_kernel<<<(unsigned)(pairs * p.max_chunks), 32 * kBfWarps, kBfSmem, stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return -1;
  bf16_combine_kernel<<<(unsigned)pairs, 256, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace lbkv
