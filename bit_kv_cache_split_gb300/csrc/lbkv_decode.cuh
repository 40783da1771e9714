// lbkv_decode.cuh -- split-KV decode attention over a 2-/4-bit affine-quantized
// KV cache with the scale and offset applied by affine folding.
//
// Method: "FOSCAR: Accelerating Decode Attention over 2- and 4-Bit KV Caches
// through Affine Folding" (arXiv:2611.09722), abstract; and the explainer
// "FOSCAR speeds up 2-bit KV decode -- Affine folding of KV dequantization":
// fold rule (acc-fold when the group's scale is constant along the summed
// axis, operand-fold otherwise; key corrections before the softmax, value
// corrections before the final division; an unscaled partial never crosses a
// group boundary) and fold table (token-wise K: acc-fold, channel-wise K:
// operand-fold on Q, token-wise V: operand-fold on P, channel-wise V: acc-fold).
//
// Kernel design (sm_103a). One CTA per (sequence, KV head, split) streams
// its 128-token slots of packed codes and fp16 scales/offsets through a ring
// in shared memory with 1-D bulk copies issued by a producer warp (mbarrier
// full/empty pairs, no multicast). Eight consumer warps in two quads own the
// ring slots alternately; each warp of a quad takes a 32-token chunk of the
// slot and keeps its own online-softmax state.
//
// Operands. A 2-bit code q masked into the low bits of a byte is the e4m3
// value q * 2^-9 (subnormal), and 4*q at bits 2..3 is 4q * 2^-9; a 4-bit code
// in the low nibble is q * 2^-9 (the subnormal and first normal binade of
// e4m3 are evenly spaced). So one LOP3 turns four packed codes into four e4m3
// tensor-core inputs, with a power-of-two position factor folded into the
// other operand. The query (and the softmax weights) enter as the sum of two
// e4m3 parts hi + lo; the bf16 query is split exactly. Both products run on
// mma.sync m16n8k32 e4m3 (full-rate fp8 tensor cores), accumulating in fp32:
//   QK^T: rows = 16 tokens, k = 32 channels, cols = (query, part);
//   PV:   rows = 16 channels, k = 32 tokens, cols = (query[, group], part).
#pragma once

#include "lbkv_device.cuh"

namespace lbkv {

constexpr int kHeadDim = 128;
constexpr int kSlotTokens = 128;
constexpr int kChunk = 32;        // tokens per consumer warp step
constexpr int kConsumerWarps = 8;
constexpr int kQuads = kConsumerWarps / 4;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr int kMaxRing = 32;
constexpr int kMaxHq = 8;
// shared-memory map: barriers | Q (fp32) and per-query constants | ring
constexpr int kBarBytes = 2 * kMaxRing * 8;
constexpr int kConstFloats = kMaxHq * kHeadDim + kMaxHq * 8;
constexpr int kRingOffset = 8192;  // >= kBarBytes + 4 * kConstFloats, 1 KiB aligned
constexpr int kMergeBytes = kConsumerWarps * kMaxHq * (kHeadDim + 2) * 4;

struct DecodeParams {
  const __nv_bfloat16* q;
  const uint8_t* k_codes;
  const __half* k_scale;
  const __half* k_off;
  const uint8_t* v_codes;
  const __half* v_scale;
  const __half* v_off;
  const int32_t* seq_lens;
  const __nv_bfloat16* k_win;
  const __nv_bfloat16* v_win;
  const int32_t* win_lens;
  float2* part_ml;  // [B][Hq][s_tot] (running max in log2 units, denominator)
  float* part_o;    // [B][Hq][s_tot][D] unnormalised output
  int32_t* status;
  int B, Hq, Hkv, hq, T_cap, group, win_cap;
  float sl2;  // softmax scale times log2(e)
  int splits, s_tot, slots_per_split;
  int n_ring, slot_bytes, slot_tx;
  int off_vc, off_ks, off_kz, off_vs, off_vz;  // byte offsets inside a slot
  int sz_k_bytes, sz_v_bytes;                  // bytes of one scale (or offset) array per slot
};

// Channel fed at k-slot kappa of QK^T k-step ks (see the A-fragment build).
template <int BITS>
__device__ __forceinline__ int qk_channel(int ks, int kappa) {
  const int c = (kappa & 15) >> 2, j = kappa & 3, r = kappa >> 4;
  if (BITS == 2) return 32 * ks + 16 * (c >> 1) + 4 * j + (c & 1) + 2 * r;
  return 32 * ks + 8 * c + 2 * j + r;
}
// Position factor of the e4m3 image of channel ch on the K side.
template <int BITS>
__device__ __forceinline__ float k_mult(int ch) {
  return (BITS == 2 && (ch & 1)) ? 4.f : 1.f;
}

// Builds one B-fragment register for QK^T: four e4m3 bytes of part `part`
// (0 = hi, 1 = lo) of x[kappa0 .. kappa0+3].
__device__ __forceinline__ uint32_t pack_split4(const float (&x)[4], int part) {
  uint32_t h01, l01, h23, l23;
  split_e4m3_pair(x[0], x[1], h01, l01);
  split_e4m3_pair(x[2], x[3], h23, l23);
  return part ? (l01 | (l23 << 16)) : (h01 | (h23 << 16));
}

// ------------------------------------------------------------------------
// The kernel. BITS: 2 or 4. KL/VL: layout of K and V (0 token-wise,
// 1 channel-wise). NT: n-tiles of QK^T (1 when Hq/Hkv <= 4, else 2). GV:
// channel groups of a token-wise V side (1 or 2); 1 for channel-wise V.
// ------------------------------------------------------------------------
template <int BITS, int KL, int VL, int NT, int GV>
__global__ void __launch_bounds__(kThreads, 1) split_decode_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int RB = kHeadDim * BITS / 8;  // bytes per token row of codes
  constexpr int NTV = NT * GV;             // n-tiles of PV
  static_assert(NTV <= 2, "at most two PV n-tiles");
  extern __shared__ __align__(1024) uint8_t smem[];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int hq = p.hq;
  const int unit = b * p.Hkv + kvh;
  const int L = min(max(p.seq_lens[b], 0), p.T_cap);  // device value: clamped, never trusted
  const int D = kHeadDim;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);  // full[kMaxRing], empty[kMaxRing]
  float* sQ = reinterpret_cast<float*>(smem + kBarBytes);  // [kMaxHq][D]
  float* sAq = sQ + kMaxHq * D;                             // [kMaxHq] token-wise K score factor
  int* sEq = reinterpret_cast<int*>(sAq + kMaxHq);          // [kMaxHq] query exponent
  float* sBz = sAq + 2 * kMaxHq;                            // [kMaxHq][4] offset factor per channel group
  uint8_t* ring = smem + kRingOffset;
  const uint32_t bar0 = smem_addr(bars);
  auto full_bar = [&](int r) { return bar0 + 8u * r; };
  auto empty_bar = [&](int r) { return bar0 + 8u * (kMaxRing + r); };

  const bool window_cta = (split == p.splits);
  const int n_slots_total = (L + kSlotTokens - 1) / kSlotTokens;
  const int j0 = split * p.slots_per_split;
  const int n = window_cta ? 0 : max(0, min(j0 + p.slots_per_split, n_slots_total) - j0);

  if (threadIdx.x == 0) {
    for (int r = 0; r < p.n_ring; ++r) {
      mbar_init(full_bar(r), 1);
      mbar_init(empty_bar(r), 4);
    }
    mbar_init_fence();
  }
  __syncthreads();

  bool failed = false;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n > 0) {
      const uint64_t pol = l2_evict_first_policy();
      const uint32_t ring0 = smem_addr(ring);
      const size_t g_k = (KL == 0) ? (size_t)(kHeadDim / p.group) : 0;
      const size_t g_v = (VL == 0) ? (size_t)(kHeadDim / p.group) : 0;
      const size_t blocks = (size_t)p.T_cap / p.group;
      int issued = 0;
      for (int j = 0; j < n; ++j) {
        const int r = j % p.n_ring;
        if (j >= p.n_ring && !mbar_wait(empty_bar(r), ((j / p.n_ring) - 1) & 1, p.status, kStatusProducerTimeout))
          break;
        const size_t t0 = (size_t)(j0 + j) * kSlotTokens;
        const size_t row0 = (size_t)unit * p.T_cap + t0;
        const uint32_t dst = ring0 + (uint32_t)r * p.slot_bytes;
        const uint32_t fb = full_bar(r);
        mbar_arrive_expect_tx(fb, p.slot_tx);
        bulk_g2s(dst, p.k_codes + row0 * RB, kSlotTokens * RB, fb, pol);
        bulk_g2s(dst + p.off_vc, p.v_codes + row0 * RB, kSlotTokens * RB, fb, pol);
        const size_t ks0 = (KL == 0) ? row0 * g_k : ((size_t)unit * blocks + t0 / p.group) * kHeadDim;
        const size_t vs0 = (VL == 0) ? row0 * g_v : ((size_t)unit * blocks + t0 / p.group) * kHeadDim;
        bulk_g2s(dst + p.off_ks, p.k_scale + ks0, p.sz_k_bytes, fb, pol);
        bulk_g2s(dst + p.off_kz, p.k_off + ks0, p.sz_k_bytes, fb, pol);
        bulk_g2s(dst + p.off_vs, p.v_scale + vs0, p.sz_v_bytes, fb, pol);
        bulk_g2s(dst + p.off_vz, p.v_off + vs0, p.sz_v_bytes, fb, pol);
        issued = j + 1;
      }
      // every copy issued must have landed before shared memory is reused or freed
      for (int j = max(0, issued - p.n_ring); j < issued; ++j)
        if (!mbar_wait(full_bar(j % p.n_ring), (j / p.n_ring) & 1, p.status, kStatusDrainTimeout)) break;
    }
  } else {
    // ----------------------------------------------------------- consumers
    // Stage Q (fp32) and the per-query constants.
    for (int idx = threadIdx.x; idx < hq * D; idx += 32 * kConsumerWarps)
      sQ[idx] = __bfloat162float(p.q[((size_t)b * p.Hq + kvh * hq) * D + idx]);
    named_sync(1, 32 * kConsumerWarps);
    if (warp < hq) {
      const int i = warp;
      float amax = 0.f;
      float gs = 0.f;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int ch = 4 * lane + u;
        const float v = sQ[i * D + ch];
        amax = fmaxf(amax, fabsf(v) / k_mult<BITS>(ch));
        gs += v;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      // channel-group sums of Q (token-wise K offset term): lanes of one group are contiguous
      const int lanes_per_group = p.group / 4;  // 8, 16 or 32
      for (int o = 1; o < 32; o <<= 1) {
        const float other = __shfl_xor_sync(0xffffffffu, gs, o);
        if (o < lanes_per_group) gs += other;
      }
      int e = 0;
      if (amax > 0.f) e = min(100, max(-100, 7 - ilog2f(amax)));
      if (lane == 0) {
        sEq[i] = e;
        sAq[i] = p.sl2 * exp2i(9 - e);
      }
      if (KL == 0 && (lane % lanes_per_group) == 0) sBz[i * 4 + lane / lanes_per_group] = p.sl2 * gs;
    }
    named_sync(1, 32 * kConsumerWarps);

    // QK^T B fragments (token-wise K: fixed for the whole CTA).
    uint32_t qB[4][NT][2];
    const int qi_b = g >> 1, qpart = g & 1;  // this lane's (query-in-tile, part) as a B column
    if (KL == 0) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int i = 4 * nt + qi_b;
        const bool live = i < hq;
        const float sc = live ? exp2i(sEq[i]) : 0.f;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            float x[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int ch = qk_channel<BITS>(ks, 16 * r + 4 * c + j);
              x[j] = live ? sQ[i * D + ch] * sc / k_mult<BITS>(ch) : 0.f;
            }
            qB[ks][nt][r] = pack_split4(x, qpart);
          }
      }
    }
    // Per-lane score constants for the S-fragment query of each n-tile (query c + 4nt).
    float sA[NT];
    int qrow[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      qrow[nt] = min(c + 4 * nt, hq - 1);
      sA[nt] = sAq[qrow[nt]];
    }

    // Online-softmax state of this warp (for query c + 4nt).
    float m_run[NT], l_part[NT], zacc[NT][GV];
    float o_run[8][2][NTV];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m_run[nt] = -INFINITY;
      l_part[nt] = 0.f;
#pragma unroll
      for (int u = 0; u < GV; ++u) zacc[nt][u] = 0.f;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int rh = 0; rh < 2; ++rh)
#pragma unroll
        for (int v = 0; v < NTV; ++v) o_run[mt][rh][v] = 0.f;

    const int quad = warp >> 2, sub = warp & 3;
    const int groups_k = (KL == 0) ? kHeadDim / p.group : 1;
    const int ks_per_group = 4 / groups_k;
    const int groups_v = (VL == 0) ? kHeadDim / p.group : 1;

    for (int j = quad; j < n && !failed; j += kQuads) {
      const int r = j % p.n_ring;
      if (!mbar_wait(full_bar(r), (j / p.n_ring) & 1, p.status, kStatusConsumerTimeout)) {
        failed = true;
        break;
      }
      const uint8_t* slot = ring + (size_t)r * p.slot_bytes;
      const uint8_t* sKc = slot;
      const uint8_t* sVc = slot + p.off_vc;
      const __half* sKs = reinterpret_cast<const __half*>(slot + p.off_ks);
      const __half* sKz = reinterpret_cast<const __half*>(slot + p.off_kz);
      const __half* sVs = reinterpret_cast<const __half*>(slot + p.off_vs);
      const __half* sVz = reinterpret_cast<const __half*>(slot + p.off_vz);
      const int rel0 = kChunk * sub;                     // chunk start inside the slot
      const int tc = (j0 + j) * kSlotTokens + rel0;      // chunk start token
      const int nv = min(kChunk, L - tc);                // valid tokens in the chunk

      if (nv > 0) {
        // ------------------------------------------------ QK^T with K fold
        // Channel-wise K: Q' = Q * s_tau / position factor, split hi/lo (operand-fold),
        // and the offset sum_d Q_d z_tau,d (one constant per query and token group).
        float cwA[NT], cwB[NT];
        if (KL == 1) {
          const int tau_rel = rel0 / p.group;
          const __half* s_tau = sKs + tau_rel * kHeadDim;
          const __half* z_tau = sKz + tau_rel * kHeadDim;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const int i = 4 * nt + qi_b;
            const bool live = i < hq;
            float xs[4][2][4];
            float amax = 0.f, zsum = 0.f;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
#pragma unroll
              for (int rr = 0; rr < 2; ++rr)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                  const int ch = qk_channel<BITS>(ks, 16 * rr + 4 * c + jj);
                  const float qv = live ? sQ[i * D + ch] : 0.f;
                  const float v = qv * __half2float(s_tau[ch]) / k_mult<BITS>(ch);
                  xs[ks][rr][jj] = v;
                  amax = fmaxf(amax, fabsf(v));
                  zsum = fmaf(qv, __half2float(z_tau[ch]), zsum);
                }
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            zsum += __shfl_xor_sync(0xffffffffu, zsum, 1);
            zsum += __shfl_xor_sync(0xffffffffu, zsum, 2);
            int e = 0;
            if (amax > 0.f) e = min(100, max(-100, 7 - ilog2f(amax)));
            const float sc = exp2i(e);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
#pragma unroll
              for (int rr = 0; rr < 2; ++rr) {
                float x[4];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) x[jj] = xs[ks][rr][jj] * sc;
                qB[ks][nt][rr] = pack_split4(x, qpart);
              }
            // hand the factors to the S-fragment lanes (query c + 4nt lives in B column 2c)
            const float fa = p.sl2 * exp2i(9 - e), fb = p.sl2 * zsum;
            cwA[nt] = __shfl_sync(0xffffffffu, fa, 8 * c);
            cwB[nt] = __shfl_sync(0xffffffffu, fb, 8 * c);
          }
        }

        float S[2][2][NT];  // [m-tile][row half][n-tile], log2 domain
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          const int row0 = rel0 + 16 * mt + g;  // slot-relative tokens of this lane's rows
          const int row1 = row0 + 8;
          float acc[NT][4];
          float sfold[2][NT];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            sfold[0][nt] = sfold[1][nt] = 0.f;
#pragma unroll
            for (int u = 0; u < 4; ++u) acc[nt][u] = 0.f;
          }
          uint32_t w0[4], w1[4];  // per k-step source words for the two rows
          if (BITS == 2) {
            const uint32_t* r0p = reinterpret_cast<const uint32_t*>(sKc + row0 * RB);
            const uint32_t* r1p = reinterpret_cast<const uint32_t*>(sKc + row1 * RB);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              w0[ks] = r0p[2 * ks + (c >> 1)];
              w1[ks] = r1p[2 * ks + (c >> 1)];
            }
          } else {
            const uint32_t* r0p = reinterpret_cast<const uint32_t*>(sKc + row0 * RB);
            const uint32_t* r1p = reinterpret_cast<const uint32_t*>(sKc + row1 * RB);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              w0[ks] = r0p[4 * ks + c];
              w1[ks] = r1p[4 * ks + c];
            }
          }
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            uint32_t a0, a1, a2, a3;
            if (BITS == 2) {
              const uint32_t m0 = (c & 1) ? 0x0C0C0C0Cu : 0x03030303u;
              a0 = w0[ks] & m0;
              a1 = w1[ks] & m0;
              a2 = (w0[ks] >> 4) & m0;
              a3 = (w1[ks] >> 4) & m0;
            } else {
              a0 = w0[ks] & 0x0F0F0F0Fu;
              a1 = w1[ks] & 0x0F0F0F0Fu;
              a2 = (w0[ks] >> 4) & 0x0F0F0F0Fu;
              a3 = (w1[ks] >> 4) & 0x0F0F0F0Fu;
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_e4m3(acc[nt], a0, a1, a2, a3, qB[ks][nt][0], qB[ks][nt][1]);
            if (KL == 0 && ((ks + 1) % ks_per_group) == 0) {
              // acc-fold of one channel group: s * (raw partial) + z * sum(Q over the group)
              const int grp = ks / ks_per_group;
              const float s0 = __half2float(sKs[row0 * groups_k + grp]);
              const float z0 = __half2float(sKz[row0 * groups_k + grp]);
              const float s1 = __half2float(sKs[row1 * groups_k + grp]);
              const float z1 = __half2float(sKz[row1 * groups_k + grp]);
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                const float raw0 = acc[nt][0] + acc[nt][1], raw1 = acc[nt][2] + acc[nt][3];
                const float bz = sBz[qrow[nt] * 4 + grp];
                sfold[0][nt] = fmaf(s0 * sA[nt], raw0, fmaf(z0, bz, sfold[0][nt]));
                sfold[1][nt] = fmaf(s1 * sA[nt], raw1, fmaf(z1, bz, sfold[1][nt]));
#pragma unroll
                for (int u = 0; u < 4; ++u) acc[nt][u] = 0.f;
              }
            }
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            float s0v, s1v;
            if (KL == 0) {
              s0v = sfold[0][nt];
              s1v = sfold[1][nt];
            } else {
              s0v = fmaf(cwA[nt], acc[nt][0] + acc[nt][1], cwB[nt]);
              s1v = fmaf(cwA[nt], acc[nt][2] + acc[nt][3], cwB[nt]);
            }
            const int t0rel = 16 * mt + g;  // chunk-relative token of row half 0
            S[mt][0][nt] = (t0rel < nv) ? s0v : -INFINITY;
            S[mt][1][nt] = (t0rel + 8 < nv) ? s1v : -INFINITY;
          }
        }

        // ------------------------------------------------ online softmax
        // Tokens of this lane, chunk-relative: T0 = g, T1 = g+8, T2 = g+16, T3 = g+24,
        // i.e. S[0][0], S[0][1], S[1][0], S[1][1].
        float P[NT][4];
        float alpha[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float mx = fmaxf(fmaxf(S[0][0][nt], S[0][1][nt]), fmaxf(S[1][0][nt], S[1][1][nt]));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float m_new = fmaxf(m_run[nt], mx);
          alpha[nt] = (m_new == -INFINITY) ? 1.f : fast_exp2(m_run[nt] - m_new);
          const float mref = (m_new == -INFINITY) ? 0.f : m_new;
          m_run[nt] = m_new;
          P[nt][0] = fast_exp2(S[0][0][nt] - mref);
          P[nt][1] = fast_exp2(S[0][1][nt] - mref);
          P[nt][2] = fast_exp2(S[1][0][nt] - mref);
          P[nt][3] = fast_exp2(S[1][1][nt] - mref);
          l_part[nt] = l_part[nt] * alpha[nt] + ((P[nt][0] + P[nt][1]) + (P[nt][2] + P[nt][3]));
#pragma unroll
          for (int u = 0; u < GV; ++u) zacc[nt][u] *= alpha[nt];
        }
        // rescale the running output (column combo c + 4v belongs to query (c + 4v) / GV)
#pragma unroll
        for (int v = 0; v < NTV; ++v) {
          float av;
          if (GV == 1) {
            av = alpha[v];
          } else {
            const int i = (c + 4 * v) / GV;
            av = __shfl_sync(0xffffffffu, alpha[0], i & 3);
          }
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            o_run[mt][0][v] *= av;
            o_run[mt][1][v] *= av;
          }
        }

        // ------------------------------------------------ P (or P') -> e4m3 hi/lo words
        const int tok[4] = {rel0 + g, rel0 + g + 8, rel0 + g + 16, rel0 + g + 24};
        const bool val[4] = {g < nv, g + 8 < nv, g + 16 < nv, g + 24 < nv};
        uint32_t pw[NT][GV][2];  // [query slot][channel group][part], bytes = tokens T0..T3
        float inv_ps[GV];        // 2^-eP (token-wise V) per channel group
        float psum_chunk[NT];    // sum of P over the chunk (channel-wise V offset term)
        if (VL == 0) {
          float sv[GV][4];
          uint32_t smax = 0;
#pragma unroll
          for (int u = 0; u < GV; ++u)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const __half h = sVs[tok[k] * groups_v + u];
              sv[u][k] = val[k] ? __half2float(h) : 0.f;
              smax = max(smax, val[k] ? (uint32_t)(__half_as_ushort(h) & 0x7fffu) : 0u);
            }
          smax = max(smax, __shfl_xor_sync(0xffffffffu, smax, 4));
          smax = max(smax, __shfl_xor_sync(0xffffffffu, smax, 8));
          smax = max(smax, __shfl_xor_sync(0xffffffffu, smax, 16));
          const float smaxf = __half2float(__ushort_as_half((unsigned short)smax));
          int e = 0;
          if (smaxf > 0.f) e = min(100, max(-100, 7 - ilog2f(smaxf)));
          const float ps = exp2i(e);
#pragma unroll
          for (int u = 0; u < GV; ++u) inv_ps[u] = exp2i(-e);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int u = 0; u < GV; ++u) {
              float x[4], zt = 0.f;
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                x[k] = P[nt][k] * sv[u][k] * ps;
                const float zz = val[k] ? __half2float(sVz[tok[k] * groups_v + u]) : 0.f;
                zt = fmaf(P[nt][k], zz, zt);
              }
              zacc[nt][u] += zt;
              uint32_t h01, l01, h23, l23;
              split_e4m3_pair(x[0], x[1], h01, l01);
              split_e4m3_pair(x[2], x[3], h23, l23);
              pw[nt][u][0] = h01 | (h23 << 16);
              pw[nt][u][1] = l01 | (l23 << 16);
            }
        } else {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            float x[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) x[k] = P[nt][k] * 128.f;
            uint32_t h01, l01, h23, l23;
            split_e4m3_pair(x[0], x[1], h01, l01);
            split_e4m3_pair(x[2], x[3], h23, l23);
            pw[nt][0][0] = h01 | (h23 << 16);
            pw[nt][0][1] = l01 | (l23 << 16);
            float ps = (P[nt][0] + P[nt][1]) + (P[nt][2] + P[nt][3]);
            ps += __shfl_xor_sync(0xffffffffu, ps, 4);
            ps += __shfl_xor_sync(0xffffffffu, ps, 8);
            ps += __shfl_xor_sync(0xffffffffu, ps, 16);
            psum_chunk[nt] = ps;
          }
        }

        // B fragments of PV. Column n = 8v + g of n-tile v is combo (4v + g/2), part g&1;
        // combo = query * GV + group. k-slot 4c + jj holds chunk token c + 8jj (reg0) and
        // k-slot 16 + 4c + jj holds token c + 4 + 8jj (reg1); those four tokens are the
        // T0..T3 of lane 4*c' + (query & 3) with c' = c resp. c + 4.
        uint32_t pB[NTV][2];
#pragma unroll
        for (int v = 0; v < NTV; ++v) {
          const int combo = 4 * v + (g >> 1);
          const int i = combo / GV, u_need = combo % GV, part = g & 1;
          const int src0 = 4 * c + (i & 3), src1 = 4 * (c + 4) + (i & 3);
          const int ntq = (GV == 1) ? v : 0;  // query slot of the source lane
          uint32_t b0 = 0, b1 = 0;
#pragma unroll
          for (int u = 0; u < GV; ++u)
#pragma unroll
            for (int pp = 0; pp < 2; ++pp) {
              const uint32_t x0 = __shfl_sync(0xffffffffu, pw[ntq][u][pp], src0);
              const uint32_t x1 = __shfl_sync(0xffffffffu, pw[ntq][u][pp], src1);
              if (u == u_need && pp == part) {
                b0 = x0;
                b1 = x1;
              }
            }
          const bool live = i < hq;
          pB[v][0] = live ? b0 : 0u;
          pB[v][1] = live ? b1 : 0u;
        }

        // ------------------------------------------------ PV
        float accv[8][NTV][4];
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int v = 0; v < NTV; ++v)
#pragma unroll
            for (int u = 0; u < 4; ++u) accv[mt][v][u] = 0.f;
        if (BITS == 2) {
          uint32_t wa[4], wb[4];
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            wa[jj] = reinterpret_cast<const uint32_t*>(sVc + (rel0 + c + 8 * jj) * RB)[g];
            wb[jj] = reinterpret_cast<const uint32_t*>(sVc + (rel0 + c + 4 + 8 * jj) * RB)[g];
          }
          uint32_t ta[4], tb[4];
          transpose4x4(wa[0], wa[1], wa[2], wa[3], ta);
          transpose4x4(wb[0], wb[1], wb[2], wb[3], tb);
#pragma unroll
          for (int bb = 0; bb < 4; ++bb) {
            const uint32_t a_p0 = ta[bb] & 0x03030303u, a_p1 = ta[bb] & 0x0C0C0C0Cu;
            const uint32_t a_p2 = (ta[bb] >> 4) & 0x03030303u, a_p3 = (ta[bb] >> 4) & 0x0C0C0C0Cu;
            const uint32_t b_p0 = tb[bb] & 0x03030303u, b_p1 = tb[bb] & 0x0C0C0C0Cu;
            const uint32_t b_p2 = (tb[bb] >> 4) & 0x03030303u, b_p3 = (tb[bb] >> 4) & 0x0C0C0C0Cu;
#pragma unroll
            for (int v = 0; v < NTV; ++v) {
              mma_e4m3(accv[2 * bb][v], a_p0, a_p1, b_p0, b_p1, pB[v][0], pB[v][1]);
              mma_e4m3(accv[2 * bb + 1][v], a_p2, a_p3, b_p2, b_p3, pB[v][0], pB[v][1]);
            }
          }
        } else {
          uint2 wa[4], wb[4];
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            wa[jj] = reinterpret_cast<const uint2*>(sVc + (rel0 + c + 8 * jj) * RB)[g];
            wb[jj] = reinterpret_cast<const uint2*>(sVc + (rel0 + c + 4 + 8 * jj) * RB)[g];
          }
#pragma unroll
          for (int uu = 0; uu < 2; ++uu) {
            uint32_t ta[4], tb[4];
            if (uu == 0) {
              transpose4x4(wa[0].x, wa[1].x, wa[2].x, wa[3].x, ta);
              transpose4x4(wb[0].x, wb[1].x, wb[2].x, wb[3].x, tb);
            } else {
              transpose4x4(wa[0].y, wa[1].y, wa[2].y, wa[3].y, ta);
              transpose4x4(wb[0].y, wb[1].y, wb[2].y, wb[3].y, tb);
            }
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) {
              const uint32_t a_lo = ta[bb] & 0x0F0F0F0Fu, a_hi = (ta[bb] >> 4) & 0x0F0F0F0Fu;
              const uint32_t b_lo = tb[bb] & 0x0F0F0F0Fu, b_hi = (tb[bb] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
              for (int v = 0; v < NTV; ++v) mma_e4m3(accv[4 * uu + bb][v], a_lo, a_hi, b_lo, b_hi, pB[v][0], pB[v][1]);
            }
          }
        }

        // ------------------------------------------------ V fold into the running output
        // Row half rh of m-tile mt is channel 16g + 2mt + rh; its e4m3 image carries a
        // position factor 4 when BITS == 2 and rh == 1.
        if (VL == 0) {
#pragma unroll
          for (int v = 0; v < NTV; ++v) {
            const int u = (GV == 1) ? 0 : ((c + 4 * v) % GV);
            const float f0 = 512.f * inv_ps[u];
            const float f1 = (BITS == 2 ? 128.f : 512.f) * inv_ps[u];
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              o_run[mt][0][v] = fmaf(accv[mt][v][0] + accv[mt][v][1], f0, o_run[mt][0][v]);
              o_run[mt][1][v] = fmaf(accv[mt][v][2] + accv[mt][v][3], f1, o_run[mt][1][v]);
            }
          }
        } else {
          // acc-fold per token group: s_tau,d * (raw partial) + z_tau,d * sum_t P_t
          const int tau_rel = rel0 / p.group;
          const __half* s_tau = sVs + tau_rel * kHeadDim;
          const __half* z_tau = sVz + tau_rel * kHeadDim;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int rh = 0; rh < 2; ++rh) {
              const int ch = 16 * g + 2 * mt + rh;
              const float s = __half2float(s_tau[ch]) * ((BITS == 2 && rh) ? 1.f : 4.f);
              const float z = __half2float(z_tau[ch]);
#pragma unroll
              for (int v = 0; v < NTV; ++v) {
                const float raw = accv[mt][v][2 * rh] + accv[mt][v][2 * rh + 1];
                o_run[mt][rh][v] = fmaf(s, raw, fmaf(z, psum_chunk[v], o_run[mt][rh][v]));
              }
            }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(r));
    }

    // ---------------------------------------------------- warp results
    if (!window_cta) {
    named_sync(1, 32 * kConsumerWarps);  // every slot consumed: the ring is free
    float* sM = reinterpret_cast<float*>(ring);            // [warps][kMaxHq]
    float* sL = sM + kConsumerWarps * kMaxHq;              // [warps][kMaxHq]
    float* sO = sL + kConsumerWarps * kMaxHq;              // [warps][kMaxHq][D]
    float lsum[NT], zsum[NT][GV];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float l = l_part[nt];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      lsum[nt] = l;
#pragma unroll
      for (int u = 0; u < GV; ++u) {
        float z = zacc[nt][u];
        z += __shfl_xor_sync(0xffffffffu, z, 4);
        z += __shfl_xor_sync(0xffffffffu, z, 8);
        z += __shfl_xor_sync(0xffffffffu, z, 16);
        zsum[nt][u] = z;
      }
      const int i = c + 4 * nt;
      if (g == 0 && i < hq) {
        sM[warp * kMaxHq + i] = m_run[nt];
        sL[warp * kMaxHq + i] = lsum[nt];
      }
    }
#pragma unroll
    for (int v = 0; v < NTV; ++v) {
      const int combo = c + 4 * v;
      const int i = combo / GV, u = combo % GV;
      // the value-offset term of (query i, group u) lives on the S lanes of query i
      float zt = 0.f;
      if (VL == 0) {
        const int ntq = (GV == 1) ? v : 0;
#pragma unroll
        for (int uu = 0; uu < GV; ++uu) {
          const float x = __shfl_sync(0xffffffffu, zsum[ntq][uu], i & 3);
          if (uu == u) zt = x;
        }
      }
      const bool mine = (i < hq) && (GV == 1 || (16 * g) / 64 == u);
      if (mine) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int rh = 0; rh < 2; ++rh) sO[(warp * kMaxHq + i) * D + 16 * g + 2 * mt + rh] = o_run[mt][rh][v] + zt;
      }
    }
    }  // !window_cta
  }

  // ---------------------------------------------------- window split
  if (window_cta && warp < kConsumerWarps) {
    float* sM = reinterpret_cast<float*>(ring);
    float* sL = sM + kConsumerWarps * kMaxHq;
    float* sO = sL + kConsumerWarps * kMaxHq;
    const int W = min(max(p.win_lens[b], 0), p.win_cap);
    float m[kMaxHq], l[kMaxHq], o[kMaxHq][4];
#pragma unroll
    for (int i = 0; i < kMaxHq; ++i) {
      m[i] = -INFINITY;
      l[i] = 0.f;
      o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    }
    const size_t wbase = (size_t)unit * p.win_cap;
    for (int t = warp; t < W; t += kConsumerWarps) {
      const uint2 kr = reinterpret_cast<const uint2*>(p.k_win + (wbase + t) * D)[lane];
      const uint2 vr = reinterpret_cast<const uint2*>(p.v_win + (wbase + t) * D)[lane];
      const __nv_bfloat162* kh = reinterpret_cast<const __nv_bfloat162*>(&kr);
      const __nv_bfloat162* vh = reinterpret_cast<const __nv_bfloat162*>(&vr);
      const float2 k01 = __bfloat1622float2(kh[0]), k23 = __bfloat1622float2(kh[1]);
      const float2 v01 = __bfloat1622float2(vh[0]), v23 = __bfloat1622float2(vh[1]);
#pragma unroll
      for (int i = 0; i < kMaxHq; ++i) {
        if (i >= hq) break;
        const float* qrow = sQ + i * D + 4 * lane;
        float d = qrow[0] * k01.x + qrow[1] * k01.y + qrow[2] * k23.x + qrow[3] * k23.y;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
        const float s = d * p.sl2;
        const float mn = fmaxf(m[i], s);
        const float a = fast_exp2(m[i] - mn);
        const float pr = fast_exp2(s - mn);
        m[i] = mn;
        l[i] = l[i] * a + pr;
        o[i][0] = o[i][0] * a + pr * v01.x;
        o[i][1] = o[i][1] * a + pr * v01.y;
        o[i][2] = o[i][2] * a + pr * v23.x;
        o[i][3] = o[i][3] * a + pr * v23.y;
      }
    }
#pragma unroll
    for (int i = 0; i < kMaxHq; ++i) {
      if (i >= hq) break;
      if (lane == 0) {
        sM[warp * kMaxHq + i] = m[i];
        sL[warp * kMaxHq + i] = l[i];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) sO[(warp * kMaxHq + i) * D + 4 * lane + u] = o[i][u];
    }
  }

  // ---------------------------------------------------- merge the warps, write the partial
  __syncthreads();
  if (warp < kConsumerWarps && !failed) {
    const float* sM = reinterpret_cast<const float*>(ring);
    const float* sL = sM + kConsumerWarps * kMaxHq;
    const float* sO = sL + kConsumerWarps * kMaxHq;
    for (int idx = threadIdx.x; idx < hq * D; idx += 32 * kConsumerWarps) {
      const int i = idx / D, ch = idx % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sM[w * kMaxHq + i]);
      float acc = 0.f, lt = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float mw = sM[w * kMaxHq + i];
          const float sc = (mw == -INFINITY) ? 0.f : fast_exp2(mw - M);
          acc = fmaf(sc, sO[(w * kMaxHq + i) * D + ch], acc);
          lt = fmaf(sc, sL[w * kMaxHq + i], lt);
        }
      }
      const size_t prow = ((size_t)b * p.Hq + kvh * hq + i) * p.s_tot + split;
      p.part_o[prow * D + ch] = acc;
      if (ch == 0) p.part_ml[prow] = make_float2(M, lt);
    }
  }
}

}  // namespace lbkv
