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
// full/empty pairs, bounded waits, no multicast). The consumer warps form
// quads; the quads own the ring slots in turn and each warp of a quad takes a
// 32-token chunk of the slot with its own online-softmax state. The CTA then
// merges its warps into one split partial, and the last split of a
// (sequence, KV head) to finish merges all splits into the bf16 output.
//
// Operands. A 2-bit code q masked into the low bits of a byte is the e4m3
// value q * 2^-9 (subnormal), and 4*q at bits 2..3 is 4q * 2^-9; a 4-bit code
// in the low nibble is q * 2^-9 (the subnormal and first normal binade of
// e4m3 are evenly spaced). So one LOP3 turns four packed codes into four e4m3
// tensor-core inputs, with a power-of-two position factor folded into the
// other operand. The query enters as the exact two-part e4m3 split hi + lo of
// its bf16 value (three parts when a channel-wise K scale multiplies it first);
// the softmax weights enter as a two-part split, and the running denominator
// and the value offsets are summed from the weights actually fed, so the
// result is an exact attention under the fed weights. Both products run on
// mma.sync m16n8k32 e4m3 (full-rate fp8 tensor cores), accumulating in fp32:
//   QK^T: rows = 16 tokens, k = 32 channels, cols = (query, part);
//   PV:   rows = 16 channels, k = 32 tokens, cols = (query[, group], part).
#pragma once

#include <type_traits>

#include "lbkv_device.cuh"

#ifndef LBKV_CONSUMER_WARPS
#define LBKV_CONSUMER_WARPS 8
#endif

namespace lbkv {

constexpr int kHeadDim = 128;
constexpr int kSlotTokens = 128;
constexpr int kChunk = 32;  // tokens per consumer warp step
constexpr int kConsumerWarps = LBKV_CONSUMER_WARPS;
static_assert(kConsumerWarps % 4 == 0, "consumer warps come in quads");
constexpr int kQuads = kConsumerWarps / 4;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr int kMaxRing = 48;
constexpr int kMaxHq = 8;
// shared-memory map: barriers | Q (fp32) and per-query constants | ring
constexpr int kBarBytes = 2 * kMaxRing * 8;
constexpr int kRingOffset = 8192;
static_assert(kBarBytes + 4 * (kMaxHq * kHeadDim + 6 * kMaxHq) <= kRingOffset, "prologue fits");
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
  int32_t* done;    // [B][Hkv] splits finished; the last one merges and resets it to 0
  __nv_bfloat16* out;
  int B, Hq, Hkv, hq, T_cap, win_cap;
  float sl2;  // softmax scale times log2(e)
  int splits, s_tot, slots_per_split;
  int n_ring, slot_bytes, slot_tx;
  int off_vc, off_ks, off_kz, off_vs, off_vz;  // byte offsets inside a slot
  int sz_k_bytes, sz_v_bytes;                  // bytes of one scale (or offset) array per slot
};

// Compile-time shape of one kernel variant.
template <int BITS_, int KL_, int VL_, int NT_, int LOG2G_>
struct Cfg {
  static constexpr int BITS = BITS_, KL = KL_, VL = VL_, NT = NT_;
  static constexpr int G = 1 << LOG2G_;                    // group size
  static constexpr int GK = (KL == 0) ? kHeadDim / G : 1;  // K channel groups per token
  static constexpr int GV = (VL == 0) ? kHeadDim / G : 1;  // V channel groups per token
  static constexpr int KSG = 4 / GK;                       // QK k-steps per K channel group
  static constexpr int NTK = (KL == 1) ? 2 * NT : NT;      // QK n-tiles (3-part query: 2 per slot)
  static constexpr int NTV = NT * GV;                      // PV n-tiles
  static constexpr int RB = kHeadDim * BITS / 8;           // bytes per token row of codes
  static_assert(NTV <= 2, "at most two PV n-tiles");
  static_assert(G >= kChunk, "a chunk never straddles a token group");
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
// (0 = hi, 1 = lo) of x[0..3].
__device__ __forceinline__ uint32_t pack_split4(const float (&x)[4], int part) {
  uint32_t h01, l01, h23, l23;
  split_e4m3_pair(x[0], x[1], h01, l01);
  split_e4m3_pair(x[2], x[3], h23, l23);
  return part ? (l01 | (l23 << 16)) : (h01 | (h23 << 16));
}

// Per-warp state, held in registers.
template <class C>
struct WarpState {
  uint32_t qB[4][C::NTK][2];  // QK^T B fragments
  float sA[C::NT];            // token-wise K: score factor of this lane's query
  int qrow[C::NT];            // this lane's query (clamped), per n-tile
  float m_run[C::NT], l_part[C::NT], zacc[C::NT][C::GV];
  float o_run[8][2][C::NTV];
};

// Everything one chunk of 32 tokens needs from shared memory.
struct ChunkSmem {
  const uint8_t* kc;
  const uint8_t* vc;
  const __half* ks;
  const __half* kz;
  const __half* vs;
  const __half* vz;
  const float* sQ;
  const float* sBz;
};

// One 32-token chunk: QK^T with the K fold, online softmax, P (or P') split,
// PV with the V fold. FULL: all 32 tokens valid (no masking).
template <class C, bool FULL>
__device__ __forceinline__ void process_chunk(WarpState<C>& st, const ChunkSmem& sm, int rel0, int nv, int hq,
                                              float sl2, int lane) {
  constexpr int BITS = C::BITS, KL = C::KL, VL = C::VL, NT = C::NT, GV = C::GV, NTK = C::NTK, NTV = C::NTV;
  constexpr int RB = C::RB, D = kHeadDim;
  const int g = lane >> 2, c = lane & 3;
  const int qi_b = g >> 1, qpart = g & 1;
  constexpr unsigned FULLMASK = 0xffffffffu;

  // ---------------------------------------------------- channel-wise K: Q' per token group
  float cwA[NT], cwB[NT];
  if (KL == 1) {
    const int tau_rel = rel0 / C::G;  // compile-time power of two
    const __half* s_tau = sm.ks + tau_rel * D;
    const __half* z_tau = sm.kz + tau_rel * D;
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
            const float qv = live ? sm.sQ[i * D + ch] : 0.f;
            const float v = qv * __half2float(s_tau[ch]) * (1.f / k_mult<BITS>(ch));
            xs[ks][rr][jj] = v;
            amax = fmaxf(amax, fabsf(v));
            zsum = fmaf(qv, __half2float(z_tau[ch]), zsum);
          }
      amax = fmaxf(amax, __shfl_xor_sync(FULLMASK, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(FULLMASK, amax, 2));
      zsum += __shfl_xor_sync(FULLMASK, zsum, 1);
      zsum += __shfl_xor_sync(FULLMASK, zsum, 2);
      int e = 0;
      if (amax > 0.f) e = min(100, max(-100, 7 - ilog2f(amax)));
      const float sc = exp2i(e);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          uint32_t h01, l01, m01, h23, l23, m23;
          split3_e4m3_pair(xs[ks][rr][0] * sc, xs[ks][rr][1] * sc, h01, l01, m01);
          split3_e4m3_pair(xs[ks][rr][2] * sc, xs[ks][rr][3] * sc, h23, l23, m23);
          st.qB[ks][2 * nt][rr] = qpart ? (l01 | (l23 << 16)) : (h01 | (h23 << 16));
          st.qB[ks][2 * nt + 1][rr] = qpart ? 0u : (m01 | (m23 << 16));
        }
      // the S-fragment lanes of query c + 4nt read B column 2c, held by lane 8c
      const float fa = sl2 * exp2i(9 - e), fb = sl2 * zsum;
      cwA[nt] = __shfl_sync(FULLMASK, fa, 8 * c);
      cwB[nt] = __shfl_sync(FULLMASK, fb, 8 * c);
    }
  }

  // ---------------------------------------------------- QK^T with the K fold
  float S[2][2][NT];  // [m-tile][row half][n-tile], log2 domain
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    const int row0 = rel0 + 16 * mt + g;  // slot-relative tokens of this lane's rows
    const int row1 = row0 + 8;
    float acc[NTK][4];
    float sfold[2][NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) sfold[0][nt] = sfold[1][nt] = 0.f;
#pragma unroll
    for (int nt = 0; nt < NTK; ++nt)
#pragma unroll
      for (int u = 0; u < 4; ++u) acc[nt][u] = 0.f;
    uint32_t w0[4], w1[4];
    const uint32_t* r0p = reinterpret_cast<const uint32_t*>(sm.kc + row0 * RB);
    const uint32_t* r1p = reinterpret_cast<const uint32_t*>(sm.kc + row1 * RB);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const int wi = (BITS == 2) ? 2 * ks + (c >> 1) : 4 * ks + c;
      w0[ks] = r0p[wi];
      w1[ks] = r1p[wi];
    }
    const uint32_t m2 = (c & 1) ? 0x0C0C0C0Cu : 0x03030303u;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      uint32_t a0, a1, a2, a3;
      if (BITS == 2) {
        a0 = w0[ks] & m2;
        a1 = w1[ks] & m2;
        a2 = (w0[ks] >> 4) & m2;
        a3 = (w1[ks] >> 4) & m2;
      } else {
        a0 = w0[ks] & 0x0F0F0F0Fu;
        a1 = w1[ks] & 0x0F0F0F0Fu;
        a2 = (w0[ks] >> 4) & 0x0F0F0F0Fu;
        a3 = (w1[ks] >> 4) & 0x0F0F0F0Fu;
      }
#pragma unroll
      for (int nt = 0; nt < NTK; ++nt) mma_e4m3(acc[nt], a0, a1, a2, a3, st.qB[ks][nt][0], st.qB[ks][nt][1]);
      if (KL == 0 && ((ks + 1) % C::KSG) == 0) {
        // acc-fold of one channel group: s * (raw partial) + z * sum(Q over the group)
        constexpr int GK = C::GK;
        const int grp = ks / C::KSG;
        const float s0 = __half2float(sm.ks[row0 * GK + grp]);
        const float z0 = __half2float(sm.kz[row0 * GK + grp]);
        const float s1 = __half2float(sm.ks[row1 * GK + grp]);
        const float z1 = __half2float(sm.kz[row1 * GK + grp]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float raw0 = acc[nt][0] + acc[nt][1], raw1 = acc[nt][2] + acc[nt][3];
          const float bz = sm.sBz[st.qrow[nt] * 4 + grp];
          sfold[0][nt] = fmaf(s0 * st.sA[nt], raw0, fmaf(z0, bz, sfold[0][nt]));
          sfold[1][nt] = fmaf(s1 * st.sA[nt], raw1, fmaf(z1, bz, sfold[1][nt]));
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
        s0v = fmaf(cwA[nt], (acc[2 * nt][0] + acc[2 * nt][1]) + acc[2 * nt + 1][0], cwB[nt]);
        s1v = fmaf(cwA[nt], (acc[2 * nt][2] + acc[2 * nt][3]) + acc[2 * nt + 1][2], cwB[nt]);
      }
      if (FULL) {
        S[mt][0][nt] = s0v;
        S[mt][1][nt] = s1v;
      } else {
        const int t0rel = 16 * mt + g;
        S[mt][0][nt] = (t0rel < nv) ? s0v : -INFINITY;
        S[mt][1][nt] = (t0rel + 8 < nv) ? s1v : -INFINITY;
      }
    }
  }

  // ---------------------------------------------------- online softmax
  // This lane's tokens, chunk-relative: T0 = g, T1 = g+8, T2 = g+16, T3 = g+24.
  float P[NT][4];
  float alpha[NT];
  bool rescale = false;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float mx = fmaxf(fmaxf(S[0][0][nt], S[0][1][nt]), fmaxf(S[1][0][nt], S[1][1][nt]));
    mx = fmaxf(mx, __shfl_xor_sync(FULLMASK, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(FULLMASK, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(FULLMASK, mx, 16));
    const float m_new = fmaxf(st.m_run[nt], mx);
    rescale |= (m_new > st.m_run[nt]);
    alpha[nt] = (m_new == -INFINITY) ? 1.f : fast_exp2(st.m_run[nt] - m_new);
    const float mref = (m_new == -INFINITY) ? 0.f : m_new;
    st.m_run[nt] = m_new;
    P[nt][0] = fast_exp2(S[0][0][nt] - mref);
    P[nt][1] = fast_exp2(S[0][1][nt] - mref);
    P[nt][2] = fast_exp2(S[1][0][nt] - mref);
    P[nt][3] = fast_exp2(S[1][1][nt] - mref);
  }
  if (__any_sync(FULLMASK, rescale)) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      st.l_part[nt] *= alpha[nt];
#pragma unroll
      for (int u = 0; u < GV; ++u) st.zacc[nt][u] *= alpha[nt];
    }
    // running output column combo c + 4v belongs to query (c + 4v) / GV
#pragma unroll
    for (int v = 0; v < NTV; ++v) {
      float av;
      if (GV == 1) {
        av = alpha[v];
      } else {
        const int i = (c + 4 * v) / GV;
        av = __shfl_sync(FULLMASK, alpha[0], i & 3);
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        st.o_run[mt][0][v] *= av;
        st.o_run[mt][1][v] *= av;
      }
    }
  }

  // ---------------------------------------------------- weights -> e4m3 hi/lo words
  // Token-wise V (operand-fold): the fed weight of token t for channel group u is
  // P_t * s_t,u scaled by 2^eP; channel-wise V: P_t * 2^7. The denominator and the
  // value offsets are summed from the fed weights w_t (fed / scale).
  const int tok0 = rel0 + g;
  uint32_t pw[NT][GV][2];
  float inv_ps = 1.f;    // 2^-eP
  float psum_chunk[NT];  // channel-wise V: sum of fed weights over the chunk
  if (VL == 0) {
    float sv[GV][4];
    uint32_t smax = 0;
#pragma unroll
    for (int u = 0; u < GV; ++u)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const bool ok = FULL || (g + 8 * k < nv);
        const __half h = sm.vs[(tok0 + 8 * k) * GV + u];
        sv[u][k] = ok ? __half2float(h) : 0.f;
        smax = max(smax, ok ? (uint32_t)(__half_as_ushort(h) & 0x7fffu) : 0u);
      }
    smax = max(smax, __shfl_xor_sync(FULLMASK, smax, 4));
    smax = max(smax, __shfl_xor_sync(FULLMASK, smax, 8));
    smax = max(smax, __shfl_xor_sync(FULLMASK, smax, 16));
    const float smaxf = __half2float(__ushort_as_half((unsigned short)smax));
    int e = 0;
    if (smaxf > 0.f) e = min(100, max(-100, 7 - ilog2f(smaxf)));
    const float ps = exp2i(e);
    inv_ps = exp2i(-e);
    float rs[GV][4];  // 2^-eP / s (unused when s == 0: the weight is then P itself)
#pragma unroll
    for (int u = 0; u < GV; ++u)
#pragma unroll
      for (int k = 0; k < 4; ++k) rs[u][k] = (sv[u][k] != 0.f) ? fast_rcp(sv[u][k]) * inv_ps : 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float lsum = 0.f;
#pragma unroll
      for (int u = 0; u < GV; ++u) {
        float x[4], f[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) x[k] = P[nt][k] * sv[u][k] * ps;
        uint32_t h01, l01, h23, l23;
        split_e4m3_pair_fed(x[0], x[1], h01, l01, f[0], f[1]);
        split_e4m3_pair_fed(x[2], x[3], h23, l23, f[2], f[3]);
        pw[nt][u][0] = h01 | (h23 << 16);
        pw[nt][u][1] = l01 | (l23 << 16);
        float zt = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float w = (sv[u][k] != 0.f) ? f[k] * rs[u][k] : P[nt][k];
          const bool ok = FULL || (g + 8 * k < nv);
          const float zz = ok ? __half2float(sm.vz[(tok0 + 8 * k) * GV + u]) : 0.f;
          zt = fmaf(w, zz, zt);
          if (u == 0) lsum += w;
        }
        st.zacc[nt][u] += zt;
      }
      st.l_part[nt] += lsum;
    }
  } else {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float f[4];
      uint32_t h01, l01, h23, l23;
      split_e4m3_pair_fed(P[nt][0] * 128.f, P[nt][1] * 128.f, h01, l01, f[0], f[1]);
      split_e4m3_pair_fed(P[nt][2] * 128.f, P[nt][3] * 128.f, h23, l23, f[2], f[3]);
      pw[nt][0][0] = h01 | (h23 << 16);
      pw[nt][0][1] = l01 | (l23 << 16);
      float ps = ((f[0] + f[1]) + (f[2] + f[3])) * (1.f / 128.f);
      st.l_part[nt] += ps;
      ps += __shfl_xor_sync(FULLMASK, ps, 4);
      ps += __shfl_xor_sync(FULLMASK, ps, 8);
      ps += __shfl_xor_sync(FULLMASK, ps, 16);
      psum_chunk[nt] = ps;
    }
  }

  // ---------------------------------------------------- PV B fragments
  // Column n = 8v + g of n-tile v is combo (4v + g/2), part g&1; combo = query * GV +
  // group. k-slot 4c + jj holds chunk token c + 8jj (reg0), k-slot 16 + 4c + jj holds
  // token c + 4 + 8jj (reg1): the T0..T3 of lane 4*c' + (query & 3), c' = c or c + 4.
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
        const uint32_t x0 = __shfl_sync(FULLMASK, pw[ntq][u][pp], src0);
        const uint32_t x1 = __shfl_sync(FULLMASK, pw[ntq][u][pp], src1);
        if (u == u_need && pp == part) {
          b0 = x0;
          b1 = x1;
        }
      }
    const bool live = i < hq;
    pB[v][0] = live ? b0 : 0u;
    pB[v][1] = live ? b1 : 0u;
  }

  // ---------------------------------------------------- PV
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
      wa[jj] = reinterpret_cast<const uint32_t*>(sm.vc + (rel0 + c + 8 * jj) * RB)[g];
      wb[jj] = reinterpret_cast<const uint32_t*>(sm.vc + (rel0 + c + 4 + 8 * jj) * RB)[g];
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
      wa[jj] = reinterpret_cast<const uint2*>(sm.vc + (rel0 + c + 8 * jj) * RB)[g];
      wb[jj] = reinterpret_cast<const uint2*>(sm.vc + (rel0 + c + 4 + 8 * jj) * RB)[g];
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

  // ---------------------------------------------------- V fold into the running output
  // Row half rh of m-tile mt is channel 16g + 2mt + rh; its e4m3 image carries a
  // position factor 4 when BITS == 2 and rh == 1.
  if (VL == 0) {
    const float f0 = 512.f * inv_ps;
    const float f1 = (BITS == 2 ? 128.f : 512.f) * inv_ps;
#pragma unroll
    for (int v = 0; v < NTV; ++v)
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        st.o_run[mt][0][v] = fmaf(accv[mt][v][0] + accv[mt][v][1], f0, st.o_run[mt][0][v]);
        st.o_run[mt][1][v] = fmaf(accv[mt][v][2] + accv[mt][v][3], f1, st.o_run[mt][1][v]);
      }
  } else {
    // acc-fold per token group: s_tau,d * (raw partial) + z_tau,d * sum_t w_t
    const int tau_rel = rel0 / C::G;
    const __half* s_tau = sm.vs + tau_rel * D;
    const __half* z_tau = sm.vz + tau_rel * D;
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
          st.o_run[mt][rh][v] = fmaf(s, raw, fmaf(z, psum_chunk[v], st.o_run[mt][rh][v]));
        }
      }
  }
}

// ------------------------------------------------------------------------
// The kernel: see the file comment. C = Cfg<BITS, KL, VL, NT, LOG2G>.
// ------------------------------------------------------------------------
template <class C>
__global__ void __launch_bounds__(kThreads, 1) split_decode_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int BITS = C::BITS, KL = C::KL, VL = C::VL, NT = C::NT, GV = C::GV, NTV = C::NTV;
  constexpr int RB = C::RB, D = kHeadDim;
  constexpr unsigned FULLMASK = 0xffffffffu;
  extern __shared__ __align__(1024) uint8_t smem[];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int hq = p.hq;
  const int unit = b * p.Hkv + kvh;
  const int L = min(max(p.seq_lens[b], 0), p.T_cap);  // device value: clamped, never trusted

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);      // full[kMaxRing], empty[kMaxRing]
  float* sQ = reinterpret_cast<float*>(smem + kBarBytes);  // [kMaxHq][D]
  float* sAq = sQ + kMaxHq * D;                            // [kMaxHq] token-wise K score factor
  int* sEq = reinterpret_cast<int*>(sAq + kMaxHq);         // [kMaxHq] query exponent
  float* sBz = sAq + 2 * kMaxHq;                           // [kMaxHq][4] offset factor per channel group
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
      const size_t blocks = (size_t)p.T_cap / C::G;
      int issued = 0, r = 0, phase = 0;
      for (int j = 0; j < n; ++j) {
        if (j >= p.n_ring && !mbar_wait(empty_bar(r), phase ^ 1, p.status, kStatusProducerTimeout)) break;
        const size_t t0 = (size_t)(j0 + j) * kSlotTokens;
        const size_t row0 = (size_t)unit * p.T_cap + t0;
        const uint32_t dst = ring0 + (uint32_t)r * p.slot_bytes;
        const uint32_t fb = full_bar(r);
        mbar_arrive_expect_tx(fb, p.slot_tx);
        bulk_g2s(dst, p.k_codes + row0 * RB, kSlotTokens * RB, fb, pol);
        bulk_g2s(dst + p.off_vc, p.v_codes + row0 * RB, kSlotTokens * RB, fb, pol);
        const size_t ks0 = (KL == 0) ? row0 * C::GK : ((size_t)unit * blocks + t0 / C::G) * kHeadDim;
        const size_t vs0 = (VL == 0) ? row0 * C::GV : ((size_t)unit * blocks + t0 / C::G) * kHeadDim;
        bulk_g2s(dst + p.off_ks, p.k_scale + ks0, p.sz_k_bytes, fb, pol);
        bulk_g2s(dst + p.off_kz, p.k_off + ks0, p.sz_k_bytes, fb, pol);
        bulk_g2s(dst + p.off_vs, p.v_scale + vs0, p.sz_v_bytes, fb, pol);
        bulk_g2s(dst + p.off_vz, p.v_off + vs0, p.sz_v_bytes, fb, pol);
        issued = j + 1;
        if (++r == p.n_ring) {
          r = 0;
          phase ^= 1;
        }
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
        amax = fmaxf(amax, fabsf(v) * (1.f / k_mult<BITS>(ch)));
        gs += v;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(FULLMASK, amax, o));
      // channel-group sums of Q (token-wise K offset term): lanes of one group are contiguous
      constexpr int lanes_per_group = C::G / 4;  // 8, 16 or 32
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float other = __shfl_xor_sync(FULLMASK, gs, o);
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

    WarpState<C> st;
    const int qi_b = g >> 1, qpart = g & 1;
    if (KL == 0) {
      // token-wise K: the exact hi/lo split of Q * 2^e / position factor, fixed for the CTA
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
              x[j] = live ? sQ[i * D + ch] * sc * (1.f / k_mult<BITS>(ch)) : 0.f;
            }
            st.qB[ks][nt][r] = pack_split4(x, qpart);
          }
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      st.qrow[nt] = min(c + 4 * nt, hq - 1);
      st.sA[nt] = sAq[st.qrow[nt]];
      st.m_run[nt] = -INFINITY;
      st.l_part[nt] = 0.f;
#pragma unroll
      for (int u = 0; u < GV; ++u) st.zacc[nt][u] = 0.f;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int rh = 0; rh < 2; ++rh)
#pragma unroll
        for (int v = 0; v < NTV; ++v) st.o_run[mt][rh][v] = 0.f;

    const int quad = warp >> 2, sub = warp & 3;
    const int rel0 = kChunk * sub;  // chunk start inside a slot
    int r = quad, phase = 0;        // ring slot and its phase for slot j
    for (int j = quad; j < n; j += kQuads) {
      if (!mbar_wait(full_bar(r), phase, p.status, kStatusConsumerTimeout)) {
        failed = true;
        break;
      }
      const uint8_t* slot = ring + (size_t)r * p.slot_bytes;
      ChunkSmem sm;
      sm.kc = slot;
      sm.vc = slot + p.off_vc;
      sm.ks = reinterpret_cast<const __half*>(slot + p.off_ks);
      sm.kz = reinterpret_cast<const __half*>(slot + p.off_kz);
      sm.vs = reinterpret_cast<const __half*>(slot + p.off_vs);
      sm.vz = reinterpret_cast<const __half*>(slot + p.off_vz);
      sm.sQ = sQ;
      sm.sBz = sBz;
      const int tc = (j0 + j) * kSlotTokens + rel0;  // chunk start token
      const int nv = min(kChunk, L - tc);            // valid tokens in the chunk
      if (nv == kChunk)
        process_chunk<C, true>(st, sm, rel0, nv, hq, p.sl2, lane);
      else if (nv > 0)
        process_chunk<C, false>(st, sm, rel0, nv, hq, p.sl2, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(r));
      r += kQuads;
      if (r >= p.n_ring) {
        r -= p.n_ring;
        phase ^= 1;
      }
    }

    // ---------------------------------------------------- warp results
    if (!window_cta) {
      named_sync(1, 32 * kConsumerWarps);  // every slot consumed: the ring is free
      float* sM = reinterpret_cast<float*>(ring);  // [warps][kMaxHq]
      float* sL = sM + kConsumerWarps * kMaxHq;    // [warps][kMaxHq]
      float* sO = sL + kConsumerWarps * kMaxHq;    // [warps][kMaxHq][D]
      float zsum[NT][GV];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float l = st.l_part[nt];
        l += __shfl_xor_sync(FULLMASK, l, 4);
        l += __shfl_xor_sync(FULLMASK, l, 8);
        l += __shfl_xor_sync(FULLMASK, l, 16);
#pragma unroll
        for (int u = 0; u < GV; ++u) {
          float z = st.zacc[nt][u];
          z += __shfl_xor_sync(FULLMASK, z, 4);
          z += __shfl_xor_sync(FULLMASK, z, 8);
          z += __shfl_xor_sync(FULLMASK, z, 16);
          zsum[nt][u] = z;
        }
        const int i = c + 4 * nt;
        if (g == 0 && i < hq) {
          sM[warp * kMaxHq + i] = st.m_run[nt];
          sL[warp * kMaxHq + i] = l;
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
            const float x = __shfl_sync(FULLMASK, zsum[ntq][uu], i & 3);
            if (uu == u) zt = x;
          }
        }
        const bool mine = (i < hq) && (GV == 1 || (16 * g) / (kHeadDim / GV) == u);
        if (mine) {
#pragma unroll
          for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int rh = 0; rh < 2; ++rh)
              sO[(warp * kMaxHq + i) * D + 16 * g + 2 * mt + rh] = st.o_run[mt][rh][v] + zt;
        }
      }
    }
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
        for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(FULLMASK, d, off);
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

  // ---------------------------------------------------- the last split merges all splits
  // out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s (zero when no token at all).
  __shared__ int s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();  // this CTA's partial is visible before the count says so
    const int prev = atomicAdd(p.done + unit, 1);
    s_last = (prev == p.s_tot - 1);
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    for (int idx = threadIdx.x; idx < hq * D; idx += kThreads) {
      const int i = idx / D, ch = idx % D;
      const size_t row = (size_t)b * p.Hq + kvh * hq + i;
      const float2* ml = p.part_ml + row * p.s_tot;
      const float* po = p.part_o + row * p.s_tot * D;
      float M = -INFINITY;
      for (int sp = 0; sp < p.s_tot; ++sp) M = fmaxf(M, __ldcg(&ml[sp].x));
      float acc = 0.f, l = 0.f;
      if (M != -INFINITY) {
        for (int sp = 0; sp < p.s_tot; ++sp) {
          const float2 x = __ldcg(&ml[sp]);
          const float sc = (x.x == -INFINITY) ? 0.f : fast_exp2(x.x - M);
          l = fmaf(sc, x.y, l);
          acc = fmaf(sc, __ldcg(&po[(size_t)sp * D + ch]), acc);
        }
      }
      p.out[row * D + ch] = __float2bfloat16_rn(l > 0.f ? acc / l : 0.f);
    }
    if (threadIdx.x == 0) p.done[unit] = 0;  // ready for the next call in stream order
  }
}

}  // namespace lbkv
