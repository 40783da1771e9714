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
// Operands. OR-ing a code q (times a power-of-two position factor m) into the
// mantissa of the fp16 magic number 1024 gives the exact fp16 value 1024 + m q,
// two codes per LOP3; the factor 1/m is folded into the other operand and the
// bias 1024 is cancelled inside the tensor core by starting each accumulator at
// -1024 * (sum of the other operand as fed). The bf16 query is exact in fp16;
// the softmax weights are fed as fp16 (11 bits), and the running denominator
// and the value offsets are summed from the weights actually fed, so the result
// is an exact attention under the fed weights. Both products run on mma.sync
// m16n8k16 fp16 with fp32 accumulators (on sm_103 this is a native tensor-core
// instruction; the e4m3 form is not, it converts its operands to fp16 first):
//   QK^T: rows = 16 tokens, k = 16 channels, cols = queries;
//   PV:   rows = 16 channels, k = 16 tokens, cols = (query[, channel group]).
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
template <int BITS_, int KL_, int VL_, int NTV_, int LOG2G_>
struct Cfg {
  static constexpr int BITS = BITS_, KL = KL_, VL = VL_, NTV = NTV_;
  static constexpr int G = 1 << LOG2G_;                    // group size
  static constexpr int GK = (KL == 0) ? kHeadDim / G : 1;  // K channel groups per token
  static constexpr int GV = (VL == 0) ? kHeadDim / G : 1;  // V channel groups per token
  static constexpr int KSG = G / 16;                       // QK k-steps per K channel group
  static constexpr int RB = kHeadDim * BITS / 8;           // bytes per token row of codes
  static_assert(NTV >= 1 && NTV <= 2, "one or two PV n-tiles");
  static_assert(G >= kChunk, "a chunk never straddles a token group");
};

// Channel fed at k-slot kappa (0..15) of QK^T k-step ks (0..7); see the K operand build.
template <int BITS>
__device__ __forceinline__ int qk_channel(int ks, int kappa) {
  const int blk = ks >> 1, h = ks & 1, c = (kappa & 7) >> 1, e = kappa & 1, up = kappa >> 3;
  const int p = 2 * h + up;
  if (BITS == 2) return 32 * blk + 16 * (c >> 1) + 4 * (c & 1) + 8 * e + p;
  return 32 * blk + 8 * c + 4 * e + p;
}
// Power-of-two position factor of the fp16 image of K channel ch (1024 + factor * q).
template <int BITS>
__device__ __forceinline__ float k_mult(int ch) {
  if (BITS == 2) return (float)(1 << (2 * (ch & 3)));
  return (ch & 1) ? 16.f : 1.f;
}
// Position factor of V m-tile mt (both of its rows).
template <int BITS>
__host__ __device__ constexpr float v_mult(int mt) {
  return BITS == 2 ? (float)(1 << (2 * (mt <= 4 ? mt : mt - 5))) : ((mt & 1) ? 16.f : 1.f);
}

// fp16 images (1024 + factor * code) of position p of an 8-code (INT2) or 4-code
// (INT4) group of two 16-bit halves: one LOP3 (plus a shared shift).
__device__ __forceinline__ uint32_t int2_half2(uint32_t x, uint32_t xs10, int p) {
  return p <= 4 ? and_or(x, 0x00030003u << (2 * p), kMagic2) : and_or(xs10, 0x00030003u << (2 * (p - 5)), kMagic2);
}
__device__ __forceinline__ uint32_t int4_half2(uint32_t x, uint32_t xs8, int p) {
  const uint32_t src = p < 2 ? x : xs8;
  return and_or(src, (p & 1) ? 0x00F000F0u : 0x000F000Fu, kMagic2);
}

// Per-warp state, held in registers. Each lane scores queries 2c and 2c+1.
template <class C>
struct WarpState {
  uint32_t qB[8][2];      // QK^T B fragments (fp16 pairs of Q' = Q 2^e / factor)
  float c1[2][C::GK];     // token-wise K: 1024 * sum of Q' over a channel group (magic bias)
  float aq[2];            // token-wise K: sigma log2(e) 2^-e
  float bz[2][C::GK];     // token-wise K: sigma log2(e) sum of Q over a channel group
  float m_run[2], l_part[2], zacc[2][C::GV];
  float o_run[8][2][C::NTV][2];  // [m-tile][row half][n-tile][column]
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
  const int* sEq;
};

// One 32-token chunk: QK^T with the K fold, online softmax, weights, PV with the
// V fold. FULL: all 32 tokens valid (no masking).
template <class C, bool FULL>
__device__ __forceinline__ void process_chunk(WarpState<C>& st, const ChunkSmem& sm, int rel0, int nv, int hq,
                                              float sl2, int lane) {
  constexpr int BITS = C::BITS, KL = C::KL, VL = C::VL, GV = C::GV, GK = C::GK, NTV = C::NTV;
  constexpr int RB = C::RB, D = kHeadDim;
  constexpr unsigned FULLMASK = 0xffffffffu;
  const int g = lane >> 2, c = lane & 3;

  // ---------------------------------------------------- channel-wise K: Q' per token group
  // Operand-fold: Q' = Q * s_tau / factor, scaled by 2^e into fp16; the offset becomes
  // sum_d Q_d z_tau,d, one constant per (query, token group), added before the softmax.
  float cwA[2] = {0.f, 0.f}, cwB[2] = {0.f, 0.f}, cwC[2] = {0.f, 0.f};
  if (KL == 1) {
    const int tau_rel = rel0 / C::G;
    const __half* s_tau = sm.ks + tau_rel * D;
    const __half* z_tau = sm.kz + tau_rel * D;
    const int q = g;  // this lane's B column
    const bool live = q < hq;
    float x[8][2][2];
    float amax = 0.f, zsum = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int ch = qk_channel<BITS>(ks, 2 * c + 8 * r + e);
          const float qv = live ? sm.sQ[q * D + ch] : 0.f;
          const float v = qv * __half2float(s_tau[ch]) * (1.f / k_mult<BITS>(ch));
          x[ks][r][e] = v;
          amax = fmaxf(amax, fabsf(v));
          zsum = fmaf(qv, __half2float(z_tau[ch]), zsum);
        }
    amax = fmaxf(amax, __shfl_xor_sync(FULLMASK, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(FULLMASK, amax, 2));
    zsum += __shfl_xor_sync(FULLMASK, zsum, 1);
    zsum += __shfl_xor_sync(FULLMASK, zsum, 2);
    int e2 = 0;
    if (amax > 0.f) e2 = min(100, max(-100, 13 - ilog2f(amax)));
    const float sc = exp2i(e2);
    float fed = 0.f;  // sum of the fp16 values actually fed (for the magic bias)
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const uint32_t h2 = f16x2_from(x[ks][r][0] * sc, x[ks][r][1] * sc);
        st.qB[ks][r] = h2;
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
        fed += f.x + f.y;
      }
    fed += __shfl_xor_sync(FULLMASK, fed, 1);
    fed += __shfl_xor_sync(FULLMASK, fed, 2);
    const float fa = sl2 * exp2i(-e2), fb = sl2 * zsum, fc = kMagicF * fed;
#pragma unroll
    for (int ql = 0; ql < 2; ++ql) {  // query 2c + ql is B column 2c + ql, held by lane 8c + 4ql
      cwA[ql] = __shfl_sync(FULLMASK, fa, 8 * c + 4 * ql);
      cwB[ql] = __shfl_sync(FULLMASK, fb, 8 * c + 4 * ql);
      cwC[ql] = __shfl_sync(FULLMASK, fc, 8 * c + 4 * ql);
    }
  }

  // ---------------------------------------------------- QK^T with the K fold
  // S[mt][row][ql]: token 16 mt + 8 row + g of the chunk, query 2c + ql (log2 domain).
  float S[2][2][2];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    const int row0 = rel0 + 16 * mt + g;
    const int row1 = row0 + 8;
    const uint32_t* r0p = reinterpret_cast<const uint32_t*>(sm.kc + row0 * RB);
    const uint32_t* r1p = reinterpret_cast<const uint32_t*>(sm.kc + row1 * RB);
    uint32_t w0[4], w1[4], s0w[4], s1w[4];
#pragma unroll
    for (int blk = 0; blk < 4; ++blk) {
      if (BITS == 2) {
        // lanes with odd c take codes 4..7 and 12..15 of the word: shift them into 0..3
        const int sh = 8 * (c & 1);
        w0[blk] = r0p[2 * blk + (c >> 1)] >> sh;
        w1[blk] = r1p[2 * blk + (c >> 1)] >> sh;
      } else {
        w0[blk] = r0p[4 * blk + c];
        w1[blk] = r1p[4 * blk + c];
        s0w[blk] = w0[blk] >> 8;
        s1w[blk] = w1[blk] >> 8;
      }
    }
    float sfold[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    float acc[4];
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int blk = ks >> 1, h = ks & 1;
      if (KL == 0 ? (ks % C::KSG == 0) : (ks == 0)) {
        // token-wise K: a fresh accumulator per channel group; channel-wise K: one for all
        // 128 channels (the scale is already in Q'). Each starts at minus the magic bias.
        const float b0 = (KL == 0) ? st.c1[0][ks / C::KSG] : cwC[0];
        const float b1 = (KL == 0) ? st.c1[1][ks / C::KSG] : cwC[1];
        acc[0] = -b0;
        acc[1] = -b1;
        acc[2] = -b0;
        acc[3] = -b1;
      }
      uint32_t a0, a1, a2, a3;
      if (BITS == 2) {
        const uint32_t mA = 0x00030003u << (4 * h), mB = 0x00030003u << (4 * h + 2);
        a0 = and_or(w0[blk], mA, kMagic2);
        a1 = and_or(w1[blk], mA, kMagic2);
        a2 = and_or(w0[blk], mB, kMagic2);
        a3 = and_or(w1[blk], mB, kMagic2);
      } else {
        a0 = int4_half2(w0[blk], s0w[blk], 2 * h);
        a1 = int4_half2(w1[blk], s1w[blk], 2 * h);
        a2 = int4_half2(w0[blk], s0w[blk], 2 * h + 1);
        a3 = int4_half2(w1[blk], s1w[blk], 2 * h + 1);
      }
      mma_f16(acc, a0, a1, a2, a3, st.qB[ks][0], st.qB[ks][1]);
      if (KL == 0 && (ks + 1) % C::KSG == 0) {
        // acc-fold of one channel group: s * (raw partial) + z * sum(Q over the group)
        const int grp = ks / C::KSG;
        const float s0 = __half2float(sm.ks[row0 * GK + grp]);
        const float z0 = __half2float(sm.kz[row0 * GK + grp]);
        const float s1 = __half2float(sm.ks[row1 * GK + grp]);
        const float z1 = __half2float(sm.kz[row1 * GK + grp]);
#pragma unroll
        for (int ql = 0; ql < 2; ++ql) {
          sfold[0][ql] = fmaf(s0 * st.aq[ql], acc[ql], fmaf(z0, st.bz[ql][grp], sfold[0][ql]));
          sfold[1][ql] = fmaf(s1 * st.aq[ql], acc[2 + ql], fmaf(z1, st.bz[ql][grp], sfold[1][ql]));
        }
      }
    }
#pragma unroll
    for (int ql = 0; ql < 2; ++ql) {
      float v0, v1;
      if (KL == 0) {
        v0 = sfold[0][ql];
        v1 = sfold[1][ql];
      } else {
        v0 = fmaf(cwA[ql], acc[ql], cwB[ql]);
        v1 = fmaf(cwA[ql], acc[2 + ql], cwB[ql]);
      }
      if (FULL) {
        S[mt][0][ql] = v0;
        S[mt][1][ql] = v1;
      } else {
        const int t0 = 16 * mt + g;
        S[mt][0][ql] = (t0 < nv) ? v0 : -INFINITY;
        S[mt][1][ql] = (t0 + 8 < nv) ? v1 : -INFINITY;
      }
    }
  }

  // ---------------------------------------------------- online softmax
  // This lane's tokens, chunk-relative: T_k = g + 8k, k = 2 mt + row.
  float P[2][4];
  float alpha[2];
  bool rescale = false;
#pragma unroll
  for (int ql = 0; ql < 2; ++ql) {
    float mx = fmaxf(fmaxf(S[0][0][ql], S[0][1][ql]), fmaxf(S[1][0][ql], S[1][1][ql]));
    mx = fmaxf(mx, __shfl_xor_sync(FULLMASK, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(FULLMASK, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(FULLMASK, mx, 16));
    const float m_new = fmaxf(st.m_run[ql], mx);
    rescale |= (m_new > st.m_run[ql]);
    alpha[ql] = (m_new == -INFINITY) ? 1.f : fast_exp2(st.m_run[ql] - m_new);
    const float mref = (m_new == -INFINITY) ? 0.f : m_new;
    st.m_run[ql] = m_new;
#pragma unroll
    for (int k = 0; k < 4; ++k) P[ql][k] = fast_exp2(S[k >> 1][k & 1][ql] - mref);
  }
  if (__any_sync(FULLMASK, rescale)) {
#pragma unroll
    for (int ql = 0; ql < 2; ++ql) {
      st.l_part[ql] *= alpha[ql];
#pragma unroll
      for (int u = 0; u < GV; ++u) st.zacc[ql][u] *= alpha[ql];
    }
    // output column 8v + 2c + e is combo (query, group) = ((8v + 2c + e) / GV, % GV)
#pragma unroll
    for (int v = 0; v < NTV; ++v)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float av;
        if (GV == 1 && NTV == 1) {
          av = alpha[e];
        } else {
          const int q = (8 * v + 2 * c + e) / GV;
          const float a0 = __shfl_sync(FULLMASK, alpha[0], 4 * g + (q >> 1));
          const float a1 = __shfl_sync(FULLMASK, alpha[1], 4 * g + (q >> 1));
          av = (q & 1) ? a1 : a0;
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          st.o_run[mt][0][v][e] *= av;
          st.o_run[mt][1][v][e] *= av;
        }
      }
  }

  // ---------------------------------------------------- weights -> fp16 words
  // Token-wise V (operand-fold): fed weight P_t * s_t,u * 2^eP per channel group u;
  // channel-wise V: P_t * 2^13. The denominator and value offsets are summed from
  // the fed weights w_t = fed / scale; the PV accumulators start at -1024 * sum(fed)
  // per column, which removes the magic bias of the V operand exactly.
  const int tok0 = rel0 + g;
  uint32_t pw[2][GV][2];  // [query][group][pair (T0,T1) / (T2,T3)]
  float colb[2][GV];      // -1024 * sum of fed weights over the chunk (reduced)
  float inv_ps = 1.f;
  float psum[2];          // channel-wise V: sum of fed weights over the chunk (reduced)
  if (VL == 0) {
    float sv[GV][4];
    uint32_t smax = 0;
#pragma unroll
    for (int u = 0; u < GV; ++u)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const bool ok = FULL || (g + 8 * k < nv);
        const __half hv = sm.vs[(tok0 + 8 * k) * GV + u];
        sv[u][k] = ok ? __half2float(hv) : 0.f;
        smax = max(smax, ok ? (uint32_t)(__half_as_ushort(hv) & 0x7fffu) : 0u);
      }
    smax = max(smax, __shfl_xor_sync(FULLMASK, smax, 4));
    smax = max(smax, __shfl_xor_sync(FULLMASK, smax, 8));
    smax = max(smax, __shfl_xor_sync(FULLMASK, smax, 16));
    const float smaxf = __half2float(__ushort_as_half((unsigned short)smax));
    int e2 = 0;
    if (smaxf > 0.f) e2 = min(100, max(-100, 13 - ilog2f(smaxf)));
    const float ps = exp2i(e2);
    inv_ps = exp2i(-e2);
#pragma unroll
    for (int ql = 0; ql < 2; ++ql) {
      float lsum = 0.f;
#pragma unroll
      for (int u = 0; u < GV; ++u) {
        float f[4];
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const uint32_t h2 = f16x2_from(P[ql][2 * kk] * sv[u][2 * kk] * ps, P[ql][2 * kk + 1] * sv[u][2 * kk + 1] * ps);
          pw[ql][u][kk] = h2;
          const float2 ff = __half22float2(*reinterpret_cast<const __half2*>(&h2));
          f[2 * kk] = ff.x;
          f[2 * kk + 1] = ff.y;
        }
        float zt = 0.f, fs = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float w = (sv[u][k] != 0.f) ? f[k] * (fast_rcp(sv[u][k]) * inv_ps) : P[ql][k];
          const bool ok = FULL || (g + 8 * k < nv);
          const float zz = ok ? __half2float(sm.vz[(tok0 + 8 * k) * GV + u]) : 0.f;
          zt = fmaf(w, zz, zt);
          fs += f[k];
          if (u == 0) lsum += w;
        }
        st.zacc[ql][u] += zt;
        fs += __shfl_xor_sync(FULLMASK, fs, 4);
        fs += __shfl_xor_sync(FULLMASK, fs, 8);
        fs += __shfl_xor_sync(FULLMASK, fs, 16);
        colb[ql][u] = -kMagicF * fs;
      }
      st.l_part[ql] += lsum;
      psum[ql] = 0.f;
    }
  } else {
#pragma unroll
    for (int ql = 0; ql < 2; ++ql) {
      float fs = 0.f;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const uint32_t h2 = f16x2_from(P[ql][2 * kk] * 8192.f, P[ql][2 * kk + 1] * 8192.f);
        pw[ql][0][kk] = h2;
        const float2 ff = __half22float2(*reinterpret_cast<const __half2*>(&h2));
        fs += ff.x + ff.y;
      }
      st.l_part[ql] += fs * (1.f / 8192.f);
      fs += __shfl_xor_sync(FULLMASK, fs, 4);
      fs += __shfl_xor_sync(FULLMASK, fs, 8);
      fs += __shfl_xor_sync(FULLMASK, fs, 16);
      psum[ql] = fs * (1.f / 8192.f);
      colb[ql][0] = -kMagicF * fs;
    }
  }

  // ---------------------------------------------------- PV B fragments and accumulator start
  // B column n = g of n-tile v is combo 8v + g; k-slots 2c, 2c+1 of PV k-step kk hold
  // chunk tokens c + 16kk and c + 8 + 16kk (the pair kk of lane 4c + q/2), and k-slots
  // 2c+8, 2c+9 the same tokens of lane 4(c+4) + q/2.
  uint32_t pB[NTV][2][2];  // [n-tile][kk][reg]
#pragma unroll
  for (int v = 0; v < NTV; ++v) {
    const int col = 8 * v + g;
    const int q = col / GV, u_need = col % GV;
    const int src0 = 4 * c + (q >> 1), src1 = 4 * (c + 4) + (q >> 1);
    const bool live = q < hq;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      uint32_t b0 = 0, b1 = 0;
#pragma unroll
      for (int ql = 0; ql < 2; ++ql)
#pragma unroll
        for (int u = 0; u < GV; ++u) {
          const uint32_t x0 = __shfl_sync(FULLMASK, pw[ql][u][kk], src0);
          const uint32_t x1 = __shfl_sync(FULLMASK, pw[ql][u][kk], src1);
          if (ql == (q & 1) && u == u_need) {
            b0 = x0;
            b1 = x1;
          }
        }
      pB[v][kk][0] = live ? b0 : 0u;
      pB[v][kk][1] = live ? b1 : 0u;
    }
  }
  float cb[NTV][2];  // starting value of output column 8v + 2c + e
#pragma unroll
  for (int v = 0; v < NTV; ++v)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      if (GV == 1 && NTV == 1) {
        cb[v][e] = colb[e][0];
      } else {
        const int col = 8 * v + 2 * c + e;
        const int q = col / GV, u_need = col % GV;
        float x = 0.f;
#pragma unroll
        for (int ql = 0; ql < 2; ++ql)
#pragma unroll
          for (int u = 0; u < GV; ++u) {
            const float y = __shfl_sync(FULLMASK, colb[ql][u], 4 * g + (q >> 1));
            if (ql == (q & 1) && u == u_need) x = y;
          }
        cb[v][e] = x;
      }
    }

  // ---------------------------------------------------- PV
  // Row half `row` of m-tile mt is channel 16g + 8row + mt (INT2) or
  // 16g + 8(mt/4) + 4row + mt%4 (INT4), with factor v_mult(mt).
  float accv[8][NTV][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int v = 0; v < NTV; ++v) {
      accv[mt][v][0] = cb[v][0];
      accv[mt][v][1] = cb[v][1];
      accv[mt][v][2] = cb[v][0];
      accv[mt][v][3] = cb[v][1];
    }
#pragma unroll
  for (int kk = 0; kk < 2; ++kk) {
    const int tA = rel0 + c + 16 * kk, tB = tA + 4;
    if (BITS == 2) {
      const uint32_t wa0 = reinterpret_cast<const uint32_t*>(sm.vc + tA * RB)[g];
      const uint32_t wa1 = reinterpret_cast<const uint32_t*>(sm.vc + (tA + 8) * RB)[g];
      const uint32_t wb0 = reinterpret_cast<const uint32_t*>(sm.vc + tB * RB)[g];
      const uint32_t wb1 = reinterpret_cast<const uint32_t*>(sm.vc + (tB + 8) * RB)[g];
      const uint32_t xal = prmt(wa0, wa1, 0x5410), xah = prmt(wa0, wa1, 0x7632);
      const uint32_t xbl = prmt(wb0, wb1, 0x5410), xbh = prmt(wb0, wb1, 0x7632);
      const uint32_t sal = xal >> 10, sah = xah >> 10, sbl = xbl >> 10, sbh = xbh >> 10;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const uint32_t a0 = int2_half2(xal, sal, mt), a1 = int2_half2(xah, sah, mt);
        const uint32_t a2 = int2_half2(xbl, sbl, mt), a3 = int2_half2(xbh, sbh, mt);
#pragma unroll
        for (int v = 0; v < NTV; ++v) mma_f16(accv[mt][v], a0, a1, a2, a3, pB[v][kk][0], pB[v][kk][1]);
      }
    } else {
      const uint2 wa0 = reinterpret_cast<const uint2*>(sm.vc + tA * RB)[g];
      const uint2 wa1 = reinterpret_cast<const uint2*>(sm.vc + (tA + 8) * RB)[g];
      const uint2 wb0 = reinterpret_cast<const uint2*>(sm.vc + tB * RB)[g];
      const uint2 wb1 = reinterpret_cast<const uint2*>(sm.vc + (tB + 8) * RB)[g];
#pragma unroll
      for (int uu = 0; uu < 2; ++uu) {
        const uint32_t ea0 = uu ? wa0.y : wa0.x, ea1 = uu ? wa1.y : wa1.x;
        const uint32_t eb0 = uu ? wb0.y : wb0.x, eb1 = uu ? wb1.y : wb1.x;
        const uint32_t xal = prmt(ea0, ea1, 0x5410), xah = prmt(ea0, ea1, 0x7632);
        const uint32_t xbl = prmt(eb0, eb1, 0x5410), xbh = prmt(eb0, eb1, 0x7632);
        const uint32_t sal = xal >> 8, sah = xah >> 8, sbl = xbl >> 8, sbh = xbh >> 8;
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
          const int mt = 4 * uu + pp;
          const uint32_t a0 = int4_half2(xal, sal, pp), a1 = int4_half2(xah, sah, pp);
          const uint32_t a2 = int4_half2(xbl, sbl, pp), a3 = int4_half2(xbh, sbh, pp);
#pragma unroll
          for (int v = 0; v < NTV; ++v) mma_f16(accv[mt][v], a0, a1, a2, a3, pB[v][kk][0], pB[v][kk][1]);
        }
      }
    }
  }

  // ---------------------------------------------------- V fold into the running output
  if (VL == 0) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const float f = inv_ps * (1.f / v_mult<BITS>(mt));
#pragma unroll
      for (int v = 0; v < NTV; ++v)
#pragma unroll
        for (int row = 0; row < 2; ++row)
#pragma unroll
          for (int e = 0; e < 2; ++e) st.o_run[mt][row][v][e] = fmaf(accv[mt][v][2 * row + e], f, st.o_run[mt][row][v][e]);
    }
  } else {
    // acc-fold per token group: s_tau,d * (raw partial) + z_tau,d * sum_t w_t
    const int tau_rel = rel0 / C::G;
    const __half* s_tau = sm.vs + tau_rel * D;
    const __half* z_tau = sm.vz + tau_rel * D;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int row = 0; row < 2; ++row) {
        const int ch = (BITS == 2) ? 16 * g + 8 * row + mt : 16 * g + 8 * (mt >> 2) + 4 * row + (mt & 3);
        const float s = __half2float(s_tau[ch]) * (1.f / (8192.f * v_mult<BITS>(mt)));
        const float z = __half2float(z_tau[ch]);
#pragma unroll
        for (int e = 0; e < 2; ++e)
          st.o_run[mt][row][0][e] = fmaf(s, accv[mt][0][2 * row + e], fmaf(z, psum[e], st.o_run[mt][row][0][e]));
      }
  }
}

// ------------------------------------------------------------------------
// The kernel: see the file comment. C = Cfg<BITS, KL, VL, NT, LOG2G>.
// ------------------------------------------------------------------------
template <class C>
__global__ void __launch_bounds__(kThreads, 1) split_decode_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int BITS = C::BITS, KL = C::KL, VL = C::VL, GV = C::GV, GK = C::GK, NTV = C::NTV;
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
      // query exponent e: max |Q / factor| * 2^e in [2^13, 2^14), so Q * 2^e / factor is an
      // exact fp16 (a bf16 has 8 significant bits); channel-group sums of Q for the K offset
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
      constexpr int lanes_per_group = C::G / 4;  // 8, 16 or 32
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float other = __shfl_xor_sync(FULLMASK, gs, o);
        if (o < lanes_per_group) gs += other;
      }
      int e = 0;
      if (amax > 0.f) e = min(100, max(-100, 13 - ilog2f(amax)));
      if (lane == 0) {
        sEq[i] = e;
        sAq[i] = p.sl2 * exp2i(-e);
      }
      if (KL == 0 && (lane % lanes_per_group) == 0) sBz[i * 4 + lane / lanes_per_group] = p.sl2 * gs;
    }
    named_sync(1, 32 * kConsumerWarps);

    WarpState<C> st;
    if (KL == 0) {
      // token-wise K: B fragments Q' = Q 2^e / factor (exact fp16), fixed for the CTA, and
      // the magic bias 1024 * sum of Q' per channel group
      const int q = g;
      const bool live = q < hq;
      const float sc = live ? exp2i(sEq[q]) : 0.f;
      float gsum[GK];
#pragma unroll
      for (int u = 0; u < GK; ++u) gsum[u] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          float x[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int ch = qk_channel<BITS>(ks, 2 * c + 8 * r + e);
            x[e] = live ? sQ[q * D + ch] * sc * (1.f / k_mult<BITS>(ch)) : 0.f;
          }
          st.qB[ks][r] = f16x2_from(x[0], x[1]);
          gsum[ks / C::KSG] += x[0] + x[1];
        }
#pragma unroll
      for (int u = 0; u < GK; ++u) {
        gsum[u] += __shfl_xor_sync(FULLMASK, gsum[u], 1);
        gsum[u] += __shfl_xor_sync(FULLMASK, gsum[u], 2);
      }
#pragma unroll
      for (int ql = 0; ql < 2; ++ql) {  // query 2c + ql is B column 2c + ql, held by lane 8c + 4ql
        const int qq = min(2 * c + ql, hq - 1);
        st.aq[ql] = sAq[qq];
#pragma unroll
        for (int u = 0; u < GK; ++u) {
          st.c1[ql][u] = kMagicF * __shfl_sync(FULLMASK, gsum[u], 8 * c + 4 * ql);
          st.bz[ql][u] = sBz[qq * 4 + u];
        }
      }
    }
#pragma unroll
    for (int ql = 0; ql < 2; ++ql) {
      st.m_run[ql] = -INFINITY;
      st.l_part[ql] = 0.f;
#pragma unroll
      for (int u = 0; u < GV; ++u) st.zacc[ql][u] = 0.f;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int row = 0; row < 2; ++row)
#pragma unroll
        for (int v = 0; v < NTV; ++v) st.o_run[mt][row][v][0] = st.o_run[mt][row][v][1] = 0.f;

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
      sm.sEq = sEq;
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
      float zsum[2][GV];
#pragma unroll
      for (int ql = 0; ql < 2; ++ql) {
        float l = st.l_part[ql];
        l += __shfl_xor_sync(FULLMASK, l, 4);
        l += __shfl_xor_sync(FULLMASK, l, 8);
        l += __shfl_xor_sync(FULLMASK, l, 16);
#pragma unroll
        for (int u = 0; u < GV; ++u) {
          float z = st.zacc[ql][u];
          z += __shfl_xor_sync(FULLMASK, z, 4);
          z += __shfl_xor_sync(FULLMASK, z, 8);
          z += __shfl_xor_sync(FULLMASK, z, 16);
          zsum[ql][u] = z;
        }
        const int i = 2 * c + ql;
        if (g == 0 && i < hq) {
          sM[warp * kMaxHq + i] = st.m_run[ql];
          sL[warp * kMaxHq + i] = l;
        }
      }
      // output column 8v + 2c + e is (query, group) = (col / GV, col % GV); its channels are
      // this lane's 16, all in channel group 16g / G
      const int u_lane = (16 * g) / C::G;
#pragma unroll
      for (int v = 0; v < NTV; ++v)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int col = 8 * v + 2 * c + e;
          const int i = col / GV, u = col % GV;
          float zt = 0.f;
          if (VL == 0) {  // the value-offset term of (query i, group u) lives on lane i/2
#pragma unroll
            for (int ql = 0; ql < 2; ++ql)
#pragma unroll
              for (int uu = 0; uu < GV; ++uu) {
                const float x = __shfl_sync(FULLMASK, zsum[ql][uu], i >> 1);
                if (ql == (i & 1) && uu == u) zt = x;
              }
          }
          if (i < hq && (GV == 1 || u == u_lane)) {
#pragma unroll
            for (int mt = 0; mt < 8; ++mt)
#pragma unroll
              for (int row = 0; row < 2; ++row) {
                const int ch = (BITS == 2) ? 16 * g + 8 * row + mt : 16 * g + 8 * (mt >> 2) + 4 * row + (mt & 3);
                sO[(warp * kMaxHq + i) * D + ch] = st.o_run[mt][row][v][e] + zt;
              }
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
