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
// Kernel design (sm_103a). A persistent grid, one CTA per SM (fewer for small
// problems). The tokens of all (sequence, KV head) pairs form items of 32, 64 or
// 128 tokens in one sequence; each CTA takes a contiguous share of it, equal once
// every pair boundary is counted as a fixed amount of work (see the work split
// below), and deals it to its warps (16, or 8) in turn.
// Each warp streams its items' packed codes and fp16 scales/offsets through its
// own ring in shared memory with 1-D bulk copies that it issues itself (an
// mbarrier per entry, bounded waits, no multicast), so no warp waits on
// another's progress. Per item a warp scores all its tokens (QK^T with the K
// fold), updates its running maximum once, then forms the weights and
// accumulates PV chunk by chunk with the V fold. Where the CTA's share moves to
// the next pair, its warps merge into one partial for the pair; the last CTA of
// a pair to finish merges the pair's partials into the bf16 output. A bf16
// window after the cached tokens is scored by a separate small kernel first.
// A paged cache (the PAGED variant) changes only the source addresses of the bulk
// copies. A cache stored rotated by the Hadamard matrix has the query rotated in
// the pair prologue and each output row rotated back before its bf16 rounding.
//
// Operands. A code q (times a power-of-two position factor m) masked into the
// mantissa bits of an fp16 half, with the exponent bits left at zero, is the exact
// fp16 subnormal m q 2^-24: two codes per LOP3, no bias. The factor 1/m is folded
// into the other operand and the 2^-24 into the fold constants (scores and outputs
// are kept in units that carry the 2^24). The tensor cores take the subnormals
// exactly; measured on this GPU against fp64 sums of query-like operands, the error
// of a product is 5e-6 of sum |q b|, against 7e-5 with the images 1024 + m q of the
// magic number 1024 and their bias removed (the large biased terms cost precision).
// The bf16 query is exact in fp16 (a rotated query is rounded to it); the
// softmax weights are fed as fp16.
// Both products run on mma.sync m16n8k16 fp16 with fp32 accumulators (native
// on sm_103; the e4m3 form of mma.sync converts its operands to fp16 first):
//   QK^T: rows = 16 tokens, k = 16 channels, cols = queries;
//   PV:   rows = 16 channels, k = 16 tokens, cols = (query, V channel group).
//
// Columns. The (query, V channel group) pairs of one KV head ("combos";
// hq * GV of them, GV = channel groups of a token-wise V side, else 1) sit on
// the 8 columns of the tiles in one of three modes: up to 4 combos, each on
// two adjacent columns (a lane then handles one combo); 8 combos, one per
// column; 16 combos on two PV n-tiles.
#pragma once

#include "lbkv_device.cuh"

namespace lbkv {

constexpr int kHeadDim = 128;
constexpr int kSlotTokens = 128;
constexpr int kChunk = 32;  // tokens of one QK^T / PV tile pass
constexpr int kMaxRing = 48;    // ring entries of all warps (one mbarrier each)
constexpr int kMergeWarps = 8;  // warps whose partials the CTA merge reads; any others fold into them first
constexpr int kWinWarps = 8;    // warps of the window kernel
constexpr int kMaxHq = 8;
// shared-memory map: barriers | Q (fp32) and per-query constants | merge area | rings
constexpr int kBarBytes = kMaxRing * 8;
constexpr int kPrologueBytes = 8192;
// token-wise K: the B fragments of Q' shared by all warps, [k-step][lane] pairs of words
constexpr int kQbOffset = kBarBytes + 4 * (kMaxHq * kHeadDim + 6 * kMaxHq);
static_assert(kQbOffset % 16 == 0 && kQbOffset + 8 * 32 * 8 <= kPrologueBytes, "prologue fits");
// channel-wise K: words per (query, lane c) row of the W fragments (16, padded so that the 16
// rows a warp reads at one k-step fall in different bank pairs)
constexpr int kWRow = 18;
static_assert(kQbOffset + 4 * kMaxHq * 4 * kWRow <= kPrologueBytes, "prologue fits");
// The tensor-core decode kernel (lbkv_decode_grp.cuh): shared-memory offset of its merge
// area, after its mbarriers, counters, prologue, query tile and weight tiles; its rings follow.
constexpr int kGrpMergeOffset = 7168 + 96 * 128 + 8192;
// Per-lane register state a warp beyond the first kMergeWarps hands over (floats):
// o_run (16 per live column, up to 2), zacc (up to 4), m and l (up to 2 each).
constexpr int kStateFloats = 16 * 2 + 4 + 2 * 2;
// Merge area for hq queries per KV head: per merge warp (m, l) of kMaxHq queries and o of
// hq queries; with more than kMergeWarps warps it also holds the handed-over states.
// Row stride (floats) of a deposited output row in the merge area: 4 past the head dim, so that
// a warp's deposit stores (query c, channels 16 g + p) fall in 8 banks instead of 2.
constexpr int kODep = kHeadDim + 4;
__host__ __device__ constexpr int merge_bytes(int hq, int warps) {
  const int deposit = 4 * kMergeWarps * (2 * kMaxHq + hq * kODep);
  const int states = (warps > kMergeWarps) ? 4 * kMergeWarps * 32 * kStateFloats : 0;
  return ((deposit > states ? deposit : states) + 127) / 128 * 128;
}

constexpr int kModeDup = 0;   // <= 4 combos: combo k on columns 2k, 2k+1
constexpr int kModePair = 1;  // 8 combos: combo k on column k
constexpr int kModeWide = 2;  // 16 combos: combo k on column k % 8 of PV n-tile k / 8

__host__ __device__ constexpr int decode_mode(int combos) {
  return combos <= 4 ? kModeDup : combos == 8 ? kModePair : combos == 16 ? kModeWide : -1;
}
// Warps per CTA: 16 (128 registers each), or 8 where a lane's state needs more
// registers: 16 pairs per KV head, or 8 pairs that are 8 different queries (two
// query slots per lane).
__host__ __device__ constexpr int decode_warps(int bits, int mode, int gv) {
  return (mode == kModeWide || (mode == kModePair && gv == 1)) ? 8 : 16;
}
// 32-token chunks per item, such that one ring entry per warp fits in shared memory:
// 128 tokens at INT2 (64 when group 32 makes the scales and offsets as large as a
// quarter of the codes), 64 at INT4 and for 16 pairs.
__host__ __device__ constexpr int unit_chunks(int bits, int mode, int log2g) {
  return mode == kModeWide ? 2 : bits == 2 ? (log2g == 5 ? 2 : 4) : 2;
}

// Byte layout of one ring entry (one item of `unit` tokens of one pair):
// K codes | K scales | K offsets | V codes | V scales | V offsets, each part 16-byte
// aligned; the K half and the V half are filled by separate bulk-copy groups.
struct EntryLayout {
  int sz_k, sz_v;                        // bytes of one scale (or offset) array, K and V side
  int off_ks, off_kz, off_vc, off_vs, off_vz;
  int tx_k, tx_v, bytes;                 // bytes of the K half, of the V half, entry stride
};
__host__ __device__ constexpr int sz_bytes(int layout, int unit, int g) {
  return layout == 0 ? unit * (kHeadDim / g) * 2 : (unit >= g ? unit / g : 1) * kHeadDim * 2;
}
__host__ __device__ constexpr EntryLayout entry_layout(int bits, int kl, int vl, int unit, int g) {
  const int rb = kHeadDim * bits / 8;
  const int szk = sz_bytes(kl, unit, g), szv = sz_bytes(vl, unit, g);
  const int off_ks = unit * rb, off_kz = off_ks + szk, off_vc = off_kz + szk;
  const int off_vs = off_vc + unit * rb, off_vz = off_vs + szv;
  return EntryLayout{szk, szv, off_ks, off_kz, off_vc, off_vs, off_vz, off_vc, unit * rb + 2 * szv,
                     (off_vz + szv + 127) / 128 * 128};
}

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
  float2* part_ml;  // [n_cta][2][hq] partials of the CTAs (running max in log2 units, denominator)
  float* part_o;    // [n_cta][2][hq][D] unnormalised output
  float2* win_ml;   // [B*Hkv][hq] the window's partial of each pair
  float* win_o;     // [B*Hkv][hq][D]
  int32_t* status;
  int32_t* done;    // [B*Hkv] CTAs finished with a pair; the last one merges and resets it to 0
  __nv_bfloat16* out;
  // Hkv, hq: KV heads and queries per KV head as the kernel sees them. With kv_shift = 1
  // every KV head is split into two halves of its queries (two "pairs" per KV head, each
  // reading the same cached data): the cached KV head of pair u is u >> kv_shift.
  int B, Hq, Hkv, hq, T_cap, win_cap, kv_shift;
  float sl2;  // softmax scale times log2(e)
  int n_cta, has_win;   // CTAs of the grid; whether a bf16 window is given
  int split_w;          // work split: the cost of a pair boundary, in items
  // Cluster mode: thread-block clusters per pair (1: the cluster writes the output; more: each
  // cluster writes its merged partial to the CTA partials, and the last one merges them)
  int cluster_split;
  int ring_off, ring_per_warp;  // shared-memory offset of the rings, entries per warp
  // Paged cache (the kernel's PAGED variant): token t of cached KV head kvh of sequence b
  // is row t mod 2^log2_page of page page_table[b * max_pages + t / 2^log2_page], in a
  // pool of num_pages pages of [Hkv][2^log2_page] rows.
  const int32_t* page_table;
  int log2_page, max_pages, num_pages;
  // Rotated cache: bit 0, the keys (cache and window) are stored as H k, so the scores
  // take H q; bit 1, the values are stored as H v, so the output is rotated back by H
  // (H: the normalized Hadamard matrix, symmetric and orthogonal).
  int rotation;
};

// Compile-time shape of one kernel variant.
template <int BITS_, int KL_, int VL_, int MODE_, int LOG2G_>
struct Cfg {
  static constexpr int BITS = BITS_, KL = KL_, VL = VL_, MODE = MODE_;
  static constexpr int G = 1 << LOG2G_;                    // group size
  static constexpr int GK = (KL == 0) ? kHeadDim / G : 1;  // K channel groups per token
  static constexpr int GV = (VL == 0) ? kHeadDim / G : 1;  // V channel groups per token
  static constexpr int KSG = G / 16;                       // QK k-steps per K channel group
  static constexpr int RB = kHeadDim * BITS / 8;           // bytes per token row of codes
  static constexpr bool DUP = (MODE == kModeDup);
  static constexpr int NTV = (MODE == kModeWide) ? 2 : 1;  // PV n-tiles
  // query slots per lane (QK^T accumulator columns 2c + j); owned combos per lane
  static constexpr int NQ = (MODE == kModeWide || (MODE == kModePair && GV == 1)) ? 2 : 1;
  static constexpr int NO = DUP ? 1 : 2 * NTV;
  static constexpr int NCH = unit_chunks(BITS, MODE, LOG2G_);  // chunks per item
  static constexpr int UNIT = kChunk * NCH;             // tokens per item
  static constexpr int WARPS = decode_warps(BITS, MODE, GV);
  static constexpr int THREADS = 32 * WARPS;
  static constexpr EntryLayout E = entry_layout(BITS, KL, VL, UNIT, G);
  static_assert(G >= kChunk, "a chunk never straddles a token group");
  static_assert(MODE != kModeWide || GV >= 2, "16 combos need several V channel groups");
};

// Query carried by QK^T column n, or -1 when the column carries no combo.
template <class C>
__device__ __forceinline__ int qk_query(int n, int hq) {
  if (C::DUP) {
    const int k = n >> 1;
    return k < hq * C::GV ? k / C::GV : -1;
  }
  if (C::MODE == kModePair) return n / C::GV;
  return (8 * (n & 1) + 2 * (n >> 1)) / C::GV;
}
// Owned combo o of lane c: its combo index, query slot and V channel group.
template <class C>
__device__ __forceinline__ int own_combo(int c, int o) {
  return C::DUP ? c : 8 * (o >> 1) + 2 * c + (o & 1);
}
template <class C>
__host__ __device__ constexpr int own_slot(int o) {
  return C::MODE == kModeWide ? (o >> 1) : (C::NQ == 2 ? o : 0);
}
template <class C>
__device__ __forceinline__ int own_group(int c, int o) {
  return C::DUP ? c % C::GV : (2 * c + (o & 1)) % C::GV;
}

// K operand mappings. Block mapping (token-wise K with several channel groups): each
// k-step stays inside one 32-channel block, lanes with odd c taking the upper byte of
// each 16-bit half. Wide mapping (one channel group, or channel-wise K): lane c takes
// whole words of its own 32 channels, all positions of each 16-bit half (positions
// past the 10-bit mantissa come from the word shifted right by 10 (INT2) or 8 (INT4)).
template <class C>
__device__ __forceinline__ constexpr bool qk_wide() {
  return C::GK == 1;
}
// Channel fed at k-slot kappa (0..15) of QK^T k-step ks (0..7).
template <class C>
__device__ __forceinline__ int qk_channel(int ks, int kappa) {
  const int c = (kappa & 7) >> 1, e = kappa & 1, up = kappa >> 3;
  if (qk_wide<C>()) {
    if (C::BITS == 2) return 16 * (2 * c + (ks >> 2)) + 8 * e + 2 * (ks & 3) + up;
    return 8 * (4 * c + (ks >> 1)) + 4 * e + 2 * (ks & 1) + up;
  }
  const int blk = ks >> 1, p = 2 * (ks & 1) + up;
  if (C::BITS == 2) return 32 * blk + 16 * (c >> 1) + 4 * (c & 1) + 8 * e + p;
  return 32 * blk + 8 * c + 4 * e + p;
}
// Power-of-two position factor of the fp16 image of K channel ch (factor * q * 2^-24).
template <class C>
__device__ __forceinline__ float k_mult(int ch) {
  if (C::BITS == 4) return (ch & 1) ? 16.f : 1.f;
  if (qk_wide<C>()) {
    const int p = ch & 7;
    return (float)(1 << (2 * (p <= 4 ? p : p - 5)));
  }
  return (float)(1 << (2 * (ch & 3)));
}
// Its exact reciprocal (a power of two formed directly, no division).
template <class C>
__device__ __forceinline__ float k_rmult(int ch) {
  if (C::BITS == 4) return (ch & 1) ? 0.0625f : 1.f;
  if (qk_wide<C>()) {
    const int p = ch & 7;
    return exp2i(-2 * (p <= 4 ? p : p - 5));
  }
  return exp2i(-2 * (ch & 3));
}
// Position factor of V m-tile mt (both of its rows).
template <int BITS>
__host__ __device__ constexpr float v_mult(int mt) {
  return BITS == 2 ? (float)(1 << (2 * (mt <= 4 ? mt : mt - 5))) : ((mt & 1) ? 16.f : 1.f);
}
// Offset, among the 16 channels 16g..16g+15 of a lane, of PV row half `row` of m-tile mt.
template <int BITS>
__host__ __device__ constexpr int pv_channel(int mt, int row) {
  return BITS == 2 ? 8 * row + mt : 8 * (mt >> 2) + 4 * row + (mt & 3);
}

// fp16 subnormal images (factor * code * 2^-24) of position p of an 8-code (INT2) or
// 4-code (INT4) group of two 16-bit halves: one AND (plus a shared shift). Positions
// past the 10 mantissa bits come from the word shifted right by 10 (INT2) or 8 (INT4).
__device__ __forceinline__ uint32_t int2_half2(uint32_t x, uint32_t xs10, int p) {
  return p <= 4 ? (x & (0x00030003u << (2 * p))) : (xs10 & (0x00030003u << (2 * (p - 5))));
}
__device__ __forceinline__ uint32_t int4_half2(uint32_t x, uint32_t xs8, int p) {
  const uint32_t src = p < 2 ? x : xs8;
  return src & ((p & 1) ? 0x00F000F0u : 0x000F000Fu);
}
// The 2^24 that brings an accumulator of subnormal images back to code units.
constexpr float kImageUnit = 16777216.f;

__device__ __forceinline__ float2 half2_to_float2(uint32_t h2) {
  return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}

// Per-warp state, held in registers.
template <class C>
struct WarpState {
  float pa[C::NQ];           // token-wise K: sigma log2(e) 2^-e (scores are kept in units of it); else 1
  float bzq[C::NQ][C::GK];   // token-wise K: 2^e * sum of Q over a channel group
  float m_run[C::NQ], l[C::NQ];
  float zacc[C::NO];         // token-wise V: sum_t P_t z_t per owned combo
  float o_run[8][2][C::NQ];  // [m-tile][row half][live column]
};

// Shared-memory view of one ring entry.
struct SlotSmem {
  const uint8_t* kc;
  const uint8_t* vc;
  const __half* ks;
  const __half* kz;
  const __half* vs;
  const __half* vz;
};

// Per-lane constants of the column layout.
struct LaneCols {
  int g, c, lane, hq, u_lane;
  int e_live;  // GV >= 2: accumulator column (0/1) of an owned pair whose V group is u_lane, or -1
};

// Channel-wise K: Q' = Q * s_tau / factor scaled into fp16 for the token group tau whose
// s/z rows are s_tau/z_tau; the offset becomes sum_d Q_d z_tau,d (one constant per query
// and group, added before the softmax).
// The pair prologue has formed, per query and lane, W = Q / factor * 2^ea (fp16, in the
// order of this lane's B fragment; max |W| in [2^7, 2^8)), in sW. Per group this lane pairs
// its 32 scales in the same order (one byte permute per word), scales them by 2^es so that
// the largest of the group's 128 is in [2^6, 2^7), and multiplies: Q' = W * s 2^es in fp16,
// one rounding of the exact product, at most 2^15. Scores come out in units of
// 2^-(ea + es) (times the 2^-24 of the code images).
template <class C>
__device__ __forceinline__ void channelwise_q(uint32_t (&qB)[8][2], float (&cwA)[C::NQ], float (&cwB)[C::NQ],
                                              const __half* s_tau, const __half* z_tau, const float* sQ,
                                              const uint32_t* sW, float sl2, const LaneCols& lc) {
  constexpr int D = kHeadDim;
  constexpr unsigned FULLMASK = 0xffffffffu;
  const int c = lc.c;
  const int qb = qk_query<C>(lc.g, lc.hq);  // this lane's B column is column g
  const bool live = qb >= 0;
  static_assert(qk_wide<C>(), "channel-wise K uses the wide K mapping");
  const int* sEq = reinterpret_cast<const int*>(sQ + kMaxHq * D + kMaxHq);
  // the maximum of the group's 128 scales (>= 0): this lane's 32, then the row's 4 lanes
  const uint32_t* s32 = reinterpret_cast<const uint32_t*>(s_tau + 32 * c);  // two scales per word
  __half2 m2;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint4 v = reinterpret_cast<const uint4*>(s32)[k];
    const __half2 a2 = __hmax2(*reinterpret_cast<const __half2*>(&v.x), *reinterpret_cast<const __half2*>(&v.y));
    const __half2 b2 = __hmax2(*reinterpret_cast<const __half2*>(&v.z), *reinterpret_cast<const __half2*>(&v.w));
    m2 = k == 0 ? __hmax2(a2, b2) : __hmax2(m2, __hmax2(a2, b2));
  }
  float smax = fmaxf(__low2float(m2), __high2float(m2));
  smax = fmaxf(smax, __shfl_xor_sync(FULLMASK, smax, 1));
  smax = fmaxf(smax, __shfl_xor_sync(FULLMASK, smax, 2));
  const int es = smax > 0.f ? min(15, max(-14, 6 - ilog2f(smax))) : 15;
  const uint32_t sc_bits = (uint32_t)(es + 15) << 10;
  const uint32_t sc2w = sc_bits | (sc_bits << 16);
  const __half2 sc2 = *reinterpret_cast<const __half2*>(&sc2w);
  // the B fragment: per scale word pair (wa, wb) the two words of k-step ks (r = 0, 1); the
  // pair's channels are k0 and k0 + 8 (INT2) or k0 + 4 (INT4) of this lane's 32
  // (a column without a query reads the zero row kMaxHq - 1, which no query has then)
  const uint2* wrow = reinterpret_cast<const uint2*>(sW + ((live ? qb : kMaxHq - 1) * 4 + c) * kWRow);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const int wa = (C::BITS == 2) ? 8 * (ks >> 2) + (ks & 3) : 4 * (ks >> 1) + (ks & 1);
    const int wb = wa + (C::BITS == 2 ? 4 : 2);
    const uint32_t sa = s32[wa], sb = s32[wb];
    const uint2 w2 = wrow[ks];  // words 2 ks (r = 0) and 2 ks + 1 (r = 1)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const uint32_t sp = prmt(sa, sb, r ? 0x7632 : 0x5410);
      const __half2 s2 = __hmul2(*reinterpret_cast<const __half2*>(&sp), sc2);
      const uint32_t wv = r ? w2.y : w2.x;
      const __half2 q2 = __hmul2(*reinterpret_cast<const __half2*>(&wv), s2);
      qB[ks][r] = *reinterpret_cast<const uint32_t*>(&q2);
    }
  }
  // the offset: sum over the lane's 32 channels of Q z, then over the 4 lanes of the row
  float zsum = 0.f;
  {
    const float* qrow = sQ + (live ? qb : 0) * D + 32 * c;
    const uint2* zrow = reinterpret_cast<const uint2*>(z_tau + 32 * c);
    // the lanes' 16 (query, c) rows start their 8 quads at different offsets, so that one
    // load of a warp falls in different banks (in order, all 16 rows would share 4 banks)
    const int rot = (2 * c + (live ? qb : 0)) & 7;
#pragma unroll 2
    for (int k4 = 0; k4 < 8; ++k4) {
      const int kk = (k4 + rot) & 7;
      const float4 q4 = reinterpret_cast<const float4*>(qrow)[kk];
      const uint2 z4 = zrow[kk];
      const float2 z01 = half2_to_float2(z4.x), z23 = half2_to_float2(z4.y);
      zsum = fmaf(q4.x, z01.x, fmaf(q4.y, z01.y, fmaf(q4.z, z23.x, fmaf(q4.w, z23.y, zsum))));
    }
  }
  zsum = live ? zsum : 0.f;
  zsum += __shfl_xor_sync(FULLMASK, zsum, 1);
  zsum += __shfl_xor_sync(FULLMASK, zsum, 2);
  const float fb = sl2 * zsum;
  // accumulator column 2c + j is B column 2c + j, held by lane 4 (2c + j)
#pragma unroll
  for (int j = 0; j < C::NQ; ++j) {
    const int qj = qk_query<C>(2 * c + j, lc.hq);
    cwA[j] = qj >= 0 ? sl2 * exp2i(-(sEq[qj] + es)) * kImageUnit : 0.f;
    cwB[j] = __shfl_sync(FULLMASK, fb, 8 * c + 4 * j);
  }
}

// QK^T of one 32-token chunk starting at slot token rel0, with the K fold.
// x[mt][row][j]: token rel0 + 16 mt + 2 g + row, query slot j; token-wise K in
// units of pa[j], channel-wise K in log2 units.
template <class C>
__device__ __forceinline__ void qk_chunk(float (&x)[2][2][C::NQ], const WarpState<C>& st, const uint32_t (&qB)[8][2],
                                         const uint2* sqb,
                                         const float (&cwA)[C::NQ], const float (&cwB)[C::NQ],
                                         const SlotSmem& sm, int rel0, const LaneCols& lc) {
  constexpr int BITS = C::BITS, KL = C::KL, GK = C::GK, RB = C::RB, NQ = C::NQ;
  const int g = lc.g, c = lc.c;
  // Channel-wise K at INT4 (rows of 64 bytes, 128-bit loads): lanes with odd g read the odd
  // token row as their row g (two shared-memory wavefronts per load instead of four) and swap
  // their two accumulator rows back before the fold. (Measured: the ragged INT4 channel-wise K
  // batch 114.0 -> 109.8 us; with token-wise K, whose fold reads per-token scales, 1 % slower.)
  const bool swk = (BITS == 4 && KL == 1) && (g & 1);
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    const int tA = rel0 + 16 * mt + 2 * g;  // row g is token tA, row g+8 token tA+1
    const uint32_t* rA = reinterpret_cast<const uint32_t*>(sm.kc + (tA + (swk ? 1 : 0)) * RB);
    const uint32_t* rB = reinterpret_cast<const uint32_t*>(sm.kc + (tA + (swk ? 0 : 1)) * RB);
    uint32_t wA[4], wB[4], sA[4], sB[4];
    if (qk_wide<C>()) {
      if (BITS == 2) {  // words 2c, 2c+1 of each row
        const uint2 va = reinterpret_cast<const uint2*>(rA)[c], vb = reinterpret_cast<const uint2*>(rB)[c];
        wA[0] = va.x, wA[1] = va.y, wB[0] = vb.x, wB[1] = vb.y;
#pragma unroll
        for (int x = 0; x < 2; ++x) sA[x] = wA[x] >> 10, sB[x] = wB[x] >> 10;
      } else {  // words 4c .. 4c+3 of each row
        const uint4 va = reinterpret_cast<const uint4*>(rA)[c], vb = reinterpret_cast<const uint4*>(rB)[c];
        wA[0] = va.x, wA[1] = va.y, wA[2] = va.z, wA[3] = va.w;
        wB[0] = vb.x, wB[1] = vb.y, wB[2] = vb.z, wB[3] = vb.w;
#pragma unroll
        for (int x = 0; x < 4; ++x) sA[x] = wA[x] >> 8, sB[x] = wB[x] >> 8;
      }
    } else {
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
        if (BITS == 2) {
          // lanes with odd c take codes 4..7 and 12..15 of the word: shift them into 0..3
          const int sh = 8 * (c & 1);
          wA[blk] = rA[2 * blk + (c >> 1)] >> sh;
          wB[blk] = rB[2 * blk + (c >> 1)] >> sh;
        } else {
          wA[blk] = rA[4 * blk + c];
          wB[blk] = rB[4 * blk + c];
          sA[blk] = wA[blk] >> 8;
          sB[blk] = wB[blk] >> 8;
        }
      }
    }
    float xs[2][NQ];
#pragma unroll
    for (int row = 0; row < 2; ++row)
#pragma unroll
      for (int j = 0; j < NQ; ++j) xs[row][j] = 0.f;
    float acc[4];
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int blk = ks >> 1, h = ks & 1;
      uint32_t a0, a1, a2, a3;
      if (qk_wide<C>()) {
        if (BITS == 2) {
          const int x = ks >> 2, p0 = 2 * (ks & 3);
          a0 = int2_half2(wA[x], sA[x], p0);
          a1 = int2_half2(wB[x], sB[x], p0);
          a2 = int2_half2(wA[x], sA[x], p0 + 1);
          a3 = int2_half2(wB[x], sB[x], p0 + 1);
        } else {
          const int x = ks >> 1, p0 = 2 * (ks & 1);
          a0 = int4_half2(wA[x], sA[x], p0);
          a1 = int4_half2(wB[x], sB[x], p0);
          a2 = int4_half2(wA[x], sA[x], p0 + 1);
          a3 = int4_half2(wB[x], sB[x], p0 + 1);
        }
      } else if (BITS == 2) {
        const uint32_t mA = 0x00030003u << (4 * h), mB = 0x00030003u << (4 * h + 2);
        a0 = wA[blk] & mA;
        a1 = wB[blk] & mA;
        a2 = wA[blk] & mB;
        a3 = wB[blk] & mB;
      } else {
        a0 = int4_half2(wA[blk], sA[blk], 2 * h);
        a1 = int4_half2(wB[blk], sB[blk], 2 * h);
        a2 = int4_half2(wA[blk], sA[blk], 2 * h + 1);
        a3 = int4_half2(wB[blk], sB[blk], 2 * h + 1);
      }
      uint32_t q0, q1;  // B fragment of this k-step
      if constexpr (KL == 0) {
        const uint2 q = sqb[ks * 32 + lc.lane];
        q0 = q.x, q1 = q.y;
      } else {
        q0 = qB[ks][0], q1 = qB[ks][1];
      }
      if (KL == 0 ? (ks % C::KSG == 0) : (ks == 0)) {
        // a fresh accumulator per K channel group (token-wise K) or per 32-token chunk
        // (channel-wise K)
        mma_f16_c(acc, a0, a1, a2, a3, q0, q1, 0.f, 0.f, 0.f, 0.f);
      } else {
        mma_f16(acc, a0, a1, a2, a3, q0, q1);
      }
      if (swk && (KL == 0 ? (ks + 1) % C::KSG == 0 : ks == 7)) {
#pragma unroll
        for (int j = 0; j < NQ; ++j) {
          const float t = acc[j];
          acc[j] = acc[2 + j];
          acc[2 + j] = t;
        }
      }
      if (KL == 0 && (ks + 1) % C::KSG == 0) {
        // acc-fold of one channel group: s * (raw partial) + z * 2^e sum(Q over the group)
        const int grp = ks / C::KSG;
        float s0, s1, z0, z1;
        if (GK == 1) {
          const float2 s2 = half2_to_float2(*reinterpret_cast<const uint32_t*>(sm.ks + tA));
          const float2 z2 = half2_to_float2(*reinterpret_cast<const uint32_t*>(sm.kz + tA));
          s0 = s2.x, s1 = s2.y, z0 = z2.x, z1 = z2.y;
        } else {
          s0 = __half2float(sm.ks[tA * GK + grp]);
          s1 = __half2float(sm.ks[(tA + 1) * GK + grp]);
          z0 = __half2float(sm.kz[tA * GK + grp]);
          z1 = __half2float(sm.kz[(tA + 1) * GK + grp]);
        }
#pragma unroll
        for (int j = 0; j < NQ; ++j) {
          xs[0][j] = fmaf(s0, acc[j], fmaf(z0, st.bzq[j][grp], xs[0][j]));
          xs[1][j] = fmaf(s1, acc[2 + j], fmaf(z1, st.bzq[j][grp], xs[1][j]));
        }
      }
    }
#pragma unroll
    for (int j = 0; j < NQ; ++j) {
      if (KL == 0) {
        x[mt][0][j] = xs[0][j];
        x[mt][1][j] = xs[1][j];
      } else {
        x[mt][0][j] = fmaf(cwA[j], acc[j], cwB[j]);
        x[mt][1][j] = fmaf(cwA[j], acc[2 + j], cwB[j]);
      }
    }
  }
}

// PV of one 32-token chunk: accv[mt][v] (+)= V^T[16 channels x 16 tokens] * B.
// Row half `row` of m-tile mt is channel 16 g + pv_channel(mt, row). fresh: the
// accumulators start at zero instead of continuing.
template <class C>
__device__ __forceinline__ void pv_chunk(float (&accv)[8][C::NTV][4], const uint32_t (&pB)[C::NTV][2][2],
                                         const SlotSmem& sm, int rel0, const LaneCols& lc, bool fresh) {
  constexpr int BITS = C::BITS, RB = C::RB, NTV = C::NTV;
  const int g = lc.g, c = lc.c;
#pragma unroll
  for (int kk = 0; kk < 2; ++kk) {
    // k-slots 2c, 2c+1 are tokens tA, tA+1; k-slots 2c+8, 2c+9 are tokens tA+8, tA+9
    const int tA = rel0 + 16 * kk + 2 * c;
    const bool first = fresh && kk == 0;
    if (BITS == 2) {
      const uint32_t wa0 = reinterpret_cast<const uint32_t*>(sm.vc + tA * RB)[g];
      const uint32_t wa1 = reinterpret_cast<const uint32_t*>(sm.vc + (tA + 1) * RB)[g];
      const uint32_t wb0 = reinterpret_cast<const uint32_t*>(sm.vc + (tA + 8) * RB)[g];
      const uint32_t wb1 = reinterpret_cast<const uint32_t*>(sm.vc + (tA + 9) * RB)[g];
      const uint32_t xal = prmt(wa0, wa1, 0x5410), xah = prmt(wa0, wa1, 0x7632);
      const uint32_t xbl = prmt(wb0, wb1, 0x5410), xbh = prmt(wb0, wb1, 0x7632);
      const uint32_t sal = xal >> 10, sah = xah >> 10, sbl = xbl >> 10, sbh = xbh >> 10;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const uint32_t a0 = int2_half2(xal, sal, mt), a1 = int2_half2(xah, sah, mt);
        const uint32_t a2 = int2_half2(xbl, sbl, mt), a3 = int2_half2(xbh, sbh, mt);
#pragma unroll
        for (int v = 0; v < NTV; ++v) {
          if (first)
            mma_f16_c(accv[mt][v], a0, a1, a2, a3, pB[v][kk][0], pB[v][kk][1], 0.f, 0.f, 0.f, 0.f);
          else
            mma_f16(accv[mt][v], a0, a1, a2, a3, pB[v][kk][0], pB[v][kk][1]);
        }
      }
    } else {
      // Lanes with odd c read the odd token row of each pair first: rows are 64 bytes (half
      // the banks), so the four row groups of one load then fall in both bank halves (two
      // shared-memory wavefronts per load instead of four); their byte permutes take the two
      // rows in the other order. (INT2 rows, 32 bytes, conflict only two ways on 32-bit loads:
      // measured, the same change there cost more than it saved.)
      const int swp = c & 1;
      const uint32_t selL = swp ? 0x1054u : 0x5410u, selH = swp ? 0x3276u : 0x7632u;
      const uint2 wa0 = reinterpret_cast<const uint2*>(sm.vc + (tA + swp) * RB)[g];
      const uint2 wa1 = reinterpret_cast<const uint2*>(sm.vc + (tA + 1 - swp) * RB)[g];
      const uint2 wb0 = reinterpret_cast<const uint2*>(sm.vc + (tA + 8 + swp) * RB)[g];
      const uint2 wb1 = reinterpret_cast<const uint2*>(sm.vc + (tA + 9 - swp) * RB)[g];
#pragma unroll
      for (int uu = 0; uu < 2; ++uu) {
        const uint32_t ea0 = uu ? wa0.y : wa0.x, ea1 = uu ? wa1.y : wa1.x;
        const uint32_t eb0 = uu ? wb0.y : wb0.x, eb1 = uu ? wb1.y : wb1.x;
        const uint32_t xal = prmt(ea0, ea1, selL), xah = prmt(ea0, ea1, selH);
        const uint32_t xbl = prmt(eb0, eb1, selL), xbh = prmt(eb0, eb1, selH);
        const uint32_t sal = xal >> 8, sah = xah >> 8, sbl = xbl >> 8, sbh = xbh >> 8;
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
          const int mt = 4 * uu + pp;
          const uint32_t a0 = int4_half2(xal, sal, pp), a1 = int4_half2(xah, sah, pp);
          const uint32_t a2 = int4_half2(xbl, sbl, pp), a3 = int4_half2(xbh, sbh, pp);
#pragma unroll
          for (int v = 0; v < NTV; ++v) {
            if (first)
              mma_f16_c(accv[mt][v], a0, a1, a2, a3, pB[v][kk][0], pB[v][kk][1], 0.f, 0.f, 0.f, 0.f);
            else
              mma_f16(accv[mt][v], a0, a1, a2, a3, pB[v][kk][0], pB[v][kk][1]);
          }
        }
      }
    }
  }
}

// Live output column i of a lane: owned combo index, or -1 when the lane's V group
// matches neither combo of the pair.
template <class C>
__device__ __forceinline__ int live_own(int i, const LaneCols& lc) {
  if (C::DUP) return 0;
  if (C::GV == 1) return i;
  return lc.e_live < 0 ? -1 : 2 * i + lc.e_live;
}
// PV n-tile and accumulator column (0/1 within the lane's pair) of live column i.
template <class C>
__device__ __forceinline__ int live_tile(int i) {
  return (C::MODE == kModeWide) ? i : 0;
}
template <class C>
__device__ __forceinline__ int live_col(int i, const LaneCols& lc) {
  return C::DUP ? 0 : (C::GV == 1 ? i : max(lc.e_live, 0));
}

// Token-wise V: operand-fold of one item (the scale is already in the weights):
// running output += accumulator * inv_ps / factor, inv_ps = 2^-eP * 2^24.
template <class C>
__device__ __forceinline__ void fold_tokenwise_v(WarpState<C>& st, const float (&accv)[8][C::NTV][4], float inv_ps,
                                                 const LaneCols& lc) {
#pragma unroll
  for (int i = 0; i < C::NQ; ++i) {
    const int v = live_tile<C>(i), e = live_col<C>(i, lc);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const float f = inv_ps * (1.f / v_mult<C::BITS>(mt));
#pragma unroll
      for (int row = 0; row < 2; ++row) {
        const float a = (e == 0) ? accv[mt][v][2 * row] : accv[mt][v][2 * row + 1];
        st.o_run[mt][row][i] = fmaf(a, f, st.o_run[mt][row][i]);
      }
    }
  }
}

// Channel-wise V: acc-fold of one token group tau whose s/z rows are s_tau/z_tau:
// running output += s_tau,d * accumulator * 2^24 / (FED factor) + z_tau,d * W,
// W = sum of the group's weights (fed sum / FED) per owned combo; the weights were fed
// as P * FED.
template <class C, int FED = 8192>
__device__ __forceinline__ void fold_channelwise_v(WarpState<C>& st, const float (&accv)[8][C::NTV][4],
                                                   const float (&Wg)[C::NO], const __half* s_tau,
                                                   const __half* z_tau, const LaneCols& lc) {
  constexpr int BITS = C::BITS;
  const uint4* sp = reinterpret_cast<const uint4*>(s_tau + 16 * lc.g);
  const uint4* zp = reinterpret_cast<const uint4*>(z_tau + 16 * lc.g);
  const uint4 s_lo = sp[0], s_hi = sp[1], z_lo = zp[0], z_hi = zp[1];
  const uint32_t sw[8] = {s_lo.x, s_lo.y, s_lo.z, s_lo.w, s_hi.x, s_hi.y, s_hi.z, s_hi.w};
  const uint32_t zw[8] = {z_lo.x, z_lo.y, z_lo.z, z_lo.w, z_hi.x, z_hi.y, z_hi.z, z_hi.w};
#pragma unroll
  for (int i = 0; i < C::NQ; ++i) {
    const int v = live_tile<C>(i), e = live_col<C>(i, lc);
    const float W = Wg[C::DUP ? 0 : i] * (1.f / (float)FED);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int row = 0; row < 2; ++row) {
        const int k = pv_channel<BITS>(mt, row);
        const float2 s2 = half2_to_float2(sw[k >> 1]);
        const float2 z2 = half2_to_float2(zw[k >> 1]);
        const float s = (k & 1) ? s2.y : s2.x;
        const float z = (k & 1) ? z2.y : z2.x;
        const float a = (e == 0) ? accv[mt][v][2 * row] : accv[mt][v][2 * row + 1];
        st.o_run[mt][row][i] = fmaf(s * (kImageUnit / ((float)FED * v_mult<BITS>(mt))), a, fmaf(z, W, st.o_run[mt][row][i]));
      }
  }
}

// One warp unit: the NCH chunks of 32 tokens of one ring entry. nv: valid tokens
// of the entry (all UNIT valid when FULL). mid() runs between the QK^T and PV
// phases and returns false when the V half of the entry did not arrive.
template <class C, bool FULL, class Mid>
__device__ __forceinline__ void process_unit(WarpState<C>& st, const SlotSmem& sm, int nv, const float* sQ, float sl2,
                                             const uint2* sqb, const LaneCols& lc, Mid&& mid) {
  constexpr int KL = C::KL, VL = C::VL, GV = C::GV, NQ = C::NQ, NO = C::NO, NTV = C::NTV;
  constexpr int NCH = C::NCH, D = kHeadDim;
  constexpr unsigned FULLMASK = 0xffffffffu;
  const int g = lc.g, c = lc.c;

  // ------------------------------------------------ phase 1: scores of the whole unit
  float x[NCH][2][2][NQ];
  uint32_t qBt[8][2];  // channel-wise K: Q' of the current token group
  float cwA[NQ], cwB[NQ];
#pragma unroll
  for (int j = 0; j < NQ; ++j) cwA[j] = cwB[j] = 0.f;
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    const int rel0 = kChunk * ch;
    if (!FULL && rel0 >= nv) {
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int row = 0; row < 2; ++row)
#pragma unroll
          for (int j = 0; j < NQ; ++j) x[ch][mt][row][j] = -INFINITY;
      continue;
    }
    if constexpr (KL == 1) {
      if (ch == 0 || (C::G <= C::UNIT && (kChunk * ch) % C::G == 0)) {
        const int tau = rel0 / C::G;
        channelwise_q<C>(qBt, cwA, cwB, sm.ks + tau * D, sm.kz + tau * D, sQ,
                         reinterpret_cast<const uint32_t*>(sqb), sl2, lc);
      }
    }
    qk_chunk<C>(x[ch], st, qBt, sqb, cwA, cwB, sm, rel0, lc);
    if (!FULL) {
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int row = 0; row < 2; ++row)
#pragma unroll
          for (int j = 0; j < NQ; ++j)
            if (rel0 + 16 * mt + 2 * g + row >= nv) x[ch][mt][row][j] = -INFINITY;
    }
  }

  // ------------------------------------------------ running maximum, once per unit
  float nm[NQ];
  {
    float mx[NQ];
    bool grow = false;
#pragma unroll
    for (int j = 0; j < NQ; ++j) {
      float m = -INFINITY;
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch)
        m = fmaxf(m, fmaxf(fmaxf(x[ch][0][0][j], x[ch][0][1][j]), fmaxf(x[ch][1][0][j], x[ch][1][1][j])));
      m = fmaxf(m, __shfl_xor_sync(FULLMASK, m, 4));
      m = fmaxf(m, __shfl_xor_sync(FULLMASK, m, 8));
      m = fmaxf(m, __shfl_xor_sync(FULLMASK, m, 16));
      mx[j] = fmaxf(st.m_run[j], m);
      grow |= (mx[j] > st.m_run[j]);
    }
    if (__any_sync(FULLMASK, grow)) {
      float alpha[NQ];
#pragma unroll
      for (int j = 0; j < NQ; ++j) {
        alpha[j] = (mx[j] == st.m_run[j]) ? 1.f : fast_exp2(st.pa[j] * (st.m_run[j] - mx[j]));
        st.l[j] *= alpha[j];
      }
#pragma unroll
      for (int o = 0; o < NO; ++o) st.zacc[o] *= alpha[own_slot<C>(o)];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int row = 0; row < 2; ++row)
#pragma unroll
          for (int i = 0; i < NQ; ++i) st.o_run[mt][row][i] *= alpha[i];
    }
#pragma unroll
    for (int j = 0; j < NQ; ++j) {
      st.m_run[j] = mx[j];
      nm[j] = -st.pa[j] * mx[j];
    }
  }

  // The K half of the entry is no longer read: mid() refills it and waits for the V half.
  if (!mid()) return;

  // ------------------------------------------------ token-wise V: weight exponent of the unit
  // Fed weight P_t s_t,u 2^eP with max(s) 2^eP in [2^13, 2^14) over the unit's valid
  // tokens: the fed values stay in the fp16 normal range.
  float ps = 8192.f, inv_ps = 1.f / 8192.f;
  if (VL == 0) {
    constexpr int WORDS = C::UNIT * GV / 2;  // scale words (two halves) of the unit
    const uint32_t* sw = reinterpret_cast<const uint32_t*>(sm.vs);
    uint32_t smax = 0;
#pragma unroll
    for (int k = 0; k < (WORDS + 31) / 32; ++k) {
      const int w = lc.lane + 32 * k;
      if (WORDS % 32 != 0 && w >= WORDS) break;
      const uint32_t s01 = sw[w];
      const bool ok0 = FULL || ((2 * w) / GV < nv), ok1 = FULL || ((2 * w + 1) / GV < nv);
      const uint32_t m0 = ok0 ? (s01 & 0x7fffu) : 0u, m1 = ok1 ? ((s01 >> 16) & 0x7fffu) : 0u;
      smax = max(smax, max(m0, m1));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) smax = max(smax, __shfl_xor_sync(FULLMASK, smax, o));
    const float smaxf = __half2float(__ushort_as_half((unsigned short)smax));
    int e2 = 0;
    if (smaxf > 0.f) e2 = min(100, max(-100, 13 - ilog2f(smaxf)));
    ps = exp2i(e2);
    inv_ps = exp2i(24 - e2);  // 2^-eP times the 2^24 of the subnormal images
  }

  // ------------------------------------------------ phase 2: weights, PV, V fold
  float accv[8][NTV][4];
  float Wg[NO];  // channel-wise V: fed-weight sum of the current token group
#pragma unroll
  for (int o = 0; o < NO; ++o) Wg[o] = 0.f;
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    const int rel0 = kChunk * ch;
    if (!FULL && rel0 >= nv) break;
    // The accumulators run over the item (token-wise V: its weights share one exponent) or
    // over a token group (channel-wise V: one scale row), starting at zero.
    const bool fresh = (ch == 0) || (VL == 1 && C::G <= C::UNIT && (kChunk * ch) % C::G == 0);
    float P[2][2][NQ];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int row = 0; row < 2; ++row)
#pragma unroll
        for (int j = 0; j < NQ; ++j) P[mt][row][j] = fast_exp2(fmaf(st.pa[j], x[ch][mt][row][j], nm[j]));
    // fed weights: pw[o][mt] = (token 16mt+2g, token 16mt+2g+1) for owned combo o
    uint32_t pw[NO][2];
    float Fc[NO];
#pragma unroll
    for (int o = 0; o < NO; ++o) Fc[o] = 0.f;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const int tA = rel0 + 16 * mt + 2 * g;
      const bool ok0 = FULL || (tA < nv), ok1 = FULL || (tA + 1 < nv);
      if (VL == 0) {
#pragma unroll
        for (int j = 0; j < NQ; ++j) st.l[j] += P[mt][0][j] + P[mt][1][j];
      }
#pragma unroll
      for (int o = 0; o < NO; ++o) {
        const int j = own_slot<C>(o);
        float f0, f1;
        if (VL == 0) {
          // token-wise V scale and offset of tokens tA, tA+1 in this combo's V group
          uint32_t s01, z01;
          if (GV == 1) {
            s01 = *reinterpret_cast<const uint32_t*>(sm.vs + tA);
            z01 = *reinterpret_cast<const uint32_t*>(sm.vz + tA);
          } else {
            const int u = own_group<C>(c, o);
            s01 = (uint32_t)__half_as_ushort(sm.vs[tA * GV + u]) |
                  ((uint32_t)__half_as_ushort(sm.vs[(tA + 1) * GV + u]) << 16);
            z01 = (uint32_t)__half_as_ushort(sm.vz[tA * GV + u]) |
                  ((uint32_t)__half_as_ushort(sm.vz[(tA + 1) * GV + u]) << 16);
          }
          const float2 s2 = half2_to_float2(s01), z2 = half2_to_float2(z01);
          // padding tokens carry weight 0 and may hold any scale bits (even NaN)
          const float sv0 = ok0 ? s2.x : 0.f, sv1 = ok1 ? s2.y : 0.f;
          const float zv0 = ok0 ? z2.x : 0.f, zv1 = ok1 ? z2.y : 0.f;
          f0 = P[mt][0][j] * (sv0 * ps);
          f1 = P[mt][1][j] * (sv1 * ps);
          st.zacc[o] = fmaf(P[mt][0][j], zv0, fmaf(P[mt][1][j], zv1, st.zacc[o]));
        } else {
          f0 = P[mt][0][j] * 8192.f;
          f1 = P[mt][1][j] * 8192.f;
        }
        pw[o][mt] = f16x2_from(f0, f1);
        if (VL == 1) {
          const float2 fb = half2_to_float2(pw[o][mt]);
          Fc[o] += fb.x + fb.y;
        }
      }
    }
    if (VL == 1) {
#pragma unroll
      for (int o = 0; o < NO; ++o) {
        st.l[own_slot<C>(o)] += Fc[o] * (1.f / 8192.f);  // this lane's tokens
        Fc[o] += __shfl_xor_sync(FULLMASK, Fc[o], 4);
        Fc[o] += __shfl_xor_sync(FULLMASK, Fc[o], 8);
        Fc[o] += __shfl_xor_sync(FULLMASK, Fc[o], 16);
        Wg[o] += Fc[o];
      }
    }
    // PV B fragments: column n = g of n-tile v belongs to lane c_o = g/2 of each token
    // row group; k-slots 2c, 2c+1 (tokens 16kk + 2c + {0,1}) come from lane 4c + c_o and
    // k-slots 2c+8, 2c+9 from lane 4(c+4) + c_o, word kk of the owned combo.
    uint32_t pB[NTV][2][2];
    const int src0 = 4 * c + (g >> 1), src1 = 4 * (c + 4) + (g >> 1);
#pragma unroll
    for (int v = 0; v < NTV; ++v)
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        if (C::DUP) {
          pB[v][kk][0] = __shfl_sync(FULLMASK, pw[0][kk], src0);
          pB[v][kk][1] = __shfl_sync(FULLMASK, pw[0][kk], src1);
        } else {
          const uint32_t x00 = __shfl_sync(FULLMASK, pw[2 * v][kk], src0);
          const uint32_t x01 = __shfl_sync(FULLMASK, pw[2 * v + 1][kk], src0);
          const uint32_t x10 = __shfl_sync(FULLMASK, pw[2 * v][kk], src1);
          const uint32_t x11 = __shfl_sync(FULLMASK, pw[2 * v + 1][kk], src1);
          pB[v][kk][0] = (g & 1) ? x01 : x00;
          pB[v][kk][1] = (g & 1) ? x11 : x10;
        }
      }
    pv_chunk<C>(accv, pB, sm, rel0, lc, fresh);

    const bool last = (ch == NCH - 1) || (!FULL && rel0 + kChunk >= nv);
    if (VL == 0) {
      if (last) fold_tokenwise_v<C>(st, accv, inv_ps, lc);
    } else {
      const bool group_end = C::G <= C::UNIT && ((kChunk * (ch + 1)) % C::G == 0);
      if (last || group_end) {
        const int tau = rel0 / C::G;  // token-group row of the entry
        fold_channelwise_v<C>(st, accv, Wg, sm.vs + tau * D, sm.vz + tau * D, lc);
#pragma unroll
        for (int o = 0; o < NO; ++o) Wg[o] = 0.f;
      }
    }
    if (!FULL && rel0 + kChunk >= nv) break;
  }
}

// ------------------------------------------------------------------------
// Work split. The items (UNIT tokens; the last one of a pair may be partial) of all
// (sequence, KV head) pairs with tokens form one sequence in pair order. On a cost axis
// every such pair costs split_w (its boundary: prologue, waiting for the slowest warp,
// merges) followed by one unit per item: item x of the q-th pair with tokens sits at cost
// x + split_w (q + 1). CTA c of the persistent grid takes the items whose cost lies in
// [T(c), T(c + 1)), T(c) = ceil(c Ct / n_cta), Ct the total cost, and deals them to its
// warps in turn; a CTA that would cover many short pairs gets fewer items. Every CTA
// derives the counts from the device lengths.
// ------------------------------------------------------------------------
__device__ __forceinline__ long long split_threshold(long long c, long long ctot, long long n_cta) {
  return (c * ctot + n_cta - 1) / n_cta;
}

// The CTA's warps deposit (m, l, o) per query here for the merge of a pair.
struct MergeArea {
  float* m;  // [kMergeWarps][kMaxHq] running maximum (log2 units)
  float* l;  // [kMergeWarps][kMaxHq] denominator
  float* o;  // [kMergeWarps][hq][D] unnormalised output
};

// Result of the CTA's scan over the sequence lengths: the items at the two ends of its
// range (end 0 its first item, end 1 one past its last), and where its first item is.
struct SplitScan {
  long long cost[32], items[32], pairs[32];  // per-warp sums over a chunk of sequences
  long long ctot;                            // total cost
  int w;                                     // boundary cost in use (0 for small problems)
  int kw[2];                                 // warp chunk holding end e's threshold
  long long base_cost[2], base_items[2], base_pairs[2];  // sums of the chunks before it
  long long x[2];                            // item index of end e
  int b0, kv0, t0;                           // sequence, pair in it and item in the pair of end 0
  long long q0;                              // pairs with tokens before the start pair
  float cm[kMaxHq], cl[kMaxHq];              // cluster mode: the CTA partial's (m, l) per query
};

// ------------------------------------------------------------------------
// The kernel: see the file comment. C = Cfg<BITS, KL, VL, MODE, LOG2G>; PAGED: the cache
// is a page pool behind a page table (only the addresses of the bulk copies differ).
// ------------------------------------------------------------------------
template <class C, bool PAGED, bool CLUSTER>
__global__ void __launch_bounds__(C::THREADS, 1) split_decode_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int BITS = C::BITS, KL = C::KL, VL = C::VL, GV = C::GV, GK = C::GK, NQ = C::NQ, NO = C::NO;
  constexpr int RB = C::RB, D = kHeadDim, UNIT = C::UNIT, W = C::WARPS;
  constexpr unsigned FULLMASK = 0xffffffffu;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ SplitScan ss;
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int cta = blockIdx.x;
  const int hq = p.hq;
  const int n_pairs = p.B * p.Hkv;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);      // per warp and entry: K half, V half
  float* sQ = reinterpret_cast<float*>(smem + kBarBytes);  // [kMaxHq][D]
  float* sAq = sQ + kMaxHq * D;                            // [kMaxHq] token-wise K score factor
  int* sEq = reinterpret_cast<int*>(sAq + kMaxHq);         // [kMaxHq] query exponent
  float* sBz = sAq + 2 * kMaxHq;                           // [kMaxHq][4] 2^e * sum of Q per channel group
  uint2* sqb = reinterpret_cast<uint2*>(smem + kQbOffset);  // [8 k-steps][32 lanes] token-wise K
  MergeArea ma;
  ma.m = reinterpret_cast<float*>(smem + kPrologueBytes);
  ma.l = ma.m + kMergeWarps * kMaxHq;
  ma.o = ma.l + kMergeWarps * kMaxHq;
  uint8_t* ring = smem + p.ring_off;

  // Valid tokens of sequence b (device value: clamped, never trusted) and items of one of
  // its pairs.
  auto seq_len = [&](int b) { return min(max(__ldg(p.seq_lens + b), 0), p.T_cap); };
  auto items_of = [&](int L) { return (L + UNIT - 1) / UNIT; };
  // Values stored rotated: n output rows staged in fp32 in shared memory, rotated back by H
  // and written as the bf16 output rows out_row0 .. out_row0 + n - 1 (one warp per row).
  auto rotate_out_rows = [&](const float* rows, int n, size_t out_row0) {
    for (int i = warp; i < n; i += W) {
      float v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = rows[i * D + 4 * lane + e];
      hadamard128(v, lane);
      store_row4(p.out + (out_row0 + i) * D, lane, v);
    }
  };

  // ---------------------------------------------------- the CTA's share of the items
  // Cluster mode (small problems): clusters s·i .. s·i + s - 1 take pair i (s = cluster_split),
  // the CTA of rank r in the j-th of them the (j·n + r)-th of equal contiguous slices of the
  // pair's items (n CTAs per cluster); no scan.
  bool cluster_pair = false;  // cluster mode: the pair has tokens (its CTAs merge in the cluster)
  if constexpr (CLUSTER) {
    const int ncta = (int)cluster_nctarank(), crank = (int)cluster_ctarank();
    const int cid = (int)cluster_id_x();
    const int up = cid / p.cluster_split;
    const int cluster_sub = cid - up * p.cluster_split;  // which of the pair's clusters
    const int b = up / p.Hkv, kv = up % p.Hkv;
    const int n = up < n_pairs ? items_of(seq_len(b)) : 0;
    cluster_pair = n > 0;
    if (threadIdx.x == 0) {
      const long long parts = (long long)ncta * p.cluster_split, rr = (long long)cluster_sub * ncta + crank;
      const long long t0 = (long long)n * rr / parts, t1 = (long long)n * (rr + 1) / parts;
      ss.x[0] = t0;
      ss.x[1] = t1;
      ss.b0 = b;
      ss.kv0 = kv;
      ss.t0 = (int)t0;
      ss.q0 = 0;
      ss.w = 0;
      ss.ctot = 1;
    }
    __syncthreads();
  } else {
    const int chunk = (p.B + W - 1) / W;  // warp w sums sequences [w chunk, (w+1) chunk)
    const int bb0 = min(p.B, warp * chunk), bb1 = min(p.B, bb0 + chunk);
    long long si = 0, sp = 0;
    for (int b = bb0 + lane; b < bb1; b += 32) {
      const long long n = items_of(seq_len(b));
      si += (long long)p.Hkv * n;
      if (n > 0) sp += p.Hkv;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      si += __shfl_xor_sync(FULLMASK, si, o);
      sp += __shfl_xor_sync(FULLMASK, sp, o);
    }
    if (lane == 0) {
      ss.items[warp] = si;
      ss.pairs[warp] = sp;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      long long tot = 0, np = 0;
      for (int w = 0; w < W; ++w) tot += ss.items[w], np += ss.pairs[w];
      // With about one item per warp the split must keep the rounds of items even instead:
      // no boundary cost below 2 items per warp (measured: batch 8 at 16K and 32K contexts,
      // 3.4 and 6.7 items per warp, 35.8 -> 32.2 us and 51.1 -> 48.2 us with the cost)
      const int sw = (tot >= 2LL * W * p.n_cta) ? p.split_w : 0;
      for (int w = 0; w < W; ++w) ss.cost[w] = ss.items[w] + (long long)sw * ss.pairs[w];
      const long long ctot = tot + (long long)sw * np;
      ss.w = sw;
      ss.ctot = ctot;
      for (int e = 0; e < 2; ++e) {
        const long long T = split_threshold(cta + e, ctot, p.n_cta);
        ss.kw[e] = W;  // past the end: no item at or after T
        ss.x[e] = tot;
        long long ac = 0, ai = 0, ap = 0;
        for (int w = 0; w < W; ++w) {
          if (T < ac + ss.cost[w]) {
            ss.kw[e] = w;
            ss.base_cost[e] = ac;
            ss.base_items[e] = ai;
            ss.base_pairs[e] = ap;
            break;
          }
          ac += ss.cost[w], ai += ss.items[w], ap += ss.pairs[w];
        }
      }
      ss.b0 = ss.kv0 = ss.t0 = 0;
      ss.q0 = 0;
    }
    __syncthreads();
    for (int e = 0; e < 2; ++e) {
      if (warp != ss.kw[e]) continue;  // the warp whose chunk of sequences holds end e
      const long long T = split_threshold(cta + e, ss.ctot, p.n_cta);
      long long rc = ss.base_cost[e], ri = ss.base_items[e], rp = ss.base_pairs[e];
      for (int base = bb0; base < bb1; base += 32) {
        const int b = base + lane;
        const long long n = (b < bb1) ? (long long)items_of(seq_len(b)) : 0;
        const long long c_b = n > 0 ? (long long)p.Hkv * (n + ss.w) : 0;
        const long long i_b = (long long)p.Hkv * n, p_b = n > 0 ? p.Hkv : 0;
        long long ic = c_b, ii = i_b, ip = p_b;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const long long yc = __shfl_up_sync(FULLMASK, ic, o);
          const long long yi = __shfl_up_sync(FULLMASK, ii, o);
          const long long yp = __shfl_up_sync(FULLMASK, ip, o);
          if (lane >= o) ic += yc, ii += yi, ip += yp;
        }
        const long long ec = rc + ic - c_b;  // cost before sequence b
        const unsigned hit = __ballot_sync(FULLMASK, c_b > 0 && T >= ec && T < ec + c_b);
        if (hit) {
          if (lane == __ffs(hit) - 1) {
            const long long off = T - ec;
            const long long kv = off / (n + ss.w), o2 = off - kv * (n + ss.w);
            const long long t = o2 > ss.w ? o2 - ss.w : 0;
            ss.x[e] = (ri + ii - i_b) + kv * n + t;
            if (e == 0) {
              ss.b0 = b;
              ss.kv0 = (int)kv;
              ss.t0 = (int)t;
              ss.q0 = (rp + ip - p_b) + kv;
            }
          }
          break;
        }
        rc += __shfl_sync(FULLMASK, ic, 31);
        ri += __shfl_sync(FULLMASK, ii, 31);
        rp += __shfl_sync(FULLMASK, ip, 31);
      }
    }
    __syncthreads();
  }
  const long long X0 = ss.x[0], X1 = ss.x[1];
  const int NL = (int)(X1 - X0);  // items of this CTA
  // The first pair's query rows, loaded now so that their latency passes while the ring's
  // first copies are issued (staged into shared memory by the first segment's prologue).
  constexpr int kQPre = (kMaxHq * kHeadDim + C::THREADS - 1) / C::THREADS;
  float qpre[kQPre];
  if (NL > 0 || cluster_pair) {
    const size_t q0 = ((size_t)ss.b0 * p.Hq + (size_t)ss.kv0 * hq) * D;
#pragma unroll
    for (int j = 0; j < kQPre; ++j) {
      const int idx = threadIdx.x + j * C::THREADS;
      qpre[j] = idx < hq * D ? __bfloat162float(p.q[q0 + idx]) : 0.f;
    }
  }

  // Each ring entry has a K half (codes, scales, offsets) and a V half, each with its own
  // mbarrier, so that the next item's K half loads while this item's PV phase runs and
  // its V half while the next QK^T phase runs.
  const int R = p.ring_per_warp;
  const uint32_t bar_w = smem_addr(bars) + 16u * (uint32_t)(warp * R);
  uint8_t* ring_w = ring + (size_t)warp * R * C::E.bytes;
  auto bar_k = [&](int r) { return bar_w + 16u * r; };
  auto bar_v = [&](int r) { return bar_w + 16u * r + 8u; };

  // Bulk copies of the K or V half of item t of pair u into entry r (lane 0 only). A
  // paged cache takes the item's page and cached KV head from the issue cursor.
  int iss_page = 0, iss_kvh = 0;  // paged cache: the issue cursor's page and cached KV head
  auto copy_half = [&](bool v_half, int u_pair, int t, int r) {
    const int u = u_pair >> p.kv_shift;  // cached KV head (sequence-major)
    const size_t t0 = (size_t)t * UNIT;
    size_t row0, blk0;  // first code row, first channel-wise scale block
    if constexpr (PAGED) {
      const size_t pu = (size_t)iss_page * (p.Hkv >> p.kv_shift) + iss_kvh;
      row0 = (pu << p.log2_page) + (t0 & ((size_t(1) << p.log2_page) - 1));
      blk0 = row0 / C::G;
    } else {
      row0 = (size_t)u * p.T_cap + t0;
      blk0 = (size_t)u * ((size_t)p.T_cap / C::G) + t0 / C::G;
    }
    const uint32_t dst = smem_addr(ring_w + (size_t)r * C::E.bytes);
    const uint64_t pol = l2_evict_first_policy();
    fence_proxy_async_smem();  // earlier reads of the half come before its refill
    if (!v_half) {
      const uint32_t fb = bar_k(r);
      const size_t ks0 = (KL == 0) ? row0 * C::GK : blk0 * kHeadDim;
      mbar_arrive_expect_tx(fb, C::E.tx_k);
      bulk_g2s(dst, p.k_codes + row0 * RB, UNIT * RB, fb, pol);
      bulk_g2s(dst + C::E.off_ks, p.k_scale + ks0, C::E.sz_k, fb, pol);
      bulk_g2s(dst + C::E.off_kz, p.k_off + ks0, C::E.sz_k, fb, pol);
    } else {
      const uint32_t fb = bar_v(r);
      const size_t vs0 = (VL == 0) ? row0 * C::GV : blk0 * kHeadDim;
      mbar_arrive_expect_tx(fb, C::E.tx_v);
      bulk_g2s(dst + C::E.off_vc, p.v_codes + row0 * RB, UNIT * RB, fb, pol);
      bulk_g2s(dst + C::E.off_vs, p.v_scale + vs0, C::E.sz_v, fb, pol);
      bulk_g2s(dst + C::E.off_vz, p.v_off + vs0, C::E.sz_v, fb, pol);
    }
  };

  // This warp's items are local indices warp, warp + W, ... of the CTA range; they go
  // through entries 0, 1, .., R-1, 0, ... of its ring in order. Cursors walk them without
  // divisions (pairs without tokens hold no items and are stepped over).
  struct Cursor {
    int i, u, t, L, n;  // local item index, pair, item within the pair, pair's tokens and items
    int r;              // ring entry of the next copy or read
    int b, kvh;         // paged cache: the pair's sequence and cached KV head
  };
  auto set_pair = [&](Cursor& k) {
    const int b = k.u / p.Hkv;
    k.L = seq_len(b);
    k.n = items_of(k.L);
    if constexpr (PAGED) {
      k.b = b;
      k.kvh = (k.u - b * p.Hkv) >> p.kv_shift;
    }
  };
  auto advance = [&](Cursor& k, int step) {  // step items forward (only while inside the range)
    k.i += step;
    k.t += step;
    if (k.i < NL) {
      while (k.t >= k.n) {
        k.t -= k.n;
        ++k.u;
        set_pair(k);
      }
    }
  };
  Cursor start;  // the CTA's first item
  start.i = 0;
  start.r = 0;
  if (NL > 0 || cluster_pair) {
    const int L0 = seq_len(ss.b0), n0 = items_of(L0);
    const int kv0 = ss.kv0;
    start.u = ss.b0 * p.Hkv + kv0;
    start.t = ss.t0;
    start.L = L0;
    start.n = n0;
    start.b = ss.b0;
    start.kvh = kv0 >> p.kv_shift;
  } else {
    start.u = n_pairs;
    start.t = 0;
    start.L = start.n = 0;
    start.b = start.kvh = 0;
  }
  Cursor iss = start;
  advance(iss, warp);
  // The issue cursor points at this warp's next item: issue_k() sends its K half,
  // issue_v() its V half and moves on (the K half always goes first).
  // A paged cache: lane 0 loads the page-table entry of the cursor's item when the cursor
  // moves there, and checks it (an entry outside the pool is recorded and read as page 0)
  // when the item's K half is issued.
  bool k_pending = false;
  int n_issued = 0;
  auto lookup_page = [&]() {
    if constexpr (PAGED) {
      if (lane == 0 && iss.i < NL) {
        iss_page = __ldg(p.page_table + (size_t)iss.b * p.max_pages + (((unsigned)iss.t * UNIT) >> p.log2_page));
        iss_kvh = iss.kvh;
      }
    }
  };
  lookup_page();
  auto issue_k = [&]() {
    if (iss.i < NL) {
      if (lane == 0) {
        if constexpr (PAGED) {
          if (iss_page < 0 || iss_page >= p.num_pages) {
            atomicExch(p.status, kStatusBadPage);
            iss_page = 0;
          }
        }
        copy_half(false, iss.u, iss.t, iss.r);
      }
      k_pending = true;
    }
  };
  auto issue_v = [&]() {
    if (!k_pending) return;
    if (lane == 0) copy_half(true, iss.u, iss.t, iss.r);
    k_pending = false;
    ++n_issued;
    if (++iss.r == R) iss.r = 0;
    advance(iss, W);
    lookup_page();
  };
  if (lane == 0) {
    for (int r = 0; r < R; ++r) {
      mbar_init(bar_k(r), 1);
      mbar_init(bar_v(r), 1);
    }
    mbar_init_fence();
  }
  __syncwarp();
  for (int r = 0; r < R; ++r) {
    issue_k();
    issue_v();
  }

  bool failed = false;
  Cursor con = start;
  advance(con, warp);
  int ph_con = 0, n_k_read = 0, n_v_read = 0;

  // ---------------------------------------------------- segments: the CTA's items of one pair
  long long x = X0;
  int u = start.u;
  long long pair_first = X0 - start.t;  // the pair's first item in the item sequence
  int pair_n = start.n;
  long long q = ss.q0;  // pairs with tokens before pair u
  // (cluster mode: one segment for every CTA of a pair with tokens, also without items, so
  // that all of them reach the cluster barriers of the merge)
  bool cluster_once = cluster_pair;
  while (x < X1 || cluster_once) {
    cluster_once = false;
    const long long xe = min(X1, pair_first + pair_n);
    const int b = u / p.Hkv, kvh = u % p.Hkv;

    // Stage Q (fp32) and the per-query constants of pair u.
    __syncthreads();  // the previous segment's merge is done with sQ and the merge area
    if (x == X0) {  // the first segment: its rows were loaded before the ring started
#pragma unroll
      for (int j = 0; j < kQPre; ++j) {
        const int idx = threadIdx.x + j * C::THREADS;
        if (idx < hq * D) sQ[idx] = qpre[j];
      }
    } else {
      for (int idx = threadIdx.x; idx < hq * D; idx += C::THREADS)
        sQ[idx] = __bfloat162float(p.q[((size_t)b * p.Hq + kvh * hq) * D + idx]);
    }
    __syncthreads();
    if (p.rotation & 1) {  // keys stored rotated: the scores take H q
      for (int i = warp; i < hq; i += W) {
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = sQ[i * D + 4 * lane + e];
        hadamard128(v, lane);
#pragma unroll
        for (int e = 0; e < 4; ++e) sQ[i * D + 4 * lane + e] = v[e];
      }
      __syncthreads();
    }
    if (warp < hq) {
      // query exponent e: max |Q / factor| * 2^e in [2^13, 2^14), so Q * 2^e / factor is an
      // exact fp16 for a bf16 query (8 significant bits; a rotated query is rounded there);
      // channel-group sums of Q for the K offset
      const int i = warp;
      float amax = 0.f;
      float gs = 0.f;
#pragma unroll
      for (int uu = 0; uu < 4; ++uu) {
        const int ch = 4 * lane + uu;
        const float v = sQ[i * D + ch];
        amax = fmaxf(amax, fabsf(v) * k_rmult<C>(ch));
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
      // (channel-wise K: max |Q / factor| * 2^e in [2^7, 2^8), the W of channelwise_q)
      if (amax > 0.f) e = min(100, max(-100, (KL == 1 ? 7 : 13) - ilog2f(amax)));
      // token-wise K scores are kept in units of sAq; the raw products carry the 2^-24 of the
      // subnormal code images, so the unit and the offset sums take the 2^24
      if (lane == 0) {
        sEq[i] = e;
        sAq[i] = p.sl2 * exp2i(24 - e);
      }
      if (KL == 0 && (lane % lanes_per_group) == 0) sBz[i * 4 + lane / lanes_per_group] = exp2i(e - 24) * gs;
    }
    __syncthreads();

    LaneCols lc;
    lc.g = g;
    lc.c = c;
    lc.lane = lane;
    lc.hq = hq;
    lc.u_lane = (GV == 1) ? 0 : (16 * g) / C::G;  // V channel group of this lane's 16 channels
    if (GV >= 2) {
      const int el = ((lc.u_lane - 2 * c) % GV + GV) % GV;
      lc.e_live = el <= 1 ? el : -1;
    } else {
      lc.e_live = 0;
    }

    WarpState<C> st;
    if (KL == 0) {
      // token-wise K: B fragments Q' = Q 2^e / factor (fp16; exact for a bf16 query) of
      // column g, the same for every warp, formed once: warp ks < 8 the k-step ks
      if (warp < 8) {
        const int ks = warp;
        const int qb = qk_query<C>(g, hq);
        const bool live = qb >= 0;
        const float sc = live ? exp2i(sEq[qb]) : 0.f;
        uint32_t qbw[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          float xx[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int ch = qk_channel<C>(ks, 2 * c + 8 * r + e);
            xx[e] = live ? sQ[qb * D + ch] * sc * k_rmult<C>(ch) : 0.f;
          }
          qbw[r] = f16x2_from(xx[0], xx[1]);
        }
        sqb[ks * 32 + lane] = make_uint2(qbw[0], qbw[1]);
      }
#pragma unroll
      for (int j = 0; j < NQ; ++j) {
        const int qs = qk_query<C>(2 * c + j, hq);
        st.pa[j] = qs >= 0 ? sAq[qs] : 1.f;
#pragma unroll
        for (int uu = 0; uu < GK; ++uu) st.bzq[j][uu] = qs >= 0 ? sBz[qs * 4 + uu] : 0.f;
      }
    } else {
      // channel-wise K: W = Q / factor * 2^e (fp16) per query and lane, in the order of the
      // lane's B fragment (word 2 ks + r: k-slots 2c + 8r, 2c + 8r + 1 of k-step ks)
      // (rows of queries q >= hq are zero: a column without a query reads one of them)
      uint32_t* sW = reinterpret_cast<uint32_t*>(sqb);  // [kMaxHq][4][kWRow]
      for (int t = threadIdx.x; t < kMaxHq * 64; t += C::THREADS) {
        const int qi = t >> 6, cc = (t >> 4) & 3, wi = t & 15, ks = wi >> 1, r = wi & 1;
        uint32_t w = 0u;
        if (qi < hq) {
          const float sc = exp2i(sEq[qi]);
          const int ch0 = qk_channel<C>(ks, 2 * cc + 8 * r), ch1 = qk_channel<C>(ks, 2 * cc + 8 * r + 1);
          w = f16x2_from(sQ[qi * D + ch0] * sc * k_rmult<C>(ch0), sQ[qi * D + ch1] * sc * k_rmult<C>(ch1));
        }
        sW[(t >> 4) * kWRow + (t & 15)] = w;
      }
#pragma unroll
      for (int j = 0; j < NQ; ++j) st.pa[j] = 1.f;
    }
#pragma unroll
    for (int j = 0; j < NQ; ++j) {
      st.m_run[j] = -INFINITY;
      st.l[j] = 0.f;
    }
#pragma unroll
    for (int o = 0; o < NO; ++o) st.zacc[o] = 0.f;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int row = 0; row < 2; ++row)
#pragma unroll
        for (int i = 0; i < NQ; ++i) st.o_run[mt][row][i] = 0.f;

    __syncthreads();  // the shared query fragments are in place

    // ---------------------------------------------------- this warp's items of the segment
    for (; !failed && con.i < NL && con.u == u; advance(con, W)) {
      const int nv = min(UNIT, con.L - con.t * UNIT);  // valid tokens of the item (>= 1)
      const int r = con.r;
      if (!mbar_wait(bar_k(r), ph_con, p.status, kStatusConsumerTimeout)) {
        failed = true;
        break;
      }
      ++n_k_read;
      const uint8_t* en = ring_w + (size_t)r * C::E.bytes;
      SlotSmem sm;
      sm.kc = en;
      sm.vc = en + C::E.off_vc;
      sm.ks = reinterpret_cast<const __half*>(en + C::E.off_ks);
      sm.kz = reinterpret_cast<const __half*>(en + C::E.off_kz);
      sm.vs = reinterpret_cast<const __half*>(en + C::E.off_vs);
      sm.vz = reinterpret_cast<const __half*>(en + C::E.off_vz);
      auto mid = [&]() {
        __syncwarp();
        issue_k();  // the K half is read: refill it with the next item's K
        if (!mbar_wait(bar_v(r), ph_con, p.status, kStatusConsumerTimeout)) {
          failed = true;
          return false;
        }
        ++n_v_read;
        return true;
      };
      if (nv == UNIT)
        process_unit<C, true>(st, sm, nv, sQ, p.sl2, sqb, lc, mid);
      else
        process_unit<C, false>(st, sm, nv, sQ, p.sl2, sqb, lc, mid);
      if (failed) break;
      if (++con.r == R) {
        con.r = 0;
        ph_con ^= 1;
      }
      __syncwarp();
      issue_v();  // the V half is read: refill it with the next item's V
    }

    // ---------------------------------------------------- warps beyond kMergeWarps fold in
    // Warp w + kMergeWarps hands its register state, lane by lane (same layout), to warp w,
    // which merges it into its own: running maxima, denominators, offsets and outputs.
    if (C::WARPS > kMergeWarps) {
      constexpr int SF = 16 * NQ + NO + 2 * NQ;
      static_assert(SF <= kStateFloats, "handed-over state fits the merge area");
      float* xs = ma.m;  // [kMergeWarps][SF][32]
      if (warp >= kMergeWarps) {
        float* d = xs + (size_t)(warp - kMergeWarps) * SF * 32 + lane;
        int k = 0;
#pragma unroll
        for (int j = 0; j < NQ; ++j) {
          d[32 * k++] = st.m_run[j];
          d[32 * k++] = st.l[j];
        }
#pragma unroll
        for (int o = 0; o < NO; ++o) d[32 * k++] = st.zacc[o];
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int row = 0; row < 2; ++row)
#pragma unroll
            for (int i = 0; i < NQ; ++i) d[32 * k++] = st.o_run[mt][row][i];
      }
      __syncthreads();
      if (warp < kMergeWarps && warp + kMergeWarps < C::WARPS) {
        const float* d = xs + (size_t)warp * SF * 32 + lane;
        float aa[NQ], ab[NQ];
        int k = 0;
#pragma unroll
        for (int j = 0; j < NQ; ++j) {
          const float mb = d[32 * k++], lb = d[32 * k++];
          const float m = fmaxf(st.m_run[j], mb);
          aa[j] = (st.m_run[j] == m) ? 1.f : fast_exp2(st.pa[j] * (st.m_run[j] - m));
          ab[j] = (mb == m) ? 1.f : fast_exp2(st.pa[j] * (mb - m));
          st.m_run[j] = m;
          st.l[j] = aa[j] * st.l[j] + ab[j] * lb;
        }
#pragma unroll
        for (int o = 0; o < NO; ++o) {
          const int j = own_slot<C>(o);
          st.zacc[o] = aa[j] * st.zacc[o] + ab[j] * d[32 * k++];
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int row = 0; row < 2; ++row)
#pragma unroll
            for (int i = 0; i < NQ; ++i) st.o_run[mt][row][i] = aa[i] * st.o_run[mt][row][i] + ab[i] * d[32 * k++];
      }
      __syncthreads();
    }

    // ---------------------------------------------------- warp results into the merge area
    if (warp < kMergeWarps) {
#pragma unroll
      for (int j = 0; j < NQ; ++j) {
        float l = st.l[j];
        l += __shfl_xor_sync(FULLMASK, l, 4);
        l += __shfl_xor_sync(FULLMASK, l, 8);
        l += __shfl_xor_sync(FULLMASK, l, 16);
        const int q = qk_query<C>(2 * c + j, hq);
        if (g == 0 && q >= 0) {
          ma.m[warp * kMaxHq + q] = (st.m_run[j] == -INFINITY) ? -INFINITY : st.pa[j] * st.m_run[j];
          ma.l[warp * kMaxHq + q] = l;
        }
      }
      float zs[NO];
#pragma unroll
      for (int o = 0; o < NO; ++o) {
        float z = st.zacc[o];
        z += __shfl_xor_sync(FULLMASK, z, 4);
        z += __shfl_xor_sync(FULLMASK, z, 8);
        z += __shfl_xor_sync(FULLMASK, z, 16);
        zs[o] = z;
      }
      // live column i holds owned combo o = (query, V group); this lane's 16 channels
      // 16g..16g+15 all lie in V group u_lane
#pragma unroll
      for (int i = 0; i < NQ; ++i) {
        const int o = live_own<C>(i, lc);
        if (o < 0) continue;
        const int combo = own_combo<C>(c, o);
        if (combo >= hq * GV || combo % GV != lc.u_lane) continue;
        const int q = combo / GV;
        float zt = 0.f;
        if (VL == 0) {
#pragma unroll
          for (int oo = 0; oo < NO; ++oo)
            if (oo == o) zt = zs[oo];
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int row = 0; row < 2; ++row)
            ma.o[(warp * hq + q) * kODep + 16 * g + pv_channel<BITS>(mt, row)] = st.o_run[mt][row][i] + zt;
      }
    }
    __syncthreads();

    // ---------------------------------------------------- merge the warps
    if constexpr (CLUSTER) {
      // Cluster mode: the CTA's partial stays in its shared memory (O over ma.o's first
      // block, (m, l) in ss.cm / ss.cl); after a cluster barrier the CTA of rank r merges
      // query rows r, r + n, ... from every CTA of the cluster (distributed shared memory)
      // with the window's partial, and a second barrier keeps each CTA's partial in place
      // until all have been read.
      for (int idx = threadIdx.x; idx < hq * D; idx += C::THREADS) {
        const int i = idx / D, ch = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kMergeWarps; ++w) M = fmaxf(M, ma.m[w * kMaxHq + i]);
        float acc = 0.f, lt = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kMergeWarps; ++w) {
            const float mw = ma.m[w * kMaxHq + i];
            const float sc = (mw == -INFINITY) ? 0.f : fast_exp2(mw - M);
            acc = fmaf(sc, ma.o[(w * hq + i) * kODep + ch], acc);
            lt = fmaf(sc, ma.l[w * kMaxHq + i], lt);
          }
        }
        ma.o[i * kODep + ch] = acc;  // read above by this thread only
        if (ch == 0) {
          ss.cm[i] = M;
          ss.cl[i] = lt;
        }
      }
      if (p.has_win) grid_dependency_wait();
      cluster_sync();
      {
        const int ncta = (int)cluster_nctarank(), crank = (int)cluster_ctarank();
        const uint32_t o_base = smem_addr(ma.o), m_base = smem_addr(ss.cm), l_base = smem_addr(ss.cl);
        for (int i = crank + ncta * warp; i < hq; i += ncta * W) {  // one warp per query row
          // lane k < ncta reads CTA k's (m, l) of the row; the maximum, the scales and the
          // denominator are warp reductions; every lane then reads its 4 channels of all the
          // CTAs' rows, four loads in flight at a time
          float mk = -INFINITY, lk = 0.f;
          if (lane < ncta) {
            mk = ld_cluster_f32(cluster_map(m_base + 4u * i, lane));
            lk = ld_cluster_f32(cluster_map(l_base + 4u * i, lane));
          }
          float M = mk;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(FULLMASK, M, o));
          float2 wml = make_float2(-INFINITY, 0.f);
          const size_t wr = (size_t)u * hq + i;
          if (p.has_win && p.cluster_split == 1) {  // (with several clusters the last adds it)
            wml = __ldcg(&p.win_ml[wr]);
            M = fmaxf(M, wml.x);
          }
          const float sck = (M == -INFINITY || mk == -INFINITY) ? 0.f : fast_exp2(mk - M);
          float lt = sck * lk;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) lt += __shfl_xor_sync(FULLMASK, lt, o);
          float v[4] = {0.f, 0.f, 0.f, 0.f};
          for (int k0 = 0; k0 < ncta; k0 += 4) {
            float4 o4[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (k0 + j < ncta) o4[j] = ld_cluster_f32x4(cluster_map(o_base + 4u * (i * kODep + 4 * lane), k0 + j));
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float sc = __shfl_sync(FULLMASK, sck, (k0 + j) & 31);
              if (k0 + j < ncta && sc != 0.f) {
                v[0] = fmaf(sc, o4[j].x, v[0]);
                v[1] = fmaf(sc, o4[j].y, v[1]);
                v[2] = fmaf(sc, o4[j].z, v[2]);
                v[3] = fmaf(sc, o4[j].w, v[3]);
              }
            }
          }
          if (p.cluster_split > 1) {
            const int sub = (int)cluster_id_x() % p.cluster_split;  // which of the pair's clusters
            const size_t prow = ((size_t)u * p.cluster_split + sub) * hq + i;
            reinterpret_cast<float4*>(p.part_o + prow * D)[lane] = make_float4(v[0], v[1], v[2], v[3]);
            if (lane == 0) p.part_ml[prow] = make_float2(M, lt);
            __threadfence();  // before the cluster barrier and the arrival count below
            continue;
          }
          if (p.has_win && M != -INFINITY && wml.x != -INFINITY) {
            const float sc = fast_exp2(wml.x - M);
            lt = fmaf(sc, wml.y, lt);
            const float4 w4 = __ldcg(reinterpret_cast<const float4*>(p.win_o + wr * D) + lane);
            v[0] = fmaf(sc, w4.x, v[0]);
            v[1] = fmaf(sc, w4.y, v[1]);
            v[2] = fmaf(sc, w4.z, v[2]);
            v[3] = fmaf(sc, w4.w, v[3]);
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) v[e] = lt > 0.f ? v[e] / lt : 0.f;
          if (p.rotation & 2) hadamard128(v, lane);
          store_row4(p.out + ((size_t)b * p.Hq + kvh * hq + i) * D, lane, v);
        }
      }
      cluster_sync();
      if (p.cluster_split > 1 && cluster_ctarank() == 0) {
        // The pair's clusters count their arrivals; the last merges their partials (and the
        // window's) into the output, one warp per query row.
        if (threadIdx.x == 0) {
          __threadfence();
          const int prev = atomicAdd(p.done + u, 1);
          s_last = (prev == p.cluster_split - 1);
        }
        __syncthreads();
        if (s_last) {
          __threadfence();
          const int ns = p.cluster_split;
          for (int i = warp; i < hq; i += W) {  // as in the cluster merge: lane k reads partial k
            const size_t wr = (size_t)u * hq + i;
            float2 mlk = make_float2(-INFINITY, 0.f);
            if (lane < ns) mlk = __ldcg(&p.part_ml[((size_t)u * ns + lane) * hq + i]);
            float M = mlk.x;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(FULLMASK, M, o));
            float2 wml = make_float2(-INFINITY, 0.f);
            if (p.has_win) {
              wml = __ldcg(&p.win_ml[wr]);
              M = fmaxf(M, wml.x);
            }
            const float sck = (M == -INFINITY || mlk.x == -INFINITY) ? 0.f : fast_exp2(mlk.x - M);
            float lt = sck * mlk.y;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) lt += __shfl_xor_sync(FULLMASK, lt, o);
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            for (int k0 = 0; k0 < ns; k0 += 4) {
              float4 o4[4];
#pragma unroll
              for (int j = 0; j < 4; ++j)
                if (k0 + j < ns)
                  o4[j] = __ldcg(reinterpret_cast<const float4*>(p.part_o + (((size_t)u * ns + k0 + j) * hq + i) * D) + lane);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float sc = __shfl_sync(FULLMASK, sck, (k0 + j) & 31);
                if (k0 + j < ns && sc != 0.f) {
                  v[0] = fmaf(sc, o4[j].x, v[0]);
                  v[1] = fmaf(sc, o4[j].y, v[1]);
                  v[2] = fmaf(sc, o4[j].z, v[2]);
                  v[3] = fmaf(sc, o4[j].w, v[3]);
                }
              }
            }
            if (p.has_win && M != -INFINITY && wml.x != -INFINITY) {
              const float sc = fast_exp2(wml.x - M);
              lt = fmaf(sc, wml.y, lt);
              const float4 w4 = __ldcg(reinterpret_cast<const float4*>(p.win_o + wr * D) + lane);
              v[0] = fmaf(sc, w4.x, v[0]);
              v[1] = fmaf(sc, w4.y, v[1]);
              v[2] = fmaf(sc, w4.z, v[2]);
              v[3] = fmaf(sc, w4.w, v[3]);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] = lt > 0.f ? v[e] / lt : 0.f;
            if (p.rotation & 2) hadamard128(v, lane);
            store_row4(p.out + ((size_t)b * p.Hq + kvh * hq + i) * D, lane, v);
          }
          if (threadIdx.x == 0) p.done[u] = 0;  // ready for the next call in stream order
        }
      }
      break;  // a cluster holds one pair: its only segment is done
    } else {
    // A pair held by this CTA alone is finished here (with the window's partial). Otherwise the
    // CTA writes its partial to its slot (1 when the pair is the second one it holds a
    // partial of, else 0) and the last contributor to arrive merges all partials (and the
    // window's) into the output.
    // The CTAs that hold items of this pair: c_first .. c_last on the cost axis (item x of
    // it costs x + wq); a CTA between them may hold none (its range inside the boundary).
    const long long pair_last = pair_first + pair_n - 1;
    const long long wq = (long long)ss.w * (q + 1);
    auto cta_at = [&](long long xi) { return (int)min((xi + wq) * p.n_cta / ss.ctot, (long long)p.n_cta - 1); };
    const int c_first = cta_at(pair_first), c_last = cta_at(pair_last);
    auto start_in_pair = [&](int cc) -> long long {  // first item of the pair CTA cc holds (clamped)
      if (cc <= c_first) return pair_first;
      return min(pair_last + 1, max(pair_first, split_threshold(cc, ss.ctot, p.n_cta) - wq));
    };
    // When every CTA range covers a cost unit or more, every CTA of the span holds items of
    // the pair; only smaller problems need the test.
    const bool sparse = ss.ctot < p.n_cta;
    auto holds = [&](int cc) { return !sparse || start_in_pair(cc + 1) > start_in_pair(cc); };
    // partial slot 1 for the last pair of a CTA that began in an earlier pair, else 0
    const int slot_first = split_threshold(c_first, ss.ctot, p.n_cta) < pair_first + wq - ss.w ? 1 : 0;
    auto slot_of = [&](int cc) { return cc == c_first ? slot_first : 0; };
    int n_contrib = c_last - c_first + 1;
    if (sparse) {
      n_contrib = 0;
      for (int cc = c_first; cc <= c_last; ++cc) n_contrib += holds(cc);
    }
    const bool alone = (n_contrib == 1);
    // the window kernel launched before this grid (programmatic dependent launch) wrote the
    // window partials read below
    if (p.has_win) grid_dependency_wait();
    for (int idx = threadIdx.x; idx < hq * D; idx += C::THREADS) {
      const int i = idx / D, ch = idx % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kMergeWarps; ++w) M = fmaxf(M, ma.m[w * kMaxHq + i]);
      float acc = 0.f, lt = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kMergeWarps; ++w) {
          const float mw = ma.m[w * kMaxHq + i];
          const float sc = (mw == -INFINITY) ? 0.f : fast_exp2(mw - M);
          acc = fmaf(sc, ma.o[(w * hq + i) * kODep + ch], acc);
          lt = fmaf(sc, ma.l[w * kMaxHq + i], lt);
        }
      }
      if (alone) {
        if (p.has_win) {  // merge the window's partial of the pair
          const size_t wr = (size_t)u * hq + i;
          const float2 wml = __ldcg(&p.win_ml[wr]);
          const float Mw = fmaxf(M, wml.x);
          if (Mw != -INFINITY) {
            const float a = (M == -INFINITY) ? 0.f : fast_exp2(M - Mw);
            const float bw = (wml.x == -INFINITY) ? 0.f : fast_exp2(wml.x - Mw);
            acc = a * acc + bw * __ldcg(&p.win_o[wr * D + ch]);
            lt = a * lt + bw * wml.y;
          }
        }
        const float o = lt > 0.f ? acc / lt : 0.f;
        if (p.rotation & 2)
          sQ[idx] = o;  // rotated back below
        else
          p.out[((size_t)b * p.Hq + kvh * hq + i) * D + ch] = __float2bfloat16_rn(o);
      } else {
        const size_t prow = ((size_t)cta * 2 + slot_of(cta)) * hq + i;
        p.part_o[prow * D + ch] = acc;
        if (ch == 0) p.part_ml[prow] = make_float2(M, lt);
      }
    }
    if (alone && (p.rotation & 2)) {
      __syncthreads();
      rotate_out_rows(sQ, hq, (size_t)b * p.Hq + kvh * hq);
    }
    if (!alone) {
      // out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s (zero when no token at all)
      __syncthreads();
      if (threadIdx.x == 0) {
        __threadfence();  // this CTA's partial is visible before the count says so
        const int prev = atomicAdd(p.done + u, 1);
        s_last = (prev == n_contrib - 1);
      }
      __syncthreads();
      if (s_last) {
        __threadfence();
        // contributor k < n_span is CTA c_first + k (those without items are skipped); the
        // window's partial comes last
        const int n_span = c_last - c_first + 1;
        const int n_used = n_span + p.has_win;
        // in the merge area (free again): per contributor and query the scale 2^(m_s - M),
        // then per contributor the partial row of query 0 (-1 without items); per query the
        // merged denominator
        float* s_sc = ma.o;                                  // [n_used][hq]
        int* s_row = reinterpret_cast<int*>(s_sc + n_used * hq);  // [n_used]
        float* s_l = ma.l;                                   // [hq]
        for (int k = threadIdx.x; k < n_used; k += C::THREADS) {
          int r = u * hq;  // window
          if (k < n_span) {
            const int cc = c_first + k;
            r = holds(cc) ? (cc * 2 + slot_of(cc)) * hq : -1;
          }
          s_row[k] = r;
        }
        __syncthreads();
        auto ml_of = [&](int k, int i) -> float2 {
          const int r = s_row[k];
          if (r < 0) return make_float2(-INFINITY, 0.f);
          return __ldcg(k == n_span ? &p.win_ml[r + i] : &p.part_ml[r + i]);
        };
        // warp i: the maximum over the partials of query i, each partial's scale and the
        // merged denominator (the partials' (m, l) of lane k held between the two steps)
        for (int i = warp; i < hq; i += W) {
          float M = -INFINITY;
          float2 ml0 = make_float2(-INFINITY, 0.f);
          if (lane < n_used) ml0 = ml_of(lane, i);
          M = ml0.x;
          for (int k = lane + 32; k < n_used; k += 32) M = fmaxf(M, ml_of(k, i).x);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(FULLMASK, M, o));
          float lt = 0.f;
          for (int k = lane; k < n_used; k += 32) {
            const float2 ml = (k == lane) ? ml0 : ml_of(k, i);
            const float sc = (M == -INFINITY || ml.x == -INFINITY) ? 0.f : fast_exp2(ml.x - M);
            s_sc[k * hq + i] = sc;
            lt = fmaf(sc, ml.y, lt);
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) lt += __shfl_xor_sync(FULLMASK, lt, o);
          if (lane == 0) s_l[i] = lt;
        }
        __syncthreads();
        // the weighted sums: a thread's loads of up to 16 partials are issued together
        for (int idx = threadIdx.x; idx < hq * D; idx += C::THREADS) {
          const int i = idx / D, ch = idx % D;
          float acc = 0.f;
          for (int k0 = 0; k0 < n_used; k0 += 16) {
            float sc[16], v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int k = k0 + j;
              sc[j] = 0.f;
              v[j] = 0.f;
              if (k < n_used) {
                sc[j] = s_sc[k * hq + i];
                if (sc[j] != 0.f) {
                  const size_t r = (size_t)(s_row[k] + i) * D + ch;
                  v[j] = __ldcg(k == n_span ? &p.win_o[r] : &p.part_o[r]);
                }
              }
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) acc = fmaf(sc[j], v[j], acc);
          }
          const float l = s_l[i];
          const float o = l > 0.f ? acc / l : 0.f;
          if (p.rotation & 2)
            sQ[idx] = o;  // rotated back below
          else
            p.out[((size_t)b * p.Hq + kvh * hq + i) * D + ch] = __float2bfloat16_rn(o);
        }
        if (p.rotation & 2) {
          __syncthreads();
          rotate_out_rows(sQ, hq, (size_t)b * p.Hq + kvh * hq);
        }
        if (threadIdx.x == 0) p.done[u] = 0;  // ready for the next call in stream order
      }
    }

    }

    // next pair with tokens
    x = xe;
    pair_first += pair_n;
    if (x < X1) {
      do {
        ++u;
        pair_n = items_of(seq_len(u / p.Hkv));
      } while (pair_n == 0);
      ++q;
    }
  }

  // ---------------------------------------------------- pairs without cached tokens
  // Their output is the window's attention alone, or zero.
  if (p.has_win) grid_dependency_wait();
  for (int bq = cta; bq < p.B; bq += p.n_cta) {
    if (seq_len(bq) != 0) continue;
    if (p.rotation & 2) {  // values stored rotated: each output row is rotated back
      for (int r = warp; r < p.Hq; r += W) {
        const size_t row = (size_t)bq * p.Hq + r;  // the window partial row is the output row
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (p.has_win) {
          const float2 ml = __ldcg(&p.win_ml[row]);
          if (ml.y > 0.f) {
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] = __ldcg(&p.win_o[row * D + 4 * lane + e]) / ml.y;
          }
        }
        hadamard128(v, lane);
        store_row4(p.out + row * D, lane, v);
      }
      continue;
    }
    for (int idx = threadIdx.x; idx < p.Hkv * hq * D; idx += C::THREADS) {
      const int kv = idx / (hq * D), i = (idx / D) % hq, ch = idx % D;
      float o = 0.f;
      if (p.has_win) {
        const long long r = (long long)(bq * p.Hkv + kv) * hq + i;
        const float2 ml = __ldcg(&p.win_ml[r]);
        if (ml.y > 0.f) o = __ldcg(&p.win_o[r * D + ch]) / ml.y;
      }
      p.out[((size_t)bq * p.Hq + kv * hq + i) * D + ch] = __float2bfloat16_rn(o);
    }
  }

  if (failed && lane == 0) {
    // every copy issued must have landed before shared memory is freed: wait (bounded)
    // for each outstanding half in issue order
    int rk = 0, pk = 0;
    for (int k = 0; k < n_issued + (k_pending ? 1 : 0); ++k) {
      if (k >= n_k_read && !mbar_wait(bar_k(rk), pk, p.status, kStatusDrainTimeout)) break;
      if (++rk == R) { rk = 0; pk ^= 1; }
    }
    int rv = 0, pv = 0;
    for (int k = 0; k < n_issued; ++k) {
      if (k >= n_v_read && !mbar_wait(bar_v(rv), pv, p.status, kStatusDrainTimeout)) break;
      if (++rv == R) { rv = 0; pv ^= 1; }
    }
  }
}

}  // namespace lbkv
