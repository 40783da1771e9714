// lbkv_decode_grp.cuh -- split-KV decode attention for a token-wise K side with the QK^T
// product on the 5th-generation tensor cores, one product per 128-token item, shared by a
// group of four warps.
//
// Method: "FOSCAR: Accelerating Decode Attention over 2- and 4-Bit KV Caches through
// Affine Folding" (arXiv:2611.09722), abstract; the explainer "FOSCAR speeds up 2-bit KV
// decode -- Affine folding of KV dequantization", fold rule and fold table (token-wise K:
// acc-fold, s times each group's partial score plus z times the query's sum over the group,
// before the softmax; token-wise V: operand-fold on the weights; channel-wise V: acc-fold of
// each token group's partial output, before the final division).
//
// Operands of the QK^T product (kind::f8f6f4, fp32 accumulators in tensor memory):
//  - A = the K codes: a code q is the e4m3 value q 2^-9 when written into the low bits of a
//    byte (the e4m3 subnormals and its first normal binade are evenly spaced, so 2- and 4-bit
//    codes need no magic-number bias); a thread spreads its token's codes into bytes, four
//    codes per shift and AND, and stores the 128 bytes as its row in tensor memory (one TMEM
//    lane per token; a warp reaches the 32 lanes of its quadrant).
//  - B = the query: Q 2^e split into e4m3 terms (the second scaled by 16, the third by 256;
//    three terms are exact for a bf16 query) in shared memory. With several K channel groups
//    per token B is block-diagonal, columns (group, query, term), so each group's partial
//    score has its own accumulator column: an unscaled partial never crosses a group boundary.
// Each thread reads its token's scores back from tensor memory and applies the acc-fold. A
// warp issues at most one tcgen05 product per ~57 cycles (measured on GB300), and a product
// with M = 128 rows costs the tensor core the same whether 32 or 128 of its rows are used
// (~9 cycles for N = 16), so an item of 128 tokens is one product: the four warps of a group
// (one per TMEM lane quadrant) each convert 32 of its tokens, and the last of them to finish
// issues the four K-steps, with no barrier (an arrival counter in shared memory).
//
// Work organisation. A persistent grid, one CTA per SM, warps in groups of four. The items
// of the CTA's share of the item sequence go to the groups in turn. A group streams its
// items through its own ring in shared memory (K half and V half per entry, 1-D bulk copies,
// mbarriers with bounded waits, no multicast); the last warp to convert an item refills the
// entry's K half and the last warp to finish an item's PV refills its V half. Each warp
// converts the next item before it consumes the current one (two A buffers and two score
// buffers per group), so that a product runs while the warps do the softmax and PV of the
// previous item. Every warp keeps its own online-softmax state over its 32 tokens of each
// item (running maximum raised only when a score exceeds it by more than 2^8, in exponent-2
// units), and its own PV accumulators (mma.sync, fed weights through shared memory and
// ldmatrix.trans). Pair boundaries, the merges of the warps and of the CTAs, the work split,
// the paged cache, the rotation and the bf16 window are those of the split-decode kernel.
#pragma once

#include "lbkv_decode.cuh"
#include "lbkv_tc.cuh"

namespace lbkv {

__host__ __device__ constexpr int tmem_pow2(int x) {
  int n = 32;
  while (n < x) n <<= 1;
  return n;
}

// Channel of K-operand element kappa (0..127) after the spread of a token's codes into
// bytes (word w of the row, shift k, byte b: element 16 w + 4 k + b at INT2, 8 w + 4 k + b at
// INT4), which permutes the channels; the query tile uses the same order.
template <int BITS>
__host__ __device__ constexpr int grp_k_channel(int kappa) {
  return BITS == 2 ? 16 * (kappa >> 4) + 4 * (kappa & 3) + ((kappa >> 2) & 3)
                   : 8 * (kappa >> 3) + 2 * (kappa & 3) + ((kappa >> 2) & 1);
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

// Compile-time shape of one variant (token-wise K); C = Cfg<BITS, 0, VL, MODE, LOG2G>.
template <class C>
struct GrpShape {
  static constexpr int UNIT = 128;              // tokens per item (4 warps x 32)
  static constexpr int GROUPS = C::WARPS / 4;   // warp groups
  // queries per KV head at most, and (query, V group) combos at most, in the column mode
  static constexpr int MQ = (C::MODE == kModeDup ? 4 : C::MODE == kModePair ? 8 : 16) / C::GV;
  static constexpr int MC = MQ * C::GV;
  // tensor memory of a group: A x2 (32 columns each), scores x2 (NS columns each)
  static constexpr int NS_MAX = (512 / GROUPS - 64) / 2;
  static constexpr int T = (C::GK * MQ * 3 <= NS_MAX) ? 3 : 2;  // e4m3 terms of the query
  static constexpr int NS = (C::GK * MQ * T + 15) / 16 * 16;
  static constexpr bool OK = C::KL == 0 && NS <= NS_MAX;
  static constexpr int TMG = 64 + 2 * NS;
  static constexpr int TMC = tmem_pow2(GROUPS * TMG);
  static constexpr EntryLayout E = entry_layout(C::BITS, 0, C::VL, UNIT, C::G);
  static constexpr int P_ROW = C::NTV * 16;  // bytes of one token's fed weights
  // shared memory: mbarriers | counters and issue cursors | Q and per-query constants |
  // B tile | weight tiles | merge area | rings
  static constexpr int MAX_RING = 12;        // ring entries per group at most
  static constexpr int CNT_OFF = 1024;
  static constexpr int Q_OFF = 2048;
  static constexpr int B_OFF = 7168;
  static constexpr int P_OFF = B_OFF + 96 * 128;
  static constexpr int MERGE_OFF = kGrpMergeOffset;
  static_assert(P_OFF + 8192 <= MERGE_OFF, "weight tiles fit");
  static_assert(GROUPS * (2 * MAX_RING + 2) * 8 <= CNT_OFF, "mbarriers fit");
  static_assert(Q_OFF + 4 * (kMaxHq * kHeadDim + 6 * kMaxHq) <= B_OFF, "prologue fits");
  static_assert(!OK || NS <= 96, "B tile fits");
  static_assert(C::WARPS * 32 * P_ROW <= 8192, "weight tiles fit");
};

// An issue cursor of a group (K half or V half), kept in shared memory and advanced by
// whichever thread issues the group's next copy.
struct GrpCursor {
  int i, u, t, L, n, b, kvh, pos;  // local item, pair, item in pair, pair tokens and items,
                                   // sequence, cached KV head, position in the group's sequence
};
// Arrival counters per group and position parity: a warp converts position j + 2 only after
// the product of j (so after every warp converted j), and finishes position j + 2 only after
// every warp converted j + 2 (so after every warp finished j): the four arrivals of a
// position never interleave with those of the next position of the same parity, while
// those of consecutive positions may.
struct GrpShared {
  unsigned conv_cnt[4][2];  // warps that converted an item (acquire-release counters)
  unsigned done_cnt[4][2];  // warps that finished an item's PV
  int n_commit[4];          // products committed per group
  int pad[4];
  GrpCursor kc[4], vc[4];   // issue cursors per group
};

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "r"(smem_addr(p)), "r"(v)
               : "memory");
  return old;
}

template <class C, bool PAGED>
__global__ void __launch_bounds__(C::THREADS, 1) grp_decode_kernel(const __grid_constant__ DecodeParams p) {
  using S = GrpShape<C>;
  static_assert(S::OK, "shape of the group variant");
  constexpr int BITS = C::BITS, VL = C::VL, GV = C::GV, GK = C::GK, NQ = C::NQ, NO = C::NO, NTV = C::NTV;
  constexpr int RB = C::RB, D = kHeadDim, UNIT = S::UNIT, W = C::WARPS, NG = S::GROUPS;
  constexpr int MQ = S::MQ, MC = S::MC, T = S::T, NS = S::NS;
  constexpr unsigned FULLMASK = 0xffffffffu;
  constexpr int FED_CW = 32;  // channel-wise V: weights fed as P * 32 (P <= 2^8 under the lazy maximum)
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ SplitScan ss;
  __shared__ int s_last;
  __shared__ uint32_t s_tmem;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int grp = warp >> 2, quad = warp & 3;
  const int cta = blockIdx.x;
  const int hq = p.hq;
  const int n_pairs = p.B * p.Hkv;
  const int R = p.ring_per_warp;  // ring entries per group

  GrpShared* gs = reinterpret_cast<GrpShared*>(smem + S::CNT_OFF);
  float* sQ = reinterpret_cast<float*>(smem + S::Q_OFF);   // [kMaxHq][D]
  int* sEq = reinterpret_cast<int*>(sQ + kMaxHq * D);      // [kMaxHq] query exponent
  float* sA = reinterpret_cast<float*>(sEq + kMaxHq);      // [kMaxHq] score factor
  float* sBz = sA + kMaxHq;                                // [kMaxHq][4] offset factors
  uint8_t* btile = smem + S::B_OFF;
  uint8_t* ptile = smem + S::P_OFF + warp * 32 * S::P_ROW;
  MergeArea ma;
  ma.m = reinterpret_cast<float*>(smem + S::MERGE_OFF);
  ma.l = ma.m + kMergeWarps * kMaxHq;
  ma.o = ma.l + kMergeWarps * kMaxHq;
  uint8_t* ring_g = smem + p.ring_off + (size_t)grp * R * S::E.bytes;
  const uint32_t bar_g = smem_addr(smem) + 8u * (uint32_t)(grp * (2 * R + 2));
  auto kbar = [&](int r) { return bar_g + 8u * r; };
  auto vbar = [&](int r) { return bar_g + 8u * (R + r); };
  auto sbar = [&](int b) { return bar_g + 8u * (2 * R + b); };

  auto seq_len = [&](int b) { return min(max(__ldg(p.seq_lens + b), 0), p.T_cap); };
  auto items_of = [&](int L) { return (L + UNIT - 1) / UNIT; };
  auto rotate_out_rows = [&](const float* rows, int n, size_t out_row0) {
    for (int i = warp; i < n; i += W) {
      float v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = rows[i * D + 4 * lane + e];
      hadamard128(v, lane);
      store_row4(p.out + (out_row0 + i) * D, lane, v);
    }
  };

  // ---------------------------------------------------- tensor memory, barriers, counters
  if (warp == 0) tc::alloc(smem_addr(&s_tmem), S::TMC);
  if (threadIdx.x == 0) {
    for (int G = 0; G < NG; ++G) {
      const uint32_t b0 = smem_addr(smem) + 8u * (uint32_t)(G * (2 * R + 2));
      for (int r = 0; r < 2 * R + 2; ++r) mbar_init(b0 + 8u * r, 1);
      gs->conv_cnt[G][0] = gs->conv_cnt[G][1] = gs->done_cnt[G][0] = gs->done_cnt[G][1] = 0u;
      gs->n_commit[G] = 0;
    }
    mbar_init_fence();
  }
  tc::fence_before_sync();

  // ---------------------------------------------------- the CTA's share of the items
  {
    const int chunk = (p.B + W - 1) / W;
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
      const int sw = (tot >= 8LL * NG * p.n_cta) ? p.split_w : 0;
      for (int w = 0; w < W; ++w) ss.cost[w] = ss.items[w] + (long long)sw * ss.pairs[w];
      const long long ctot = tot + (long long)sw * np;
      ss.w = sw;
      ss.ctot = ctot;
      for (int e = 0; e < 2; ++e) {
        const long long Tt = split_threshold(cta + e, ctot, p.n_cta);
        ss.kw[e] = W;
        ss.x[e] = tot;
        long long ac = 0, ai = 0, ap = 0;
        for (int w = 0; w < W; ++w) {
          if (Tt < ac + ss.cost[w]) {
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
      if (warp != ss.kw[e]) continue;
      const long long Tt = split_threshold(cta + e, ss.ctot, p.n_cta);
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
        const long long ec = rc + ic - c_b;
        const unsigned hit = __ballot_sync(FULLMASK, c_b > 0 && Tt >= ec && Tt < ec + c_b);
        if (hit) {
          if (lane == __ffs(hit) - 1) {
            const long long off = Tt - ec;
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
  tc::fence_after_sync();
  const uint32_t tm_g = s_tmem + (uint32_t)(grp * S::TMG);  // this group's columns (lane 0)
  const uint32_t tm_lane = (uint32_t)(32 * quad) << 16;      // this warp's lane quadrant
  const long long X0 = ss.x[0], X1 = ss.x[1];
  const int NL = (int)(X1 - X0);

  // ---------------------------------------------------- cursors over the item sequence
  auto set_pair = [&](GrpCursor& k) {
    const int b = k.u / p.Hkv;
    k.L = seq_len(b);
    k.n = items_of(k.L);
    k.b = b;
    k.kvh = (k.u - b * p.Hkv) >> p.kv_shift;
  };
  auto advance = [&](GrpCursor& k, int step) {
    k.i += step;
    k.t += step;
    k.pos += 1;
    if (k.i < NL) {
      while (k.t >= k.n) {
        k.t -= k.n;
        ++k.u;
        set_pair(k);
      }
    }
  };
  GrpCursor start;
  start.i = 0;
  start.pos = -1;  // the first advance (by the group index) lands on position 0
  if (NL > 0) {
    start.u = ss.b0 * p.Hkv + ss.kv0;
    start.t = ss.t0;
    start.L = seq_len(ss.b0);
    start.n = items_of(start.L);
    start.b = ss.b0;
    start.kvh = ss.kv0 >> p.kv_shift;
  } else {
    start.u = n_pairs;
    start.t = 0;
    start.L = start.n = 0;
    start.b = start.kvh = 0;
  }

  // Bulk copies of the K or V half of the cursor's item into its ring entry (pos mod R).
  auto copy_half = [&](bool v_half, const GrpCursor& k) {
    const int r = k.pos % R;
    const int u = k.u >> p.kv_shift;
    const size_t t0 = (size_t)k.t * UNIT;
    size_t row0, blk0;
    if constexpr (PAGED) {
      int page = __ldg(p.page_table + (size_t)k.b * p.max_pages + (((unsigned)k.t * UNIT) >> p.log2_page));
      if (page < 0 || page >= p.num_pages) {
        atomicExch(p.status, kStatusBadPage);
        page = 0;
      }
      const size_t pu = (size_t)page * (p.Hkv >> p.kv_shift) + k.kvh;
      row0 = (pu << p.log2_page) + (t0 & ((size_t(1) << p.log2_page) - 1));
      blk0 = row0 / C::G;
    } else {
      row0 = (size_t)u * p.T_cap + t0;
      blk0 = (size_t)u * ((size_t)p.T_cap / C::G) + t0 / C::G;
    }
    const uint32_t dst = smem_addr(ring_g + (size_t)r * S::E.bytes);
    const uint64_t pol = l2_evict_first_policy();
    fence_proxy_async_smem();
    if (!v_half) {
      const uint32_t fb = kbar(r);
      mbar_arrive_expect_tx(fb, S::E.tx_k);
      bulk_g2s(dst, p.k_codes + row0 * RB, UNIT * RB, fb, pol);
      bulk_g2s(dst + S::E.off_ks, p.k_scale + row0 * GK, S::E.sz_k, fb, pol);
      bulk_g2s(dst + S::E.off_kz, p.k_off + row0 * GK, S::E.sz_k, fb, pol);
    } else {
      const uint32_t fb = vbar(r);
      const size_t vs0 = (VL == 0) ? row0 * GV : blk0 * kHeadDim;
      mbar_arrive_expect_tx(fb, S::E.tx_v);
      bulk_g2s(dst + S::E.off_vc, p.v_codes + row0 * RB, UNIT * RB, fb, pol);
      bulk_g2s(dst + S::E.off_vs, p.v_scale + vs0, S::E.sz_v, fb, pol);
      bulk_g2s(dst + S::E.off_vz, p.v_off + vs0, S::E.sz_v, fb, pol);
    }
  };
  // Issues the half of the group's next item if it is in the CTA's range (cursor in shared memory).
  auto issue_next = [&](bool v_half) {
    GrpCursor k = v_half ? gs->vc[grp] : gs->kc[grp];
    if (k.i >= NL) return;
    copy_half(v_half, k);
    advance(k, NG);
    if (v_half)
      gs->vc[grp] = k;
    else
      gs->kc[grp] = k;
  };

  // The first R items of each group, by the group's first thread.
  if (quad == 0 && lane == 0) {
    GrpCursor k = start;
    advance(k, grp);
    gs->kc[grp] = k;
    gs->vc[grp] = k;
    for (int r = 0; r < R; ++r) issue_next(false);
    for (int r = 0; r < R; ++r) issue_next(true);
  }

  // this warp's position in the group's items: the next item to convert
  GrpCursor cv = start;
  advance(cv, grp);
  int cv_r = 0, con_r = 0;         // ring entries of the next conversion and consumption
  uint32_t cv_ph = 0, con_ph = 0;  // their mbarrier phase parities
  bool failed = false;

  LaneCols lc;
  lc.g = g;
  lc.c = c;
  lc.lane = lane;
  lc.hq = hq;
  lc.u_lane = (GV == 1) ? 0 : (16 * g) / C::G;
  if (GV >= 2) {
    const int el = ((lc.u_lane - 2 * c) % GV + GV) % GV;
    lc.e_live = el <= 1 ? el : -1;
  } else {
    lc.e_live = 0;
  }
  int qslot[NQ];  // query of this lane's PV accumulator slot (or -1)
#pragma unroll
  for (int j = 0; j < NQ; ++j) qslot[j] = qk_query<C>(2 * c + j, hq);
  constexpr uint32_t idesc = tc::idesc_e4m3(128, NS);

  // Converts the K half of item position `pos` (entry cv_r) into this warp's lane quadrant of
  // A buffer pos & 1; keeps the token's K scales/offsets (half2 (s, z) per channel group).
  // The last warp of the group to arrive issues the product into score buffer pos & 1 and
  // refills the entry's K half with the group's next item.
  auto convert = [&](int pos, uint32_t (&ksz)[GK]) {
    if (!failed && !mbar_wait(kbar(cv_r), cv_ph, p.status, kStatusConsumerTimeout)) failed = true;
    const uint8_t* en = ring_g + (size_t)cv_r * S::E.bytes;
    const int tk = 32 * quad + lane;
    uint32_t out[32];
    if (BITS == 2) {
      const uint4* row = reinterpret_cast<const uint4*>(en + tk * RB);
      const int h = (lane >> 2) & 1;  // read order that keeps 8 lanes on 32 different banks
      const uint4 a = row[h], b2 = row[h ^ 1];
      const uint4 lo = h ? b2 : a, hi = h ? a : b2;
      const uint32_t wv[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) out[4 * j + kk] = (wv[j] >> (2 * kk)) & 0x03030303u;
    } else {
      const uint4* row = reinterpret_cast<const uint4*>(en + tk * RB);
#pragma unroll
      for (int s4 = 0; s4 < 4; ++s4) {
        const uint4 q4 = row[s4];
        const uint32_t wv[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          out[2 * (4 * s4 + j)] = wv[j] & 0x0F0F0F0Fu;
          out[2 * (4 * s4 + j) + 1] = (wv[j] >> 4) & 0x0F0F0F0Fu;
        }
      }
    }
    const __half* ks = reinterpret_cast<const __half*>(en + S::E.off_ks);
    const __half* kz = reinterpret_cast<const __half*>(en + S::E.off_kz);
#pragma unroll
    for (int cc = 0; cc < GK; ++cc)
      ksz[cc] = (uint32_t)__half_as_ushort(ks[tk * GK + cc]) | ((uint32_t)__half_as_ushort(kz[tk * GK + cc]) << 16);
    const int buf = pos & 1;
    tc::st32(tm_g + 32u * buf + tm_lane, out);
    tc::wait_st();
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) {
      const unsigned prev = atom_add_acq_rel(&gs->conv_cnt[grp][buf], 1u);
      if ((prev & 3u) == 3u) {  // the group's last warp: product, then the K refill
        tc::fence_after_sync();
        const uint32_t bb = smem_addr(btile);
#pragma unroll
        for (int s4 = 0; s4 < 4; ++s4)
          tc::mma_f8f6f4_ts(tm_g + 64u + (uint32_t)NS * buf, tm_g + 32u * buf + 8u * s4,
                            tc::smem_desc(bb + 256u * s4, 128u, 1024u), idesc, s4 > 0);
        tc::commit(sbar(buf));
        gs->n_commit[grp] += 1;
        if (!failed) issue_next(false);
      }
    }
    __syncwarp();
    if (++cv_r == R) cv_r = 0, cv_ph ^= 1u;
  };

  // ---------------------------------------------------- segments: the CTA's items of one pair
  long long x = X0;
  int u = start.u;
  long long pair_first = X0 - start.t;
  int pair_n = start.n;
  long long q = ss.q0;
  while (x < X1) {
    const long long xe = min(X1, pair_first + pair_n);
    const int b = u / p.Hkv, kvh = u % p.Hkv;

    // -------------------------------------------------- pair prologue: Q, constants, the B tile
    __syncthreads();
    for (int idx = threadIdx.x; idx < hq * D; idx += C::THREADS)
      sQ[idx] = __bfloat162float(p.q[((size_t)b * p.Hq + kvh * hq) * D + idx]);
    __syncthreads();
    if (p.rotation & 1) {
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
    for (int i = warp; i < kMaxHq; i += W) {
      // query exponent e: max |Q| 2^e in [2^7, 2^8) (the e4m3 terms reach 448); per K channel
      // group the query's sum (the offset term's other operand)
      float amax = 0.f, gsum = 0.f;
      if (i < hq) {
#pragma unroll
        for (int uu = 0; uu < 4; ++uu) {
          const float v = sQ[i * D + 4 * lane + uu];
          amax = fmaxf(amax, fabsf(v));
          gsum += v;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(FULLMASK, amax, o));
      constexpr int lanes_per_group = C::G / 4;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float other = __shfl_xor_sync(FULLMASK, gsum, o);
        if (o < lanes_per_group) gsum += other;
      }
      int e = 0;
      if (amax > 0.f) e = min(100, max(-100, 7 - ilog2f(amax)));
      if (lane == 0) {
        sEq[i] = e;
        // scores in exponent-2 units: sl2 * sum_c (s_c raw_c + z_c sum Q_c), raw_c = (product)
        // 2^(9 - e): the codes enter as q 2^-9, the query as Q 2^e
        sA[i] = i < hq ? p.sl2 * exp2i(9 - e) : 0.f;
      }
      if ((lane % lanes_per_group) == 0) sBz[i * 4 + lane / lanes_per_group] = i < hq ? p.sl2 * gsum : 0.f;
    }
    __syncthreads();
    for (int wi = threadIdx.x; wi < NS * 32; wi += C::THREADS) {
      const int n = wi >> 5, k4 = (wi & 31) * 4;
      const int cg = n / (MQ * T), i = (n / T) % MQ, tau = n % T;
      uint32_t word = 0;
      if (n < GK * MQ * T && i < hq) {
        const float sc = exp2i(sEq[i]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int ch = grp_k_channel<BITS>(k4 + j);
          if (ch / C::G != cg) continue;
          const float xq = sQ[i * D + ch] * sc;
          const uint32_t t0 = e4m3_rn(xq);
          const float r1 = (xq - e4m3_to_f32(t0)) * 16.f;
          const uint32_t t1 = e4m3_rn(r1);
          const float r2 = (r1 - e4m3_to_f32(t1)) * 16.f;
          const uint32_t t2 = e4m3_rn(r2);
          word |= (tau == 0 ? t0 : tau == 1 ? t1 : t2) << (8 * j);
        }
      }
      *reinterpret_cast<uint32_t*>(btile + (n >> 3) * 1024 + (k4 >> 4) * 128 + (n & 7) * 16 + (k4 & 15)) = word;
    }
    fence_proxy_async_smem();  // the tile is read by the tensor cores
    __syncthreads();

    // -------------------------------------------------- per-warp state of the segment
    WarpState<C> st;
    float m_run[MQ], lsum[MQ], zacc[VL == 0 ? MC : 1];
#pragma unroll
    for (int i = 0; i < MQ; ++i) m_run[i] = -INFINITY, lsum[i] = 0.f;
#pragma unroll
    for (int k2 = 0; k2 < (VL == 0 ? MC : 1); ++k2) zacc[k2] = 0.f;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int row = 0; row < 2; ++row)
#pragma unroll
        for (int i = 0; i < NQ; ++i) st.o_run[mt][row][i] = 0.f;

    // consumes the item at position pos with nv valid tokens (scores in buffer pos & 1,
    // entry con_r), then arrives; the group's last warp to arrive refills the entry's V half
    auto consume = [&](int pos, int nv, const uint32_t (&ksz)[GK]) {
      const int buf = pos & 1;
      const uint32_t sph = (uint32_t)((pos >> 1) & 1);
      const int tk = 32 * quad + lane;
      const bool live = !failed && 32 * quad < nv;  // warp-uniform
      if (live) {
        if (!mbar_wait(sbar(buf), sph, p.status, kStatusConsumerTimeout)) failed = true;
      }
      if (live && !failed) {
        tc::fence_after_sync();
        float dcol[NS];
#pragma unroll
        for (int cb = 0; cb < NS / 16; ++cb) {
          float d16[16];
          tc::ld16(tm_g + 64u + (uint32_t)NS * buf + tm_lane + 16u * cb, d16);
#pragma unroll
          for (int j = 0; j < 16; ++j) dcol[16 * cb + j] = d16[j];
        }
        tc::wait_ld();
        tc::fence_before_sync();  // the buffer is overwritten by a later product
        float xs[MQ];
        {
          float acc[MQ], off[MQ];
#pragma unroll
          for (int i = 0; i < MQ; ++i) acc[i] = off[i] = 0.f;
#pragma unroll
          for (int cg = 0; cg < GK; ++cg) {
            const float2 sz = half2_to_float2(ksz[cg]);
#pragma unroll
            for (int i = 0; i < MQ; ++i) {
              const int n0 = (cg * MQ + i) * T;
              float raw = fmaf(dcol[n0 + 1], 0.0625f, dcol[n0]);
              if (T == 3) raw = fmaf(dcol[n0 + 2], 0.00390625f, raw);
              acc[i] = fmaf(sz.x, raw, acc[i]);
              off[i] = fmaf(sz.y, sBz[i * 4 + cg], off[i]);
            }
          }
#pragma unroll
          for (int i = 0; i < MQ; ++i) xs[i] = (tk < nv) ? fmaf(sA[i], acc[i], off[i]) : -INFINITY;
        }
        // running maximum, raised only by more than 2^8 (the weights of this item stay below 2^8)
        {
          bool grow = false;
#pragma unroll
          for (int i = 0; i < MQ; ++i) grow |= (xs[i] > m_run[i] + 8.f);
          if (__any_sync(FULLMASK, grow)) {
            float alpha[MQ];
#pragma unroll
            for (int i = 0; i < MQ; ++i) {
              float mx = xs[i];
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(FULLMASK, mx, o));
              const float mn = fmaxf(m_run[i], mx);
              alpha[i] = (mn == -INFINITY) ? 1.f : fast_exp2(m_run[i] - mn);
              m_run[i] = mn;
              lsum[i] *= alpha[i];
            }
            if (VL == 0) {
#pragma unroll
              for (int k2 = 0; k2 < MC; ++k2) zacc[k2] *= alpha[k2 / GV];
            }
#pragma unroll
            for (int j = 0; j < NQ; ++j) {
              float a = 1.f;
#pragma unroll
              for (int i = 0; i < MQ; ++i)
                if (i == qslot[j]) a = alpha[i];
#pragma unroll
              for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                for (int row = 0; row < 2; ++row) st.o_run[mt][row][j] *= a;
            }
          }
        }
        float P[MQ];
#pragma unroll
        for (int i = 0; i < MQ; ++i) {
          P[i] = fast_exp2(xs[i] - m_run[i]);  // -inf (padding) gives 0
          lsum[i] += P[i];
        }
        if (!mbar_wait(vbar(con_r), con_ph, p.status, kStatusConsumerTimeout)) failed = true;
        const uint8_t* en = ring_g + (size_t)con_r * S::E.bytes;
        SlotSmem sm;
        sm.kc = en;
        sm.vc = en + S::E.off_vc;
        sm.ks = reinterpret_cast<const __half*>(en + S::E.off_ks);
        sm.kz = reinterpret_cast<const __half*>(en + S::E.off_kz);
        sm.vs = reinterpret_cast<const __half*>(en + S::E.off_vs);
        sm.vz = reinterpret_cast<const __half*>(en + S::E.off_vz);
        // fed weights per (query, V group) combo, fp16: token-wise V P s 2^eP with max(s) 2^eP
        // in [2^6, 2^7) over the warp's valid tokens (fed values below 2^15); channel-wise V P * 32
        float fw[MC];
        float inv_ps = 1.f;
        if (VL == 0) {
          float sv[GV], zv[GV];
          uint32_t sb = 0;
          const bool okt = tk < nv;
#pragma unroll
          for (int uu = 0; uu < GV; ++uu) {
            const __half hs = sm.vs[tk * GV + uu], hz = sm.vz[tk * GV + uu];
            sv[uu] = okt ? __half2float(hs) : 0.f;  // padding tokens may hold any scale bits
            zv[uu] = okt ? __half2float(hz) : 0.f;
            sb = max(sb, okt ? (uint32_t)(__half_as_ushort(hs) & 0x7fffu) : 0u);
          }
          sb = __reduce_max_sync(FULLMASK, sb);
          const float smaxf = __half2float(__ushort_as_half((unsigned short)sb));
          int e2 = 0;
          if (smaxf > 0.f) e2 = min(100, max(-100, 6 - ilog2f(smaxf)));
          const float ps = exp2i(e2);
          inv_ps = exp2i(24 - e2);  // 2^-eP times the 2^24 of the subnormal V code images
#pragma unroll
          for (int k2 = 0; k2 < MC; ++k2) {
            const int i = k2 / GV, uu = k2 % GV;
            fw[k2] = P[i] * (sv[uu] * ps);
            zacc[k2] = fmaf(P[i], zv[uu], zacc[k2]);
          }
        } else {
#pragma unroll
          for (int k2 = 0; k2 < MC; ++k2) fw[k2] = P[k2] * (float)FED_CW;
        }
        // this token's row: column n of PV n-tile v holds combo DUP ? n / 2 : 8 v + n
        {
          uint32_t rw[NTV * 4];
#pragma unroll
          for (int j = 0; j < NTV * 4; ++j)
            rw[j] = C::DUP ? f16x2_from(fw[j], fw[j]) : f16x2_from(fw[2 * j], fw[2 * j + 1]);
#pragma unroll
          for (int v = 0; v < NTV; ++v)
            *reinterpret_cast<uint4*>(ptile + lane * S::P_ROW + 16 * v) =
                make_uint4(rw[4 * v], rw[4 * v + 1], rw[4 * v + 2], rw[4 * v + 3]);
        }
        __syncwarp();
        uint32_t pB[NTV][2][2];
#pragma unroll
        for (int v = 0; v < NTV; ++v)
          ldsm_x4_trans(smem_addr(ptile + lane * S::P_ROW + 16 * v), pB[v][0][0], pB[v][0][1], pB[v][1][0],
                        pB[v][1][1]);
        // channel-wise V: the sum of the fp16 weights fed to each PV accumulator column,
        // formed by the tensor cores with an all-ones A operand (the group's weight sum W)
        float fsum[NTV][2];
        if (VL == 1) {
          constexpr uint32_t kOnes2 = 0x3c003c00u;
#pragma unroll
          for (int v = 0; v < NTV; ++v) {
            float fs[4];
            mma_f16_c(fs, kOnes2, kOnes2, kOnes2, kOnes2, pB[v][0][0], pB[v][0][1], 0.f, 0.f, 0.f, 0.f);
            mma_f16(fs, kOnes2, kOnes2, kOnes2, kOnes2, pB[v][1][0], pB[v][1][1]);
            fsum[v][0] = fs[0];
            fsum[v][1] = fs[1];
          }
        }
        float accv[8][NTV][4];
        pv_chunk<C>(accv, pB, sm, 32 * quad, lc, true);
        if (VL == 0) {
          fold_tokenwise_v<C>(st, accv, inv_ps, lc);
        } else {
          float Wg[NO];
#pragma unroll
          for (int o = 0; o < NO; ++o) Wg[o] = fsum[0][C::DUP ? 0 : (o & 1)];
          const int tau = (32 * quad) / C::G;  // the warp's 32 tokens lie inside one token group
          fold_channelwise_v<C, FED_CW>(st, accv, Wg, sm.vs + tau * D, sm.vz + tau * D, lc);
        }
      }
      __syncwarp();  // the weight tile and the entry's V half are read
      if (lane == 0) {
        const unsigned prev = atom_add_acq_rel(&gs->done_cnt[grp][buf], 1u);
        if ((prev & 3u) == 3u && !failed) issue_next(true);  // the group's last warp: V refill
      }
      __syncwarp();
      if (++con_r == R) con_r = 0, con_ph ^= 1u;
    };

    // -------------------------------------------------- the group's items of this segment
    if (cv.i < NL && cv.u == u) {
      uint32_t ksz_cur[GK], ksz_nx[GK];
      int pos = cv.pos;
      int nv_cur = min(UNIT, cv.L - cv.t * UNIT);
      convert(pos, ksz_cur);
      advance(cv, NG);
      while (true) {
        const bool has_next = cv.i < NL && cv.u == u;
        int nv_nx = 0;
        if (has_next) {
          nv_nx = min(UNIT, cv.L - cv.t * UNIT);
          convert(pos + 1, ksz_nx);
          advance(cv, NG);
        }
        consume(pos, nv_cur, ksz_cur);
        if (!has_next) break;
        ++pos;
        nv_cur = nv_nx;
#pragma unroll
        for (int cc = 0; cc < GK; ++cc) ksz_cur[cc] = ksz_nx[cc];
      }
    }

    // -------------------------------------------------- warp totals into the merge format
    {
      float lt[MQ], zt[VL == 0 ? MC : 1];
#pragma unroll
      for (int i = 0; i < MQ; ++i) {
        float v = lsum[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULLMASK, v, o);
        lt[i] = v;
      }
      if (VL == 0) {
#pragma unroll
        for (int k2 = 0; k2 < MC; ++k2) {
          float v = zacc[k2];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULLMASK, v, o);
          zt[k2] = v;
        }
      }
      // per lane slot j (query qslot[j]): the running maximum (exponent-2 units, so pa = 1),
      // the warp's denominator and offset sums held by the lanes with g == 0 only
#pragma unroll
      for (int j = 0; j < NQ; ++j) {
        float m = -INFINITY, l = 0.f;
#pragma unroll
        for (int i = 0; i < MQ; ++i)
          if (i == qslot[j]) m = m_run[i], l = lt[i];
        st.m_run[j] = m;
        st.l[j] = (g == 0) ? l : 0.f;
      }
#pragma unroll
      for (int o = 0; o < NO; ++o) {
        float z = 0.f;
        if (VL == 0) {
          const int combo = own_combo<C>(c, o);
#pragma unroll
          for (int k2 = 0; k2 < MC; ++k2)
            if (k2 == combo) z = zt[k2];
        }
        st.zacc[o] = (g == 0) ? z : 0.f;
      }
    }

    // ---------------------------------------------------- warps beyond kMergeWarps fold in
    __syncthreads();
    if (C::WARPS > kMergeWarps) {
      constexpr int SF = 16 * NQ + NO + 2 * NQ;
      static_assert(SF <= kStateFloats, "handed-over state fits the merge area");
      float* xsa = ma.m;
      if (warp >= kMergeWarps) {
        float* d = xsa + (size_t)(warp - kMergeWarps) * SF * 32 + lane;
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
        const float* d = xsa + (size_t)warp * SF * 32 + lane;
        float aa[NQ], ab[NQ];
        int k = 0;
#pragma unroll
        for (int j = 0; j < NQ; ++j) {
          const float mb = d[32 * k++], lb = d[32 * k++];
          const float m = fmaxf(st.m_run[j], mb);
          aa[j] = (st.m_run[j] == m) ? 1.f : fast_exp2(st.m_run[j] - m);
          ab[j] = (mb == m) ? 1.f : fast_exp2(mb - m);
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
        const int qq = qslot[j];
        if (g == 0 && qq >= 0) {
          ma.m[warp * kMaxHq + qq] = st.m_run[j];
          ma.l[warp * kMaxHq + qq] = l;
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
#pragma unroll
      for (int i = 0; i < NQ; ++i) {
        const int o = live_own<C>(i, lc);
        if (o < 0) continue;
        const int combo = own_combo<C>(c, o);
        if (combo >= hq * GV || combo % GV != lc.u_lane) continue;
        const int qq = combo / GV;
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
            ma.o[(warp * hq + qq) * D + 16 * g + pv_channel<BITS>(mt, row)] = st.o_run[mt][row][i] + zt;
      }
    }
    __syncthreads();

    // ---------------------------------------------------- merge the warps, then the CTAs
    const long long pair_last = pair_first + pair_n - 1;
    const long long wq = (long long)ss.w * (q + 1);
    auto cta_at = [&](long long xi) { return (int)min((xi + wq) * p.n_cta / ss.ctot, (long long)p.n_cta - 1); };
    const int c_first = cta_at(pair_first), c_last = cta_at(pair_last);
    auto start_in_pair = [&](int cc) -> long long {
      if (cc <= c_first) return pair_first;
      return min(pair_last + 1, max(pair_first, split_threshold(cc, ss.ctot, p.n_cta) - wq));
    };
    const bool sparse = ss.ctot < p.n_cta;
    auto holds = [&](int cc) { return !sparse || start_in_pair(cc + 1) > start_in_pair(cc); };
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
          acc = fmaf(sc, ma.o[(w * hq + i) * D + ch], acc);
          lt = fmaf(sc, ma.l[w * kMaxHq + i], lt);
        }
      }
      if (alone) {
        if (p.has_win) {
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
          sQ[idx] = o;
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
      __syncthreads();
      if (threadIdx.x == 0) {
        __threadfence();
        const int prev = atomicAdd(p.done + u, 1);
        s_last = (prev == n_contrib - 1);
      }
      __syncthreads();
      if (s_last) {
        __threadfence();
        const int n_span = c_last - c_first + 1;
        const int n_used = n_span + p.has_win;
        auto row_of = [&](int k, int i) -> long long {
          if (k == n_span) return (long long)u * hq + i;
          const int cc = c_first + k;
          if (!holds(cc)) return -1;
          return ((long long)cc * 2 + slot_of(cc)) * hq + i;
        };
        auto ml_of = [&](int k, int i) -> float2 {
          const long long rr = row_of(k, i);
          if (rr < 0) return make_float2(-INFINITY, 0.f);
          return __ldcg(k == n_span ? &p.win_ml[rr] : &p.part_ml[rr]);
        };
        float* s_sc = ma.o;
        float* s_l = ma.l;
        for (int i = warp; i < hq; i += W) {
          float M = -INFINITY;
          for (int k = lane; k < n_used; k += 32) M = fmaxf(M, ml_of(k, i).x);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(FULLMASK, M, o));
          float lt = 0.f;
          for (int k = lane; k < n_used; k += 32) {
            const float2 ml = ml_of(k, i);
            const float sc = (M == -INFINITY || ml.x == -INFINITY) ? 0.f : fast_exp2(ml.x - M);
            s_sc[k * hq + i] = sc;
            lt = fmaf(sc, ml.y, lt);
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) lt += __shfl_xor_sync(FULLMASK, lt, o);
          if (lane == 0) s_l[i] = lt;
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < hq * D; idx += C::THREADS) {
          const int i = idx / D, ch = idx % D;
          float acc = 0.f;
#pragma unroll 4
          for (int k = 0; k < n_used; ++k) {
            const float sc = s_sc[k * hq + i];
            if (sc == 0.f) continue;
            const long long rr = row_of(k, i);
            acc = fmaf(sc, __ldcg(k == n_span ? &p.win_o[rr * D + ch] : &p.part_o[rr * D + ch]), acc);
          }
          const float l = s_l[i];
          const float o = l > 0.f ? acc / l : 0.f;
          if (p.rotation & 2)
            sQ[idx] = o;
          else
            p.out[((size_t)b * p.Hq + kvh * hq + i) * D + ch] = __float2bfloat16_rn(o);
        }
        if (p.rotation & 2) {
          __syncthreads();
          rotate_out_rows(sQ, hq, (size_t)b * p.Hq + kvh * hq);
        }
        if (threadIdx.x == 0) p.done[u] = 0;
      }
    }

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
  if (p.has_win) grid_dependency_wait();
  for (int bq = cta; bq < p.B; bq += p.n_cta) {
    if (seq_len(bq) != 0) continue;
    if (p.rotation & 2) {
      for (int rr = warp; rr < p.Hq; rr += W) {
        const size_t row = (size_t)bq * p.Hq + rr;
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
        const long long rr = (long long)(bq * p.Hkv + kv) * hq + i;
        const float2 ml = __ldcg(&p.win_ml[rr]);
        if (ml.y > 0.f) o = __ldcg(&p.win_o[rr * D + ch]) / ml.y;
      }
      p.out[((size_t)bq * p.Hq + kv * hq + i) * D + ch] = __float2bfloat16_rn(o);
    }
  }

  // ---------------------------------------------------- drain, then free the tensor memory
  // After a wait gave up the group's issued copies and committed products must still complete
  // before shared and tensor memory are released: each entry's last issued phase and each
  // score buffer's last commit (bounded waits).
  __syncthreads();
  if (quad == 0 && lane == 0) {
    bool any_failed = false;
    // (the failure flags are per thread; a timed-out wait also recorded the status word)
    any_failed = __ldcg(p.status) != 0;
    if (any_failed) {
      const int nk = gs->kc[grp].pos, nvv = gs->vc[grp].pos;
      for (int j = max(0, nk - R); j < nk; ++j)
        if (!mbar_wait(kbar(j % R), (uint32_t)((j / R) & 1), p.status, kStatusDrainTimeout)) break;
      for (int j = max(0, nvv - R); j < nvv; ++j)
        if (!mbar_wait(vbar(j % R), (uint32_t)((j / R) & 1), p.status, kStatusDrainTimeout)) break;
      const int nc = gs->n_commit[grp];
      for (int k2 = max(0, nc - 2); k2 < nc; ++k2)
        if (!mbar_wait(sbar(k2 & 1), (uint32_t)((k2 >> 1) & 1), p.status, kStatusDrainTimeout)) break;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::dealloc(s_tmem, S::TMC);
}

}  // namespace lbkv
