// lbkv_decode_tc.cuh -- split-KV decode attention over a 2-/4-bit affine-quantized KV
// cache with a token-wise K side, the QK^T product on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory) and the PV product on mma.sync.
//
// Method: "FOSCAR: Accelerating Decode Attention over 2- and 4-Bit KV Caches through
// Affine Folding" (arXiv:2611.09722), abstract; the explainer "FOSCAR speeds up 2-bit KV
// decode -- Affine folding of KV dequantization": fold rule and fold table (token-wise K:
// acc-fold, the group's partial score times s plus z times the sum of the query over the
// group, before the softmax; token-wise V: operand-fold on the weights; channel-wise V:
// acc-fold of each token group's partial output, before the final division).
//
// Why a second kernel. The mma.sync kernel turns every code into an fp16 operand with one
// LOP3 per two codes on the half-rate ALU pipe and spends 32 mma.sync per 32-token step;
// on GB300 that needs about 94 % of the whole instruction-issue budget at the HBM peak.
// Here the K side costs one shift and one AND per four codes and no warp-level products:
//  - A code q is the e4m3 value q * 2^-9 when written into the low bits of a byte (the
//    subnormal range of e4m3 and its first normal binade are evenly spaced, so INT2 and
//    INT4 codes need no magic-number bias). A thread owns one token: it spreads the
//    token's codes into bytes, four codes per word, and stores the 128 bytes as its row
//    of the A operand in tensor memory (lane = token).
//  - The B operand holds the query: Q * 2^e per query, split into three e4m3 terms (the
//    second and third scaled by 16 and 256), exact for a bf16 query; with several K
//    channel groups per token, B is block-diagonal (columns (group, query, term)), so each
//    group's partial score lands in its own accumulator column: an unscaled partial never
//    crosses a group boundary.
//  - One thread issues the four K-steps of 32 channels (kind::f8f6f4, M = 128 tokens);
//    each thread then reads its token's row of scores from tensor memory and applies the
//    acc-fold (s times the partial, plus z times the query's sum over the group).
// The PV product stays on mma.sync: its A operand (V transposed) comes from the codes by
// the magic-number images, two tokens interleaved per PRMT, exactly as in the other
// kernel, and its B operand (the weights, fed as fp16) goes from the token-per-thread
// layout of the scores to the fragment layout through shared memory (ldmatrix.trans).
//
// Work organisation. A persistent grid, one CTA per SM. The CTA's warps form groups of
// four (one warp per tensor-memory lane quadrant); an item is 128 tokens of one (sequence,
// KV head) pair, processed by one group, each warp owning 32 tokens. The items of the CTA's
// share go to the groups in turn. A group streams its items through its own ring of
// entries in shared memory (K half and V half, 1-D bulk copies issued by the group's first
// thread, completion on mbarriers with bounded waits, no multicast), converts the K half
// of the next item and issues its QK^T product before it finishes the current item (two
// accumulator buffers). Every warp keeps its own online-softmax state: its 32 tokens form
// one PV chunk per item, with a running maximum that is only raised when a score exceeds
// it by more than 2^8 (in exponent-2 units), so that the common case needs no cross-lane
// reduction. Pair boundaries, the merges of the warps and of the CTAs, the work split, the
// paged cache, the rotation and the bf16 window are those of the other kernel.
#pragma once

#include "lbkv_decode.cuh"
#include "lbkv_tc.cuh"

namespace lbkv {

__host__ __device__ constexpr int tmem_pow2(int x) {
  int n = 32;
  while (n < x) n <<= 1;
  return n;
}

// Compile-time shape of one variant (token-wise K).
template <int BITS_, int VL_, int MODE_, int LOG2G_>
struct TcCfg : Cfg<BITS_, 0, VL_, MODE_, LOG2G_> {
  using Base = Cfg<BITS_, 0, VL_, MODE_, LOG2G_>;
  static constexpr int UNIT = 128;                // tokens per item (4 warps x 32)
  static constexpr int GROUPS = Base::WARPS / 4;  // warp groups
  // queries per KV head at most, and (query, V group) combos at most, for the column mode
  static constexpr int MQ = (MODE_ == kModeDup ? 4 : MODE_ == kModePair ? 8 : 16) / Base::GV;
  static constexpr int MC = MQ * Base::GV;
  // e4m3 terms of the query (3 where tensor memory allows, else 2) and score columns
  static constexpr int NS3 = (Base::GK * MQ * 3 + 15) / 16 * 16;
  static constexpr int T = (GROUPS * 2 * (32 + NS3) <= 512) ? 3 : 2;
  static constexpr int NS = (Base::GK * MQ * T + 15) / 16 * 16;
  static constexpr int TMG = 2 * (32 + NS);  // tensor-memory columns of a group: A x2, scores x2
  static constexpr int TMC = tmem_pow2(GROUPS * TMG);
  static constexpr EntryLayout E = entry_layout(BITS_, 0, VL_, UNIT, Base::G);
  // shared memory: barriers | flags | Q and per-query constants | B tile | weight tiles | merge | rings
  static constexpr int FLAG_OFF = 1024;
  static constexpr int Q_OFF = 1088;
  static constexpr int B_OFF = 6144;
  static constexpr int P_ROW = Base::NTV * 16;  // bytes of one token's fed weights
  static constexpr int P_OFF = B_OFF + NS * 128;
  static constexpr int MERGE_OFF = P_OFF + Base::WARPS * 32 * P_ROW;
  static constexpr int MAX_RING = 12;  // ring entries per group at most (mbarrier space)
  static_assert(GROUPS * TMG <= 512, "tensor memory of the groups");
  static_assert(NS % 16 == 0 && NS <= 256, "N of an M = 128 product");
  static_assert(GROUPS * (2 * MAX_RING + 2) * 8 <= FLAG_OFF, "mbarriers fit");
  static_assert(Q_OFF + 4 * (kMaxHq * kHeadDim + kMaxHq + kMaxHq + 4 * kMaxHq) <= B_OFF, "prologue fits");
  static_assert(MERGE_OFF % 128 == 0, "merge area alignment");
};

// fp32 -> e4m3 (nearest, saturating) and back.
__device__ __forceinline__ uint32_t e4m3_rn(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.f), "f"(x));
  return r & 0xffu;
}
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)b));
  return __half2float(__ushort_as_half((unsigned short)(r & 0xffffu)));
}

// Channel of K-operand element kappa (0..127): the K side's codes are spread into bytes
// (word w of a token's row, shift k, byte b), which permutes the channels.
template <int BITS>
__host__ __device__ constexpr int tc_k_channel(int kappa) {
  return BITS == 2 ? 16 * (kappa >> 4) + 4 * (kappa & 3) + ((kappa >> 2) & 3)
                   : 8 * (kappa >> 3) + 2 * (kappa & 3) + ((kappa >> 2) & 1);
}

__device__ __forceinline__ void group_barrier(int grp) {
  asm volatile("bar.sync %0, 128;" ::"r"(1 + grp) : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

template <class C, bool PAGED>
__global__ void __launch_bounds__(C::THREADS, 1) tc_decode_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int BITS = C::BITS, VL = C::VL, GV = C::GV, GK = C::GK, NQ = C::NQ, NO = C::NO, NTV = C::NTV;
  constexpr int RB = C::RB, D = kHeadDim, UNIT = C::UNIT, W = C::WARPS, NG = C::GROUPS;
  constexpr int MQ = C::MQ, MC = C::MC, T = C::T, NS = C::NS;
  constexpr unsigned FULLMASK = 0xffffffffu;
  constexpr int FED_CW = 32;  // channel-wise V: weights fed as P * 32 (P <= 2^8 under the lazy maximum)
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ SplitScan ss;
  __shared__ int s_last;
  __shared__ uint32_t s_tmem;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int grp = warp >> 2, quad = warp & 3;
  const bool leader = (quad == 0) && (lane == 0);
  const int cta = blockIdx.x;
  const int hq = p.hq;
  const int n_pairs = p.B * p.Hkv;
  const int R = p.ring_per_warp;  // ring entries per group

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  volatile int* gfail = reinterpret_cast<volatile int*>(smem + C::FLAG_OFF);  // [NG] a wait of the group gave up
  float* sQ = reinterpret_cast<float*>(smem + C::Q_OFF);                     // [kMaxHq][D]
  int* sEq = reinterpret_cast<int*>(sQ + kMaxHq * D);                        // [kMaxHq] query exponent
  float* sA = reinterpret_cast<float*>(sEq + kMaxHq);                        // [kMaxHq] score factor
  float* sBz = sA + kMaxHq;                                                  // [kMaxHq][4] offset factors
  uint8_t* btile = smem + C::B_OFF;
  uint8_t* ptile = smem + C::P_OFF + warp * 32 * C::P_ROW;
  MergeArea ma;
  ma.m = reinterpret_cast<float*>(smem + C::MERGE_OFF);
  ma.l = ma.m + kMergeWarps * kMaxHq;
  ma.o = ma.l + kMergeWarps * kMaxHq;
  uint8_t* ring_g = smem + p.ring_off + (size_t)grp * R * C::E.bytes;
  const uint32_t bar_g = smem_addr(bars) + 8u * (uint32_t)(grp * (2 * R + 2));
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

  // ---------------------------------------------------- tensor memory and barriers
  if (warp == 0) tc::alloc(smem_addr(&s_tmem), C::TMC);
  if (threadIdx.x == 0) {
    for (int G = 0; G < NG; ++G) {
      const uint32_t b0 = smem_addr(bars) + 8u * (uint32_t)(G * (2 * R + 2));
      for (int r = 0; r < 2 * R + 2; ++r) mbar_init(b0 + 8u * r, 1);
      gfail[G] = 0;
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
  const uint32_t tm_g = s_tmem + (uint32_t)(grp * C::TMG);  // this group's columns
  const uint32_t tm_lane = (uint32_t)(32 * quad) << 16;      // this warp's lane quadrant
  auto tm_a = [&](int buf) { return tm_g + 32u * buf; };
  auto tm_s = [&](int buf) { return tm_g + 64u + (uint32_t)NS * buf; };
  const long long X0 = ss.x[0], X1 = ss.x[1];
  const int NL = (int)(X1 - X0);

  // ---------------------------------------------------- cursors over the group's items
  struct Cursor {
    int i, u, t, L, n;  // local item index, pair, item within the pair, pair's tokens and items
    int b, kvh;         // the pair's sequence and cached KV head
  };
  auto set_pair = [&](Cursor& k) {
    const int b = k.u / p.Hkv;
    k.L = seq_len(b);
    k.n = items_of(k.L);
    k.b = b;
    k.kvh = (k.u - b * p.Hkv) >> p.kv_shift;
  };
  auto advance = [&](Cursor& k, int step) {
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
  Cursor start;
  start.i = 0;
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

  // Bulk copies of the K or V half of the cursor's item into entry r (the group's first
  // thread only). A paged cache takes the item's page from the page table.
  auto copy_half = [&](bool v_half, const Cursor& k, int r) {
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
    const uint32_t dst = smem_addr(ring_g + (size_t)r * C::E.bytes);
    const uint64_t pol = l2_evict_first_policy();
    fence_proxy_async_smem();
    if (!v_half) {
      const uint32_t fb = kbar(r);
      mbar_arrive_expect_tx(fb, C::E.tx_k);
      bulk_g2s(dst, p.k_codes + row0 * RB, UNIT * RB, fb, pol);
      bulk_g2s(dst + C::E.off_ks, p.k_scale + row0 * GK, C::E.sz_k, fb, pol);
      bulk_g2s(dst + C::E.off_kz, p.k_off + row0 * GK, C::E.sz_k, fb, pol);
    } else {
      const uint32_t fb = vbar(r);
      const size_t vs0 = (VL == 0) ? row0 * GV : blk0 * kHeadDim;
      mbar_arrive_expect_tx(fb, C::E.tx_v);
      bulk_g2s(dst + C::E.off_vc, p.v_codes + row0 * RB, UNIT * RB, fb, pol);
      bulk_g2s(dst + C::E.off_vs, p.v_scale + vs0, C::E.sz_v, fb, pol);
      bulk_g2s(dst + C::E.off_vz, p.v_off + vs0, C::E.sz_v, fb, pol);
    }
  };

  // The group's items are local indices grp, grp + NG, ... of the CTA range, position j
  // of the group going through ring entry j mod R. The first thread keeps an issue cursor
  // per half; it issues the first R items, then refills an entry's K half once the group
  // has converted it and its V half once the group is done with the item.
  Cursor kis = start, vis = start;
  advance(kis, grp);
  advance(vis, grp);
  int kis_pos = 0, vis_pos = 0;
  if (leader) {
    for (; kis_pos < R && kis.i < NL; ++kis_pos) {
      copy_half(false, kis, kis_pos);
      advance(kis, NG);
    }
    for (; vis_pos < R && vis.i < NL; ++vis_pos) {
      copy_half(true, vis, vis_pos);
      advance(vis, NG);
    }
  }

  // consumer positions: next item to convert, next item to consume; products issued
  Cursor cv = start, con = start;
  advance(cv, grp);
  advance(con, grp);
  int cv_pos = 0, con_pos = 0;   // positions in the group's item sequence
  int cv_r = 0, con_r = 0;       // their ring entries (position mod R)
  uint32_t cv_ph = 0, con_ph = 0;  // and mbarrier phase parities (position / R mod 2)
  int kis_r = 0, vis_r = 0;  // ring entries of the next refills (the issue positions mod R)
  bool gf = false;      // the group gave up waiting (uniform: read after a group barrier)
  bool failed = false;  // this thread's own wait gave up
  int n_commit = 0;     // products committed by the leader (S barrier completions issued)

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
  const uint32_t idesc = tc::idesc_e4m3(128, NS);

  // Converts the K half of the item at `k` (position pos) into this warp's lane quadrant of
  // A buffer `buf` and keeps the token's K scales/offsets (half2 (s, z) per group).
  auto convert = [&](const Cursor& k, int r, uint32_t ph, int buf, uint32_t (&ksz)[GK]) {
    if (!gf && !failed && !mbar_wait(kbar(r), ph, p.status, kStatusConsumerTimeout)) {
      failed = true;
      gfail[grp] = 1;
    }
    const uint8_t* en = ring_g + (size_t)r * C::E.bytes;
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
      uint4 q4[4];
#pragma unroll
      for (int s = 0; s < 4; ++s) q4[s] = row[s];
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const uint32_t wv[4] = {q4[s].x, q4[s].y, q4[s].z, q4[s].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          out[2 * (4 * s + j)] = wv[j] & 0x0F0F0F0Fu;
          out[2 * (4 * s + j) + 1] = (wv[j] >> 4) & 0x0F0F0F0Fu;
        }
      }
    }
    const __half* ks = reinterpret_cast<const __half*>(en + C::E.off_ks);
    const __half* kz = reinterpret_cast<const __half*>(en + C::E.off_kz);
#pragma unroll
    for (int cc = 0; cc < GK; ++cc)
      ksz[cc] = (uint32_t)__half_as_ushort(ks[tk * GK + cc]) | ((uint32_t)__half_as_ushort(kz[tk * GK + cc]) << 16);
    tc::st32(tm_a(buf) + tm_lane, out);
    tc::wait_st();
    tc::fence_before_sync();
  };

  // After the group barrier that follows a conversion: the product of that item.
  auto issue_qk = [&](int buf) {
    if (!leader) return;
    tc::fence_after_sync();
    if (!gf) {
      const uint32_t bbase = smem_addr(btile);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        tc::mma_f8f6f4_ts(tm_s(buf), tm_a(buf) + 8u * s, tc::smem_desc(bbase + 256u * s, 128u, 1024u), idesc, s > 0);
      tc::commit(sbar(buf));
      ++n_commit;
    }
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

    // -------------------------------------------------- pair prologue: Q, the B tile, constants
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
      // query exponent e: max |Q| 2^e in [2^7, 2^8) (e4m3 reaches 448); per K channel group
      // the query's sum (the offset term's other operand)
      float amax = 0.f, gs = 0.f;
      if (i < hq) {
#pragma unroll
        for (int uu = 0; uu < 4; ++uu) {
          const float v = sQ[i * D + 4 * lane + uu];
          amax = fmaxf(amax, fabsf(v));
          gs += v;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(FULLMASK, amax, o));
      constexpr int lanes_per_group = C::G / 4;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float other = __shfl_xor_sync(FULLMASK, gs, o);
        if (o < lanes_per_group) gs += other;
      }
      int e = 0;
      if (amax > 0.f) e = min(100, max(-100, 7 - ilog2f(amax)));
      if (lane == 0) {
        sEq[i] = e;
        // scores in exponent-2 units: sl2 * sum_c (s_c * raw_c + z_c * sum Q_c), raw_c =
        // (accumulator) * 2^(9 - e): codes entered as q 2^-9, the query as Q 2^e
        sA[i] = i < hq ? p.sl2 * exp2i(9 - e) : 0.f;
      }
      if ((lane % lanes_per_group) == 0) sBz[i * 4 + lane / lanes_per_group] = i < hq ? p.sl2 * gs : 0.f;
    }
    __syncthreads();
    // B tile: column n = (K channel group cg, query i, term tau), element kappa; 4 bytes per store
    for (int wi = threadIdx.x; wi < NS * 32; wi += C::THREADS) {
      const int n = wi >> 5, k4 = (wi & 31) * 4;
      const int cg = n / (MQ * T), i = (n / T) % MQ, tau = n % T;
      uint32_t word = 0;
      if (n < GK * MQ * T && i < hq) {
        const float sc = exp2i(sEq[i]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int ch = tc_k_channel<BITS>(k4 + j);
          if (ch / C::G != cg) continue;
          const float xq = sQ[i * D + ch] * sc;
          const uint32_t t0 = e4m3_rn(xq);
          const float r1 = (xq - e4m3_to_f32(t0)) * 16.f;
          const uint32_t t1 = e4m3_rn(r1);
          const float r2 = (r1 - e4m3_to_f32(t1)) * 16.f;
          const uint32_t t2 = e4m3_rn(r2);
          const uint32_t tv = tau == 0 ? t0 : tau == 1 ? t1 : t2;
          word |= tv << (8 * j);
        }
      }
      const int off = (n >> 3) * 1024 + (k4 >> 4) * 128 + (n & 7) * 16 + (k4 & 15);
      *reinterpret_cast<uint32_t*>(btile + off) = word;
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

    // consumes the item at `k` (position pos, scores in buffer buf, token's K scales ksz)
    auto consume = [&](const Cursor& k, int pos, int r, uint32_t ph, const uint32_t (&ksz)[GK]) {
      const int buf = pos & 1;
      const uint32_t sph = (uint32_t)((pos >> 1) & 1);
      const int nv = min(UNIT, k.L - k.t * UNIT);
      const int tk = 32 * quad + lane;
      if (!gf && !failed && !mbar_wait(sbar(buf), sph, p.status, kStatusConsumerTimeout)) {
        failed = true;
        gfail[grp] = 1;
      }
      if (gf || 32 * quad >= nv) return;  // no valid token in this warp's 32 (or the group gave up)
      tc::fence_after_sync();
      // ------------------------------------------------ scores (exponent-2 units)
      float dcol[NS];
#pragma unroll
      for (int cb = 0; cb < NS / 16; ++cb) {
        float d16[16];
        tc::ld16(tm_s(buf) + tm_lane + 16u * cb, d16);
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
      // ------------------------------------------------ running maximum: raised only when a
      // score exceeds it by more than 2^8 (then the weights of this item stay below 2^8)
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
      // ------------------------------------------------ V half of the entry
      if (!failed && !mbar_wait(vbar(r), ph, p.status, kStatusConsumerTimeout)) {
        failed = true;
        gfail[grp] = 1;
      }
      const uint8_t* en = ring_g + (size_t)r * C::E.bytes;
      SlotSmem sm;
      sm.kc = en;
      sm.vc = en + C::E.off_vc;
      sm.ks = reinterpret_cast<const __half*>(en + C::E.off_ks);
      sm.kz = reinterpret_cast<const __half*>(en + C::E.off_kz);
      sm.vs = reinterpret_cast<const __half*>(en + C::E.off_vs);
      sm.vz = reinterpret_cast<const __half*>(en + C::E.off_vz);
      // fed weights per (query, V group) combo, fp16: token-wise V P s 2^eP with max(s) 2^eP in
      // [2^6, 2^7) over the warp's valid tokens (fed values below 2^15); channel-wise V P * 32
      float fw[MC];
      float inv_ps = 1.f;
      if (VL == 0) {
        float sv[GV], zv[GV];
        uint32_t sb = 0;
        const bool ok = tk < nv;
#pragma unroll
        for (int uu = 0; uu < GV; ++uu) {
          const __half hs = sm.vs[tk * GV + uu], hz = sm.vz[tk * GV + uu];
          sv[uu] = ok ? __half2float(hs) : 0.f;
          zv[uu] = ok ? __half2float(hz) : 0.f;
          sb = max(sb, ok ? (uint32_t)(__half_as_ushort(hs) & 0x7fffu) : 0u);
        }
        sb = __reduce_max_sync(FULLMASK, sb);
        const float smaxf = __half2float(__ushort_as_half((unsigned short)sb));
        int e2 = 0;
        if (smaxf > 0.f) e2 = min(100, max(-100, 6 - ilog2f(smaxf)));
        const float ps = exp2i(e2);
        inv_ps = exp2i(-e2);
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
      // this token's row of fed weights: column n of PV n-tile v holds combo DUP ? n / 2 : 8 v + n
      {
        uint32_t rw[NTV * 4];
#pragma unroll
        for (int j = 0; j < NTV * 4; ++j) {
          if (C::DUP) {
            rw[j] = f16x2_from(fw[j], fw[j]);
          } else {
            rw[j] = f16x2_from(fw[2 * j], fw[2 * j + 1]);
          }
        }
#pragma unroll
        for (int v = 0; v < NTV; ++v)
          *reinterpret_cast<uint4*>(ptile + lane * C::P_ROW + 16 * v) =
              make_uint4(rw[4 * v], rw[4 * v + 1], rw[4 * v + 2], rw[4 * v + 3]);
      }
      __syncwarp();
      uint32_t pB[NTV][2][2];
#pragma unroll
      for (int v = 0; v < NTV; ++v)
        ldsm_x4_trans(smem_addr(ptile + lane * C::P_ROW + 16 * v), pB[v][0][0], pB[v][0][1], pB[v][1][0],
                      pB[v][1][1]);
      // minus the magic bias of each PV accumulator column: 1024 times the sum of the fp16 weights
      // fed to it, formed by the tensor cores with an all-ones A operand
      float cb[NTV][2], fsum[NTV][2];
      {
        constexpr uint32_t kOnes2 = 0x3c003c00u;
#pragma unroll
        for (int v = 0; v < NTV; ++v) {
          float fs[4];
          mma_f16_c(fs, kOnes2, kOnes2, kOnes2, kOnes2, pB[v][0][0], pB[v][0][1], 0.f, 0.f, 0.f, 0.f);
          mma_f16(fs, kOnes2, kOnes2, kOnes2, kOnes2, pB[v][1][0], pB[v][1][1]);
          cb[v][0] = -kMagicF * fs[0];
          cb[v][1] = -kMagicF * fs[1];
          fsum[v][0] = fs[0];
          fsum[v][1] = fs[1];
        }
      }
      float accv[8][NTV][4];
      pv_chunk<C>(accv, pB, sm, 32 * quad, lc, true, cb);
      if (VL == 0) {
        fold_tokenwise_v<C>(st, accv, inv_ps, lc);
      } else {
        float Wg[NO];
#pragma unroll
        for (int o = 0; o < NO; ++o) Wg[o] = fsum[0][C::DUP ? 0 : (o & 1)];
        const int tau = (32 * quad) / C::G;
        fold_channelwise_v<C, FED_CW>(st, accv, Wg, sm.vs + tau * D, sm.vz + tau * D, lc);
      }
      __syncwarp();  // the weight tile is read before the next item writes it
    };

    // -------------------------------------------------- the group's items of this segment
    if (cv.i < NL && cv.u == u) {
      uint32_t ksz_cur[GK], ksz_nx[GK];
      convert(cv, cv_r, cv_ph, cv_pos & 1, ksz_cur);
      group_barrier(grp);
      gf = gfail[grp] != 0;
      issue_qk(cv_pos & 1);
      if (leader && !gf && !failed && kis.i < NL) {  // the converted entry's K half is free
        copy_half(false, kis, kis_r);
        advance(kis, NG);
        ++kis_pos;
        if (++kis_r == R) kis_r = 0;
      }
      advance(cv, NG);
      ++cv_pos;
      if (++cv_r == R) cv_r = 0, cv_ph ^= 1u;
      for (; con.i < NL && con.u == u; advance(con, NG), ++con_pos, con_r = (con_r + 1 == R) ? 0 : con_r + 1,
                                        con_ph ^= (con_r == 0) ? 1u : 0u) {
        const bool has_next = cv.i < NL && cv.u == u;
        if (has_next) {
          convert(cv, cv_r, cv_ph, cv_pos & 1, ksz_nx);
          group_barrier(grp);
          gf = gfail[grp] != 0;
          issue_qk(cv_pos & 1);
          if (leader && !gf && !failed && kis.i < NL) {
            copy_half(false, kis, kis_r);
            advance(kis, NG);
            ++kis_pos;
            if (++kis_r == R) kis_r = 0;
          }
          advance(cv, NG);
          ++cv_pos;
          if (++cv_r == R) cv_r = 0, cv_ph ^= 1u;
        }
        consume(con, con_pos, con_r, con_ph, ksz_cur);
        group_barrier(grp);  // every warp is done with the item's V half and its scores
        gf = gfail[grp] != 0;
        if (leader && !gf && !failed && vis.i < NL) {
          copy_half(true, vis, vis_r);
          advance(vis, NG);
          ++vis_pos;
          if (++vis_r == R) vis_r = 0;
        }
        if (has_next) {
#pragma unroll
          for (int cc = 0; cc < GK; ++cc) ksz_cur[cc] = ksz_nx[cc];
        }
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
        st.pa[j] = 1.f;
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
    if (C::WARPS > kMergeWarps) {
      constexpr int SF = 16 * NQ + NO + 2 * NQ;
      static_assert(SF <= kStateFloats, "handed-over state fits the merge area");
      float* xsa = ma.m;
      __syncthreads();
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
    } else {
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
  // After a wait gave up: every bulk copy issued and every product committed must have
  // completed before shared and tensor memory are released (bounded waits).
  // Once a wait gave up no entry is refilled, so each entry has at most its last issued
  // copy outstanding: waiting for that phase (already complete when it was consumed) drains it.
  if (leader && (gf || failed || gfail[grp])) {
    for (int j = max(0, kis_pos - R); j < kis_pos; ++j)
      if (!mbar_wait(kbar(j % R), (uint32_t)((j / R) & 1), p.status, kStatusDrainTimeout)) break;
    for (int j = max(0, vis_pos - R); j < vis_pos; ++j)
      if (!mbar_wait(vbar(j % R), (uint32_t)((j / R) & 1), p.status, kStatusDrainTimeout)) break;
    // the leader's products: commit k went to buffer k & 1 as its (k >> 1)-th completion
    for (int k2 = max(0, n_commit - 2); k2 < n_commit; ++k2)
      if (!mbar_wait(sbar(k2 & 1), (uint32_t)((k2 >> 1) & 1), p.status, kStatusDrainTimeout)) break;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::dealloc(s_tmem, C::TMC);
}

}  // namespace lbkv
