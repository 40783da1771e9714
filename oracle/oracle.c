/*
 * oracle.c -- plain, slow fp64 CPU oracle for decode attention over a 2-/4-bit
 * affine-quantized KV cache.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE. Only the test suite, the smoke check
 * and the benchmark's CPU-baseline leg load this file's shared object. It
 * shares no source, header, table or helper with the CUDA library; the two are
 * compared against each other, so they must stay independent.
 *
 * Sources (cited by page title and part):
 *  [ABS] "FOSCAR: Accelerating Decode Attention over 2- and 4-Bit KV Caches
 *        through Affine Folding" (arXiv:2611.09722), abstract.
 *  [EXP] "FOSCAR speeds up 2-bit KV decode -- Affine folding of KV
 *        dequantization" (learnaivisually.com explainer): the receipt
 *        paragraph, the quantization-format paragraph, the fold-rule
 *        paragraph, the fold table, the instruction-budget paragraph and the
 *        accuracy/break-even paragraph.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - a code q is an unsigned b-bit integer and the stored value is s*q + z
 *    with z an additive offset ([EXP] quantization-format paragraph);
 *  - codes are packed along head_dim, code i of a byte in bits [b*i, b*i+b);
 *  - query head h reads KV head h / (Hq/Hkv);
 *  - a sequence with no tokens yields an all-zero output row;
 *  - the quantizer is min/max per group with round-to-nearest-even;
 *  - the rotation that [EXP] names as an accuracy recipe (OSCAR's rotations;
 *    the related "KVarN -- Hadamard-rotated 2-bit KV cache" explainer) is the
 *    normalized Hadamard matrix of order head_dim applied to each stored key
 *    and/or value row; attention over rotated keys takes the query rotated by
 *    the same matrix, and the output over rotated values is rotated back by it
 *    (H is symmetric and orthogonal, so H^-1 = H);
 *  - a row is rotated as stored in IEEE single precision by the Walsh-Hadamard
 *    butterflies (stages of span 1, 2, 4, ...; the lower index takes a + b, the
 *    upper a - b), scaled by fp32(1/sqrt(n)) and rounded to bf16.
 *
 * Parity status of every exported function is pinned by tests under tests/
 * (golden fixtures, closed forms, library routines, brute force); none is
 * "parity unpinned".
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#include "oracle.h"

/* ------------------------------------------------------------------ */
/* Number formats, written from the IEEE-754 binary16 and bfloat16     */
/* definitions.                                                        */
/* ------------------------------------------------------------------ */

double oracle_bf16_to_f64(uint16_t h) {
  /* bfloat16 is the top half of an IEEE single. */
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

double oracle_fp16_to_f64(uint16_t h) {
  /* binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
  int sign = h >> 15;
  int e = (h >> 10) & 31;
  int m = h & 1023;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
  return sign ? -v : v;
}

/* Nearest binary16 to a finite or infinite double that is itself an exact
 * float, ties to even (nearbyint runs in the default round-to-nearest-even
 * mode; every scaling below is by a power of two and therefore exact). */
uint16_t oracle_f64_to_fp16(double x) {
  uint16_t sign = (signbit(x) ? 0x8000 : 0);
  double a = fabs(x);
  if (isnan(x)) return 0x7e00;
  if (a >= 65520.0) return sign | 0x7c00; /* 65520 ties to the even 2^16 -> inf */
  if (a < ldexp(1.0, -14)) {
    double q = nearbyint(ldexp(a, 24)); /* subnormal step 2^-24 */
    return sign | (uint16_t)q;          /* q == 1024 encodes the least normal */
  }
  int ex;
  frexp(a, &ex); /* a = f * 2^ex, f in [0.5, 1) */
  int E = ex - 1;
  double q = nearbyint(ldexp(a, 10 - E)); /* in [1024, 2048] */
  if (q == 2048.0) {
    q = 1024.0;
    E += 1;
  }
  if (E + 15 >= 31) return sign | 0x7c00;
  return sign | (uint16_t)(((E + 15) << 10) | ((int)q - 1024));
}

/* ------------------------------------------------------------------ */
/* Code unpacking: code i of a byte sits in bits [b*i, b*i+b), and     */
/* codes run along head_dim.                                           */
/* ------------------------------------------------------------------ */

int oracle_unpack_code(const uint8_t* row, int bits, int d) {
  int per_byte = 8 / bits;
  int byte = d / per_byte;
  int shift = bits * (d % per_byte);
  return (row[byte] >> shift) & ((1 << bits) - 1);
}

/* ------------------------------------------------------------------ */
/* Shared argument checks and indexing                                 */
/* ------------------------------------------------------------------ */

static int check_args(const oracle_decode_args* a) {
  if (a->B < 0 || a->Hq <= 0 || a->Hkv <= 0 || a->D <= 0 || a->T_cap < 0) return ORACLE_EINVAL;
  if (a->Hq % a->Hkv) return ORACLE_EINVAL;
  if (a->bits != 2 && a->bits != 4) return ORACLE_EINVAL;
  if (a->group <= 0) return ORACLE_EINVAL;
  if ((a->D * a->bits) % 8) return ORACLE_EINVAL;
  for (int side = 0; side < 2; ++side) {
    int lay = side ? a->v_layout : a->k_layout;
    if (lay == ORACLE_TOKENWISE) {
      if (a->D % a->group) return ORACLE_EINVAL;
    } else if (lay == ORACLE_CHANNELWISE) {
      if (a->T_cap % a->group) return ORACLE_EINVAL;
    } else {
      return ORACLE_EINVAL;
    }
  }
  for (int b = 0; b < a->B; ++b) {
    if (a->seq_lens[b] < 0 || a->seq_lens[b] > a->T_cap) return ORACLE_EINVAL;
    if (a->win_lens && (a->win_lens[b] < 0 || a->win_lens[b] > a->win_cap)) return ORACLE_EINVAL;
  }
  if (a->rotation & ~(ORACLE_ROTATE_K | ORACLE_ROTATE_V)) return ORACLE_EINVAL;
  if (a->rotation && (a->D & (a->D - 1))) return ORACLE_EINVAL;
  return ORACLE_OK;
}

/* Index of the (s, z) pair that covers cached value (t, d) of (b, kv). */
static size_t sz_index(const oracle_decode_args* a, int layout, int b, int kv, int t, int d) {
  size_t unit = (size_t)b * a->Hkv + kv;
  if (layout == ORACLE_TOKENWISE) {
    int groups = a->D / a->group; /* D/g pairs per token, along channels */
    return (unit * a->T_cap + t) * groups + d / a->group;
  }
  /* channel-wise: one pair per channel per block of g tokens */
  int blocks = a->T_cap / a->group;
  return (unit * blocks + t / a->group) * a->D + d;
}

static const uint8_t* code_row(const oracle_decode_args* a, const uint8_t* codes, int b, int kv, int t) {
  size_t row_bytes = (size_t)a->D * a->bits / 8;
  return codes + (((size_t)b * a->Hkv + kv) * a->T_cap + t) * row_bytes;
}

/* Dequantized cached value s*q + z ([EXP] quantization-format paragraph). */
static double dequant(const oracle_decode_args* a, int side, int b, int kv, int t, int d) {
  const uint8_t* codes = side ? a->v_codes : a->k_codes;
  const uint16_t* sc = side ? a->v_scale : a->k_scale;
  const uint16_t* of = side ? a->v_off : a->k_off;
  int layout = side ? a->v_layout : a->k_layout;
  int q = oracle_unpack_code(code_row(a, codes, b, kv, t), a->bits, d);
  size_t i = sz_index(a, layout, b, kv, t, d);
  return oracle_fp16_to_f64(sc[i]) * (double)q + oracle_fp16_to_f64(of[i]);
}

static double window_value(const oracle_decode_args* a, const uint16_t* win, int b, int kv, int w, int d) {
  return oracle_bf16_to_f64(win[((((size_t)b * a->Hkv + kv) * a->win_cap) + w) * a->D + d]);
}

static double scale_of(const oracle_decode_args* a) {
  return a->sm_scale > 0.0 ? a->sm_scale : 1.0 / sqrt((double)a->D);
}

/* ------------------------------------------------------------------ */
/* Plain definition: dequantize every value, textbook softmax attention */
/* ([ABS]: the folded kernel preserves the dequantized attention output */
/* in exact arithmetic, so this is what it must reproduce).             */
/* ------------------------------------------------------------------ */

static int popcount_u32(unsigned x) {
  int c = 0;
  for (; x; x &= x - 1) ++c;
  return c;
}

int oracle_hadamard(int n, double* out) {
  if (n <= 0 || (n & (n - 1))) return ORACLE_EINVAL;
  double inv = 1.0 / sqrt((double)n);
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < n; ++j) out[(size_t)i * n + j] = (popcount_u32((unsigned)(i & j)) & 1) ? -inv : inv;
  return ORACLE_OK;
}

/* y <- H y (fp64, n x n matrix product). */
static void hadamard_apply(double* y, int n) {
  double* H = (double*)malloc(sizeof(double) * n * n);
  double* t = (double*)malloc(sizeof(double) * n);
  oracle_hadamard(n, H);
  for (int i = 0; i < n; ++i) {
    double acc = 0.0;
    for (int j = 0; j < n; ++j) acc += H[(size_t)i * n + j] * y[j];
    t[i] = acc;
  }
  for (int i = 0; i < n; ++i) y[i] = t[i];
  free(H);
  free(t);
}

static void decode_row_ref(const oracle_decode_args* a, int b, int h, double* out) {
  int hq = a->Hq / a->Hkv;
  int kv = h / hq;
  int L = a->seq_lens[b];
  int W = a->win_lens ? a->win_lens[b] : 0;
  int n = L + W;
  int D = a->D;
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  if (n == 0) return;

  double* Q = (double*)malloc(sizeof(double) * D);
  double* S = (double*)malloc(sizeof(double) * n);
  for (int d = 0; d < D; ++d) Q[d] = oracle_bf16_to_f64(a->q[((size_t)b * a->Hq + h) * D + d]);
  /* keys stored as H k: q . k = (H q) . (H k) */
  if (a->rotation & ORACLE_ROTATE_K) hadamard_apply(Q, D);
  double sigma = scale_of(a);

  /* 1-3: unpack, dequantize, score. Window tokens follow the cached ones. */
  for (int t = 0; t < n; ++t) {
    double acc = 0.0;
    for (int d = 0; d < D; ++d) {
      double k = t < L ? dequant(a, 0, b, kv, t, d) : window_value(a, a->k_win, b, kv, t - L, d);
      acc += Q[d] * k;
    }
    S[t] = sigma * acc;
  }
  /* 4: softmax with the maximum subtracted. */
  double M = S[0];
  for (int t = 1; t < n; ++t)
    if (S[t] > M) M = S[t];
  double l = 0.0;
  for (int t = 0; t < n; ++t) {
    S[t] = exp(S[t] - M);
    l += S[t];
  }
  /* 5: weighted sum of dequantized values, divided by the denominator. */
  for (int t = 0; t < n; ++t) {
    double p = S[t];
    for (int d = 0; d < D; ++d) {
      double v = t < L ? dequant(a, 1, b, kv, t, d) : window_value(a, a->v_win, b, kv, t - L, d);
      out[d] += p * v;
    }
  }
  for (int d = 0; d < D; ++d) out[d] /= l;
  /* values stored as H v: sum_t p_t v_t = H (sum_t p_t H v_t) */
  if (a->rotation & ORACLE_ROTATE_V) hadamard_apply(out, D);
  free(Q);
  free(S);
}

typedef struct {
  const oracle_decode_args* a;
  const int32_t* rows;
  int n_rows;
  int tid, nthreads;
  double* out;
} row_job;

static void* row_worker(void* p) {
  row_job* j = (row_job*)p;
  for (int r = j->tid; r < j->n_rows; r += j->nthreads) {
    int b, h;
    if (j->rows) {
      b = j->rows[2 * r];
      h = j->rows[2 * r + 1];
    } else {
      b = r / j->a->Hq;
      h = r % j->a->Hq;
    }
    decode_row_ref(j->a, b, h, j->out + (size_t)r * j->a->D);
  }
  return NULL;
}

int oracle_decode_ref(const oracle_decode_args* a, const int32_t* rows, int n_rows, int n_threads, double* out) {
  int st = check_args(a);
  if (st) return st;
  if (!rows) n_rows = a->B * a->Hq;
  for (int r = 0; rows && r < n_rows; ++r)
    if (rows[2 * r] < 0 || rows[2 * r] >= a->B || rows[2 * r + 1] < 0 || rows[2 * r + 1] >= a->Hq) return ORACLE_EINVAL;
  if (n_threads <= 0) n_threads = (int)sysconf(_SC_NPROCESSORS_ONLN);
  if (n_threads > n_rows) n_threads = n_rows > 0 ? n_rows : 1;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * n_threads);
  row_job* jobs = (row_job*)malloc(sizeof(row_job) * n_threads);
  for (int i = 0; i < n_threads; ++i) {
    jobs[i] = (row_job){a, rows, n_rows, i, n_threads, out};
    if (n_threads == 1)
      row_worker(&jobs[i]);
    else
      pthread_create(&th[i], NULL, row_worker, &jobs[i]);
  }
  if (n_threads > 1)
    for (int i = 0; i < n_threads; ++i) pthread_join(th[i], NULL);
  free(th);
  free(jobs);
  return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* The fold primitives ([EXP] receipt paragraph and fold rule).         */
/* ------------------------------------------------------------------ */

/* Unfolded: convert every code, then weight and sum. */
double oracle_weighted_dequant_sum(const double* w, const int* q, const double* s, const double* z, int n) {
  double acc = 0.0;
  for (int i = 0; i < n; ++i) acc += w[i] * (s[i] * q[i] + z[i]);
  return acc;
}

/* acc-fold: one scale and one offset shared along the summed axis; the raw
 * weighted sum of codes is scaled once and the offset times the weight sum
 * is added once. */
double oracle_acc_fold(const double* w, const int* q, int n, double s, double z) {
  double raw = 0.0, wsum = 0.0;
  for (int i = 0; i < n; ++i) {
    raw += w[i] * q[i];
    wsum += w[i];
  }
  return s * raw + z * wsum;
}

/* operand-fold: the scale changes along the summed axis, so each weight is
 * pre-multiplied by its line's scale; the offsets become one extra term. */
double oracle_operand_fold(const double* w, const int* q, int n, const double* s, const double* z) {
  double acc = 0.0, off = 0.0;
  for (int i = 0; i < n; ++i) {
    acc += (w[i] * s[i]) * q[i];
    off += w[i] * z[i];
  }
  return acc + off;
}

/* Which fold the fold table assigns to a (side, layout) pair:
 * token-wise K -> acc, channel-wise K -> operand, token-wise V -> operand,
 * channel-wise V -> acc ([EXP] fold table). The rule behind it: acc-fold when
 * the group's scale is constant along the summed axis, operand-fold when it
 * changes along it. QK^T sums over channels and PV sums over tokens. */
int oracle_fold_kind(int side, int layout) {
  int sums_over_channels = (side == 0);
  int group_runs_along_channels = (layout == ORACLE_TOKENWISE);
  /* scale constant along the summed axis <=> the group runs along it */
  return (sums_over_channels == group_runs_along_channels) ? ORACLE_ACC_FOLD : ORACLE_OPERAND_FOLD;
}

/* ------------------------------------------------------------------ */
/* Folded decode: the four fold formulas applied literally inside an    */
/* online (FlashAttention) softmax, with the ordering rules: key-side   */
/* corrections land before the softmax, value-side corrections before   */
/* the final division by the denominator ([EXP] fold rule, fold table). */
/* `block` is the number of tokens per online-softmax step; with a      */
/* channel-wise layout it must be a multiple of the token group.        */
/* `misorder` plants one of two ordering mistakes for negative tests:   */
/*   1 = the key offset term reaches the scores only after the softmax  */
/*       weights are formed (so the weights never see it);              */
/*   2 = the value offset term is added after the division by l.        */
/* ops[0] counts scale/offset applications over every query head, ops[1] */
/* the stored quantized K and V values, each counted once per KV head    */
/* ([EXP] instruction-budget paragraph: operations per stored value).   */
/* ------------------------------------------------------------------ */

static void decode_row_folded(const oracle_decode_args* a, int b, int h, int block, int misorder, double* out,
                              double* ops) {
  const int D = a->D, g = a->group;
  int hq = a->Hq / a->Hkv;
  int kv = h / hq;
  int L = a->seq_lens[b];
  int W = a->win_lens ? a->win_lens[b] : 0;
  double sigma = scale_of(a);
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  if (L + W == 0) return;

  double* Q = (double*)malloc(sizeof(double) * D);
  for (int d = 0; d < D; ++d) Q[d] = oracle_bf16_to_f64(a->q[((size_t)b * a->Hq + h) * D + d]);
  int nK = D / g; /* channel groups when the layout is token-wise */
  double* Qsum = (double*)calloc(nK > 0 ? nK : 1, sizeof(double));
  if (a->k_layout == ORACLE_TOKENWISE)
    for (int d = 0; d < D; ++d) Qsum[d / g] += Q[d];

  double* O = (double*)calloc(D, sizeof(double));      /* running sum of scaled/raw products */
  double* Zacc = (double*)calloc(D, sizeof(double));   /* running value-offset term */
  double* S = (double*)malloc(sizeof(double) * (block > 0 ? block : 1));
  double* Kfix = (double*)malloc(sizeof(double) * (block > 0 ? block : 1)); /* key offset per token */
  double* Qp = (double*)malloc(sizeof(double) * D);
  double m = -INFINITY, l = 0.0;

  for (int t0 = 0; t0 < L; t0 += block) {
    int t1 = t0 + block < L ? t0 + block : L;
    int nb = t1 - t0;
    /* ---- scores: K side ---- */
    for (int t = t0; t < t1; ++t) {
      double raw_total = 0.0, fix = 0.0;
      const uint8_t* row = code_row(a, a->k_codes, b, kv, t);
      if (a->k_layout == ORACLE_TOKENWISE) {
        /* acc-fold: each channel group's raw partial sum is scaled on its
         * own (an unscaled partial never crosses a group boundary), and
         * z times the sum of the query over that group is added. */
        for (int c = 0; c < nK; ++c) {
          double raw = 0.0;
          for (int d = c * g; d < (c + 1) * g; ++d) raw += Q[d] * oracle_unpack_code(row, a->bits, d);
          size_t i = sz_index(a, ORACLE_TOKENWISE, b, kv, t, c * g);
          double s = oracle_fp16_to_f64(a->k_scale[i]), z = oracle_fp16_to_f64(a->k_off[i]);
          raw_total += s * raw;
          fix += z * Qsum[c];
          ops[0] += 2;
        }
      } else {
        /* operand-fold: the query is multiplied by the scale of the token
         * group before the product; the offset becomes sum_d Q_d z_d, one
         * constant per (query, token group). */
        int tau = t / g;
        if (t == t0 || t % g == 0) {
          for (int d = 0; d < D; ++d) {
            size_t i = sz_index(a, ORACLE_CHANNELWISE, b, kv, t, d);
            Qp[d] = Q[d] * oracle_fp16_to_f64(a->k_scale[i]);
            ops[0] += 1;
          }
          (void)tau;
        }
        for (int d = 0; d < D; ++d) raw_total += Qp[d] * oracle_unpack_code(row, a->bits, d);
        if (t == t0 || t % g == 0) {
          double off = 0.0;
          for (int d = 0; d < D; ++d) {
            size_t i = sz_index(a, ORACLE_CHANNELWISE, b, kv, t, d);
            off += Q[d] * oracle_fp16_to_f64(a->k_off[i]);
            ops[0] += 1;
          }
          Kfix[0] = off; /* reused for the rest of the token group */
        }
        fix = Kfix[0];
      }
      S[t - t0] = sigma * (raw_total + (misorder == 1 ? 0.0 : fix));
      if (h % hq == 0) ops[1] += D; /* stored values are shared by the h_q query heads */
    }
    /* ---- online softmax (unchanged FlashAttention step) ---- */
    double mb = m;
    for (int j = 0; j < nb; ++j)
      if (S[j] > mb) mb = S[j];
    double alpha = (m == -INFINITY) ? 0.0 : exp(m - mb);
    for (int d = 0; d < D; ++d) {
      O[d] *= alpha;
      Zacc[d] *= alpha;
    }
    l *= alpha;
    m = mb;
    for (int j = 0; j < nb; ++j) {
      S[j] = exp(S[j] - m);
      l += S[j];
    }
    /* ---- PV: V side ---- */
    if (a->v_layout == ORACLE_TOKENWISE) {
      /* operand-fold: P' = P * s of each token's channel group; the offset
       * becomes sum_t P_t z_t per channel group. */
      for (int t = t0; t < t1; ++t) {
        const uint8_t* row = code_row(a, a->v_codes, b, kv, t);
        double p = S[t - t0];
        for (int c = 0; c < D / g; ++c) {
          size_t i = sz_index(a, ORACLE_TOKENWISE, b, kv, t, c * g);
          double pp = p * oracle_fp16_to_f64(a->v_scale[i]);
          double pz = p * oracle_fp16_to_f64(a->v_off[i]);
          ops[0] += 2;
          for (int d = c * g; d < (c + 1) * g; ++d) {
            O[d] += pp * oracle_unpack_code(row, a->bits, d);
            Zacc[d] += pz;
          }
        }
        if (h % hq == 0) ops[1] += D;
      }
    } else {
      /* acc-fold: within one token group the raw partial sum_t P_t q_td is
       * scaled by s_d once, and z_d times sum_t P_t is added once; the
       * partial never crosses a token-group boundary. */
      for (int u0 = t0; u0 < t1;) {
        int u1 = (u0 / g + 1) * g;
        if (u1 > t1) u1 = t1;
        double psum = 0.0;
        for (int t = u0; t < u1; ++t) psum += S[t - t0];
        for (int d = 0; d < D; ++d) {
          double raw = 0.0;
          for (int t = u0; t < u1; ++t)
            raw += S[t - t0] * oracle_unpack_code(code_row(a, a->v_codes, b, kv, t), a->bits, d);
          size_t i = sz_index(a, ORACLE_CHANNELWISE, b, kv, u0, d);
          O[d] += oracle_fp16_to_f64(a->v_scale[i]) * raw;
          Zacc[d] += oracle_fp16_to_f64(a->v_off[i]) * psum;
          ops[0] += 2;
        }
        if (h % hq == 0) ops[1] += (double)(u1 - u0) * D;
        u0 = u1;
      }
    }
  }

  /* Full-precision window tokens: one more plain online-softmax step. */
  if (W > 0) {
    double* Sw = (double*)malloc(sizeof(double) * W);
    double mb = m;
    for (int w = 0; w < W; ++w) {
      double acc = 0.0;
      for (int d = 0; d < D; ++d) acc += Q[d] * window_value(a, a->k_win, b, kv, w, d);
      Sw[w] = sigma * acc;
      if (Sw[w] > mb) mb = Sw[w];
    }
    double alpha = (m == -INFINITY) ? 0.0 : exp(m - mb);
    for (int d = 0; d < D; ++d) {
      O[d] *= alpha;
      Zacc[d] *= alpha;
    }
    l *= alpha;
    m = mb;
    for (int w = 0; w < W; ++w) {
      double p = exp(Sw[w] - m);
      l += p;
      for (int d = 0; d < D; ++d) O[d] += p * window_value(a, a->v_win, b, kv, w, d);
    }
    free(Sw);
  }

  /* Value-side corrections land before the final division by l. */
  for (int d = 0; d < D; ++d) out[d] = (misorder == 2) ? O[d] / l + Zacc[d] : (O[d] + Zacc[d]) / l;

  free(Q);
  free(Qsum);
  free(O);
  free(Zacc);
  free(S);
  free(Kfix);
  free(Qp);
}

int oracle_decode_folded(const oracle_decode_args* a, int block, int misorder, double* out, double* ops) {
  int st = check_args(a);
  if (st) return st;
  if (block <= 0 || a->rotation) return ORACLE_EINVAL;
  if ((a->k_layout == ORACLE_CHANNELWISE || a->v_layout == ORACLE_CHANNELWISE) && block % a->group) return ORACLE_EINVAL;
  ops[0] = ops[1] = 0.0;
  for (int b = 0; b < a->B; ++b)
    for (int h = 0; h < a->Hq; ++h) decode_row_folded(a, b, h, block, misorder, out + ((size_t)b * a->Hq + h) * a->D, ops);
  return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* Quantizer (min/max per group, round-to-nearest-even), in IEEE single */
/* precision with every operation rounded on its own (built without     */
/* FMA contraction):                                                   */
/*   s = fp16((max - min) / (2^b - 1)),  z = fp16(min),                 */
/*   q = clamp(rne((x - z) / s), 0, 2^b - 1), q = 0 when s == 0.         */
/* Padding tokens (t >= seq_len) get code 0; their s and z are left as  */
/* they were.                                                          */
/* ------------------------------------------------------------------ */

static float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* bf16 rounding of an fp32 value: nearest, ties to even; NaN stays NaN. */
static uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t lsb = (u >> 16) & 1u;
  return (uint16_t)((u + 0x7fffu + lsb) >> 16);
}

int oracle_rotate_rows(const uint16_t* x, size_t rows, int n, float* y32, uint16_t* y16) {
  if (n <= 0 || (n & (n - 1))) return ORACLE_EINVAL;
  volatile float c = (float)(1.0 / sqrt((double)n));
  float* y = (float*)malloc(sizeof(float) * n);
  for (size_t r = 0; r < rows; ++r) {
    for (int i = 0; i < n; ++i) y[i] = bf16_to_f32(x[r * n + i]);
    for (int span = 1; span < n; span <<= 1)
      for (int i = 0; i < n; ++i) {
        if (i & span) continue;
        volatile float lo = y[i], hi = y[i + span];
        volatile float s = lo + hi, d = lo - hi;
        y[i] = s;
        y[i + span] = d;
      }
    for (int i = 0; i < n; ++i) {
      volatile float v = y[i] * c;
      if (y32) y32[r * n + i] = v;
      if (y16) y16[r * n + i] = f32_to_bf16(v);
    }
  }
  free(y);
  return ORACLE_OK;
}

static void quantize_group(const float* x, int n, int bits, uint16_t* s_out, uint16_t* z_out, int* q_out) {
  float mn = x[0], mx = x[0];
  for (int i = 1; i < n; ++i) {
    if (x[i] < mn) mn = x[i];
    if (x[i] > mx) mx = x[i];
  }
  /* a signed zero extreme is read as +0 (x + 0 maps -0 to +0 and keeps every
   * other value), so that s and z never carry a negative zero */
  mn = mn + 0.0f;
  mx = mx + 0.0f;
  volatile float range = mx - mn;
  volatile float step = range / (float)((1 << bits) - 1);
  uint16_t sh = oracle_f64_to_fp16((double)step);
  uint16_t zh = oracle_f64_to_fp16((double)mn);
  float sf = (float)oracle_fp16_to_f64(sh);
  float zf = (float)oracle_fp16_to_f64(zh);
  int qmax = (1 << bits) - 1;
  for (int i = 0; i < n; ++i) {
    if (sf == 0.0f) {
      q_out[i] = 0;
      continue;
    }
    volatile float diff = x[i] - zf;
    volatile float v = diff / sf;
    float r = nearbyintf(v);
    int q = (r < 0.0f) ? 0 : (r > (float)qmax ? qmax : (int)r);
    q_out[i] = q;
  }
  *s_out = sh;
  *z_out = zh;
}

static void put_code(uint8_t* row, int bits, int d, int q) {
  int per_byte = 8 / bits;
  row[d / per_byte] |= (uint8_t)(q << (bits * (d % per_byte)));
}

int oracle_pack(int B, int Hkv, int D, int T_cap, int bits, int layout, int group, const uint16_t* x,
                const int32_t* seq_lens, uint8_t* codes, uint16_t* scale, uint16_t* off) {
  if (B < 0 || Hkv <= 0 || D <= 0 || T_cap < 0 || group <= 0) return ORACLE_EINVAL;
  if (bits != 2 && bits != 4) return ORACLE_EINVAL;
  if ((D * bits) % 8) return ORACLE_EINVAL;
  if (layout == ORACLE_TOKENWISE && D % group) return ORACLE_EINVAL;
  if (layout == ORACLE_CHANNELWISE && T_cap % group) return ORACLE_EINVAL;
  if (layout != ORACLE_TOKENWISE && layout != ORACLE_CHANNELWISE) return ORACLE_EINVAL;
  for (int b = 0; b < B; ++b)
    if (seq_lens[b] < 0 || seq_lens[b] > T_cap) return ORACLE_EINVAL;

  size_t row_bytes = (size_t)D * bits / 8;
  float* buf = (float*)malloc(sizeof(float) * (group > 0 ? group : 1));
  int* qs = (int*)malloc(sizeof(int) * (group > 0 ? group : 1));
  for (int b = 0; b < B; ++b) {
    int L = seq_lens[b];
    for (int kv = 0; kv < Hkv; ++kv) {
      size_t unit = (size_t)b * Hkv + kv;
      uint8_t* ucodes = codes + unit * T_cap * row_bytes;
      memset(ucodes, 0, (size_t)T_cap * row_bytes);
      const uint16_t* ux = x + unit * T_cap * D;
      if (layout == ORACLE_TOKENWISE) {
        /* group = g consecutive channels of one token */
        int groups = D / group;
        for (int t = 0; t < L; ++t) {
          for (int c = 0; c < groups; ++c) {
            for (int j = 0; j < group; ++j) buf[j] = bf16_to_f32(ux[(size_t)t * D + c * group + j]);
            size_t si = (unit * T_cap + t) * groups + c;
            quantize_group(buf, group, bits, &scale[si], &off[si], qs);
            for (int j = 0; j < group; ++j) put_code(ucodes + (size_t)t * row_bytes, bits, c * group + j, qs[j]);
          }
        }
      } else {
        /* group = g consecutive tokens of one channel; the last group
         * covers only the valid tokens. */
        int blocks = T_cap / group;
        for (int tau = 0; tau * group < L; ++tau) {
          int t0 = tau * group;
          int n = (t0 + group <= L) ? group : L - t0;
          for (int d = 0; d < D; ++d) {
            for (int j = 0; j < n; ++j) buf[j] = bf16_to_f32(ux[(size_t)(t0 + j) * D + d]);
            size_t si = (unit * blocks + tau) * D + d;
            quantize_group(buf, n, bits, &scale[si], &off[si], qs);
            for (int j = 0; j < n; ++j) put_code(ucodes + (size_t)(t0 + j) * row_bytes, bits, d, qs[j]);
          }
        }
      }
    }
  }
  free(buf);
  free(qs);
  return ORACLE_OK;
}
