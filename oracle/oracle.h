/*
 * oracle.h -- interface of the fp64 CPU oracle (test infrastructure only).
 *
 * This header belongs to the oracle alone: the CUDA library neither includes
 * it nor shares any type or constant with it.
 *
 * Layouts (all arrays dense, row-major, host memory):
 *   q        bf16 bits  [B][Hq][D]
 *   *_codes  uint8      [B][Hkv][T_cap][D*bits/8], code i of a byte in bits
 *                       [bits*i, bits*i+bits), codes along head_dim
 *   token-wise  *_scale / *_off  fp16 bits [B][Hkv][T_cap][D/group]
 *   channel-wise *_scale / *_off fp16 bits [B][Hkv][T_cap/group][D]
 *   seq_lens int32 [B] (quantized tokens per sequence)
 *   k_win / v_win bf16 bits [B][Hkv][win_cap][D], win_lens int32 [B]
 *                       (optional full-precision window after the cached tokens)
 *   rotation   bit 0: the keys (cache and window) are stored rotated by the
 *              normalized Hadamard matrix H over head_dim, bit 1: the values are
 *              (see oracle_hadamard and decode_row_ref in oracle.c)
 */
#ifndef LBKV_ORACLE_H
#define LBKV_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_OK = 0, ORACLE_EINVAL = -1 };
enum { ORACLE_TOKENWISE = 0, ORACLE_CHANNELWISE = 1 };
enum { ORACLE_ACC_FOLD = 0, ORACLE_OPERAND_FOLD = 1 };
enum { ORACLE_ROTATE_K = 1, ORACLE_ROTATE_V = 2 };

typedef struct {
  int B, Hq, Hkv, D, T_cap, bits, k_layout, v_layout, group;
  double sm_scale; /* <= 0 selects 1/sqrt(D) */
  const uint16_t* q;
  const uint8_t* k_codes;
  const uint16_t* k_scale;
  const uint16_t* k_off;
  const uint8_t* v_codes;
  const uint16_t* v_scale;
  const uint16_t* v_off;
  const int32_t* seq_lens;
  const uint16_t* k_win; /* NULL: no window */
  const uint16_t* v_win;
  const int32_t* win_lens;
  int win_cap;
  int rotation; /* ORACLE_ROTATE_K | ORACLE_ROTATE_V, or 0 */
} oracle_decode_args;

double oracle_bf16_to_f64(uint16_t h);
double oracle_fp16_to_f64(uint16_t h);
uint16_t oracle_f64_to_fp16(double x);
int oracle_unpack_code(const uint8_t* row, int bits, int d);

/* Plain definition. rows: n_rows (b, h) pairs, or NULL for every row in
 * (b, h) order; out: [n_rows][D]. n_threads <= 0 uses every online core. */
int oracle_decode_ref(const oracle_decode_args* a, const int32_t* rows, int n_rows, int n_threads, double* out);

/* Folded path (see oracle.c); out: [B][Hq][D]; ops: [2]. */
int oracle_decode_folded(const oracle_decode_args* a, int block, int misorder, double* out, double* ops);

double oracle_weighted_dequant_sum(const double* w, const int* q, const double* s, const double* z, int n);
double oracle_acc_fold(const double* w, const int* q, int n, double s, double z);
double oracle_operand_fold(const double* w, const int* q, int n, const double* s, const double* z);
int oracle_fold_kind(int side, int layout);

/* Normalized Hadamard matrix of order n (a power of two), fp64: H[i][j] =
 * (-1)^popcount(i & j) / sqrt(n); out: [n][n]. */
int oracle_hadamard(int n, double* out);

/* Rotation of bf16 rows of n channels (n a power of two) as stored: the
 * Walsh-Hadamard butterflies in IEEE single precision, scaled by
 * fp32(1/sqrt(n)); y32 receives the fp32 results ([rows][n], may be NULL),
 * y16 their bf16 roundings (nearest, ties to even; may be NULL). */
int oracle_rotate_rows(const uint16_t* x, size_t rows, int n, float* y32, uint16_t* y16);

int oracle_pack(int B, int Hkv, int D, int T_cap, int bits, int layout, int group, const uint16_t* x,
                const int32_t* seq_lens, uint8_t* codes, uint16_t* scale, uint16_t* off);

#ifdef __cplusplus
}
#endif
#endif
