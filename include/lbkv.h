/*
 * lbkv.h -- C ABI of a GB300 (sm_103a) library for single-token decode
 * attention read directly from a 2- or 4-bit affine-quantized KV cache.
 *
 * What it computes. For every sequence b and query head h (KV head
 * kv = h / (Hq / Hkv)) over the L_b cached tokens, optionally followed by a
 * window of full-precision bf16 tokens:
 *     out[b][h] = sum_t softmax_t(sigma * Q[b][h] . K_t) * V_t
 * where every cached value is s * q + z: an unsigned b-bit code q sharing one
 * fp16 scale s and one fp16 offset z with its group ("FOSCAR speeds up 2-bit
 * KV decode -- Affine folding of KV dequantization", quantization-format
 * paragraph). The library never materialises s * q + z: following the fold
 * rule and fold table of that explainer (and the abstract of "FOSCAR:
 * Accelerating Decode Attention over 2- and 4-Bit KV Caches through Affine
 * Folding", arXiv:2611.09722), it applies s and z once per group, either to a
 * partial result (acc-fold: token-wise K, channel-wise V) or to the other
 * operand (operand-fold: channel-wise K, token-wise V); key corrections land
 * before the softmax and value corrections before the final division.
 *
 * Layout (all device memory, dense, row-major, owned by the caller):
 *   q          bf16  [B][Hq][D]
 *   k_codes    uint8 [B][Hkv][T_cap][D*bits/8]   (same for v_codes)
 *              code i of a byte sits in bits [bits*i, bits*i + bits);
 *              codes run along head_dim (channel d is code d of its row)
 *   token-wise scale/offset   fp16 [B][Hkv][T_cap][D/group]
 *              (one pair per token per group of `group` channels)
 *   channel-wise scale/offset fp16 [B][Hkv][T_cap/group][D]
 *              (one pair per channel per block of `group` tokens; a block
 *              that ends past L_b covers only the valid tokens)
 *   seq_lens   int32 [B], 0 <= L_b <= T_cap (tokens >= L_b are ignored)
 *   out        bf16  [B][Hq][D]
 *
 * Conventions shared by every entry point:
 *   - all pointers are device pointers, 16-byte aligned, owned by the caller;
 *     the library never allocates, frees or synchronizes (except
 *     lbkv_device_status, which is documented as synchronizing);
 *   - calls are asynchronous on `stream` (NULL = the legacy default stream);
 *   - arguments are validated before anything is launched; on a validation
 *     error nothing is written and a negative lbkv_status is returned;
 *   - a launch failure returns LBKV_ECUDA (cudaGetLastError after launch);
 *   - the calls are thread-safe (no global mutable state besides a per-device
 *     cache of the multiprocessor count).
 */
#ifndef LBKV_H
#define LBKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LBKV_API __attribute__((visibility("default")))
#else
#define LBKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Identical to cudaStream_t; declared here so that callers need no CUDA header. */
typedef struct CUstream_st* lbkv_stream_t;

/* Group orientation of a cache side ("FOSCAR speeds up 2-bit KV decode", fold table). */
typedef enum {
  LBKV_TOKENWISE = 0,   /* a group is `group` consecutive channels of one token */
  LBKV_CHANNELWISE = 1  /* a group is `group` consecutive tokens of one channel */
} lbkv_layout;

/* Rotated cache (lbkv_desc.rotation): the stored rows of a side were rotated over head_dim
 * by the normalized Hadamard matrix H, H[i][j] = (-1)^popcount(i & j) / sqrt(128), as an
 * accuracy recipe for 2-bit caches (OSCAR's rotations, accuracy paragraph of the explainer
 * "FOSCAR speeds up 2-bit KV decode"; the explainer "KVarN -- Hadamard-rotated 2-bit KV
 * cache"). H is symmetric and orthogonal, so decode folds it into the query (keys) and
 * the output (values): q . k = (H q) . (H k), and sum_t p_t v_t = H sum_t p_t (H v_t). */
typedef enum {
  LBKV_ROTATE_K = 1, /* keys stored as H k (cache and window) */
  LBKV_ROTATE_V = 2  /* values stored as H v (cache and window) */
} lbkv_rotation;

typedef enum {
  LBKV_OK = 0,
  LBKV_EINVAL = -1,        /* a null pointer, a bad size or an out-of-range argument */
  LBKV_EALIGN = -2,        /* a pointer that is not 16-byte aligned */
  LBKV_EUNSUPPORTED = -3,  /* valid but not implemented (see lbkv_decode_attn) */
  LBKV_EWORKSPACE = -4,    /* workspace missing or smaller than lbkv_workspace_bytes */
  LBKV_ECUDA = -5,         /* a CUDA launch or runtime call failed */
  LBKV_EDEVICE = -6,       /* a kernel reported a device-side error (lbkv_device_status) */
  LBKV_ESCRATCH = -7       /* lbkv_decode_attn_noalloc: the call needs more scratch than the
                              library's fixed array holds (lbkv_noalloc_scratch_bytes) */
} lbkv_status;

/* Shapes, scale, optional bf16 window and workspace of one decode call. */
typedef struct lbkv_desc {
  int32_t batch;         /* B >= 0 */
  int32_t num_q_heads;   /* Hq, a multiple of num_kv_heads */
  int32_t num_kv_heads;  /* Hkv >= 1; Hq / Hkv must be 1, 2, 4 or 8 */
  int32_t head_dim;      /* D; must be 128 */
  int32_t max_seq_len;   /* T_cap: token stride of codes and scales, a positive multiple of 128 */
  float sm_scale;        /* softmax scale sigma; <= 0 selects 1/sqrt(head_dim) */
  const void* k_win;     /* bf16 [B][Hkv][win_cap][D] tokens attended after the cached ones, or NULL */
  const void* v_win;     /* bf16 [B][Hkv][win_cap][D], NULL exactly when k_win is NULL */
  const int32_t* win_lens; /* int32 [B], 0 <= win_lens[b] <= win_cap; NULL when k_win is NULL */
  int32_t win_cap;       /* 1..128 when k_win is set */
  void* workspace;       /* device scratch of >= lbkv_workspace_bytes(...) bytes, 256-byte aligned,
                            zero-filled once after allocation: it holds the device status word,
                            one split counter per (sequence, KV head) that every call leaves at
                            zero, and the split partials. Calls that share a workspace must be
                            ordered (one stream); concurrent calls need their own. After
                            lbkv_device_status reports an error, zero it again. */
  size_t workspace_bytes;
  /* Paged cache (optional; page_table NULL: the contiguous layout above). The codes,
   * scales and offsets of every call then live in pools of pages: codes
   * [num_pages][Hkv][page_tokens][D*bits/8], token-wise scales/offsets
   * [num_pages][Hkv][page_tokens][D/group], channel-wise [num_pages][Hkv][page_tokens/group][D];
   * token t of sequence b is row t mod page_tokens of page page_table[b][t / page_tokens].
   * page_tokens is a power of two >= 128, max_seq_len <= max_pages * page_tokens, and
   * the entries for the pages that hold a sequence's tokens lie in [0, num_pages) (an entry
   * outside is read as page 0 and recorded as device status 5). The bf16 window, q and out
   * are not paged. */
  const int32_t* page_table; /* int32 [B][max_pages] device, or NULL */
  int32_t page_tokens;
  int32_t max_pages;
  int32_t num_pages;
  int32_t rotation; /* lbkv_rotation bits of the stored rows, 0 for none (see above) */
} lbkv_desc;

/* Bytes of workspace lbkv_decode_attn needs for this descriptor and format on
 * the current device (the split-KV partials: a running maximum, a softmax
 * denominator and a head_dim vector per query head and split). Returns 0 when
 * the arguments are invalid. Reads only desc's shape fields. */
LBKV_API size_t lbkv_workspace_bytes(const lbkv_desc* desc, int bits, int k_layout, int v_layout, int group);

/* Decode attention for one new token per sequence, split-KV over the cache.
 *   q, k_codes, k_scale, k_off, v_codes, v_scale, v_off, seq_lens, out: see the layout above;
 *   bits: 2 or 4; k_layout / v_layout: lbkv_layout; group: 32, 64 or 128
 *   (a divisor of head_dim for a token-wise side, a token count for a
 *   channel-wise side).
 * Supported: every combination of bits, layouts and group above with
 *   Hq/Hkv in {1, 2, 4, 8} (other ratios, groups or head_dim give
 *   LBKV_EUNSUPPORTED). For a token-wise V side with group 32 and Hq/Hkv = 8
 *   the queries of each KV head are processed in two halves, each reading
 *   the KV head's cached data (twice the cache traffic for that case).
 * Precision: tensor-core products on exact fp16 images of the codes; the bf16
 * query enters exactly (fp16; rounded to fp16 after a channel-wise K scale
 * multiplies it) and the softmax weights as fp16; accumulation and every fold
 * step in fp32; output rounded to bf16.
 * Rotated cache (desc->rotation): the query is rotated by H in fp32 before the scores
 * (LBKV_ROTATE_K) and the output rotated back by H in fp32 before its bf16 rounding
 * (LBKV_ROTATE_V); the window must be stored the same way.
 * Errors: LBKV_EINVAL / LBKV_EALIGN / LBKV_EUNSUPPORTED / LBKV_EWORKSPACE before
 * any launch; LBKV_ECUDA on a launch failure. A sequence with no cached and no
 * window tokens yields a zero output row. */
LBKV_API int lbkv_decode_attn(const lbkv_desc* desc, const void* q, const uint8_t* k_codes, const void* k_scale,
                     const void* k_off, const uint8_t* v_codes, const void* v_scale, const void* v_off,
                     const int32_t* seq_lens, int bits, int k_layout, int v_layout, int group, void* out,
                     lbkv_stream_t stream);

/* The launch lbkv_decode_attn makes for this descriptor and format on the current device,
 * without running it (the device is queried for its SM count and thread-block cluster
 * occupancy; desc's pointers are only tested for NULL, as lbkv_decode_attn tests them):
 *   grid: CTAs of the decode kernel (0 for an empty batch);
 *   cluster: CTAs per thread-block cluster, or 0 for the split-decode grid (the CTAs take
 *     equal shares of all pairs' items after a scan of the lengths, and the last CTA of a
 *     pair merges its partials);
 *   split: clusters per (sequence, KV head) pair: 1, the cluster merges its CTAs in
 *     distributed shared memory and writes the output; more, each cluster writes one partial
 *     and the pair's last cluster merges them.
 * A call whose cluster launch the device refuses runs on the split-decode grid instead.
 * Errors: those lbkv_decode_attn returns for invalid arguments; LBKV_EINVAL for a NULL
 * output pointer. */
LBKV_API int lbkv_decode_launch_info(const lbkv_desc* desc, int bits, int k_layout, int v_layout, int group,
                                     int* grid, int* cluster, int* split);

/* Quantize a bf16 cache side x [B][Hkv][T_cap][D] into the layout above
 * (the value model s * q + z is the explainer's quantization-format
 * paragraph; the quantizer is this library's reading): per group
 *   s = fp16((max - min) / (2^bits - 1)), z = fp16(min),
 *   q = clamp(round_half_even((x - z) / s), 0, 2^bits - 1), q = 0 when s == 0,
 * each operation in IEEE single precision rounded on its own. A channel-wise
 * group that ends past L_b uses only its valid tokens. Codes of tokens
 * t >= L_b are written as 0; their scales and offsets are left untouched.
 * Paged cache (desc->page_table): x stays [B][Hkv][T_cap][D]; codes, scales and
 * offsets are the page pools, of which only the rows of tokens t < L_b (channel-wise:
 * the groups that hold one) are written. A token whose page-table entry lies outside
 * the pool is not stored and, if desc->workspace is given (256-byte aligned), its
 * status word records 5.
 * Uses desc's batch, num_kv_heads, head_dim (128), max_seq_len, paged fields and
 * workspace (optional). Errors as for lbkv_decode_attn. */
LBKV_API int lbkv_pack(const lbkv_desc* desc, const void* x, const int32_t* seq_lens, int bits, int layout, int group,
              uint8_t* codes, void* scale, void* off, lbkv_stream_t stream);

/* Quantize-on-append: store the K and V of the token a decode step just produced
 * (the step before the decode path when serving, which the abstract of "FOSCAR:
 * Accelerating Decode Attention over 2- and 4-Bit KV Caches through Affine Folding"
 * integrates into SGLang; how a token is appended is this library's reading), with the
 * same quantizer as lbkv_pack.
 *   k_new, v_new: bf16 [B][Hkv][D] device, the new token of every (sequence, KV head).
 *   seq_lens: int32 [B] device, the cached tokens L_b; advanced in place.
 * Both sides token-wise: the token is quantized per group of `group` channels into
 * position L_b, and L_b += 1. Otherwise (a channel-wise side, whose groups span
 * `group` tokens) both sides go through the bf16 window of desc (k_win, v_win,
 * win_lens, win_cap >= group required): the token is copied into window slot
 * W_b = win_lens[b] and W_b += 1; when the window then holds `group` tokens they are
 * quantized into positions L_b .. L_b + group - 1 (token-wise side: per token;
 * channel-wise side: as one group), L_b += group and W_b = 0. The cache then holds
 * exactly what lbkv_pack would produce from the same bf16 history.
 * A sequence whose token does not fit (L_b == max_seq_len; a channel-wise L_b that is
 * not a multiple of group or has no room for a group; W_b >= group) is left unchanged,
 * and if desc->workspace is given its status word records 4 (see lbkv_device_status).
 * A side named in desc->rotation is rotated on the way in, as lbkv_rotate does, into the
 * cache and the window alike.
 * Codes, scales and offsets as for lbkv_pack (paged cache included: a token whose
 * page-table entry lies outside the pool is not stored, status 5); all pointers 16-byte
 * aligned. Uses desc's batch, num_kv_heads, head_dim, max_seq_len, window fields, paged
 * fields, rotation and workspace (optional). Asynchronous on `stream`. Errors as for lbkv_pack. */
LBKV_API int lbkv_append(const lbkv_desc* desc, const void* k_new, const void* v_new, int32_t* seq_lens, int bits,
                         int k_layout, int v_layout, int group, uint8_t* k_codes, void* k_scale, void* k_off,
                         uint8_t* v_codes, void* v_scale, void* v_off, lbkv_stream_t stream);

/* Rotate bf16 rows of head_dim = 128 channels by the normalized Hadamard matrix H (see
 * lbkv_rotation): y[r] = bf16(H x[r]) for r < rows, the step before lbkv_pack for a cache
 * stored rotated. Computed as the Walsh-Hadamard butterflies in IEEE single precision
 * (stages of span 1, 2, 4, ..., 64; the lower channel of a pair takes a + b, the upper
 * a - b), each value then scaled by fp32(1/sqrt(128)) and rounded to bf16 (nearest, ties
 * to even), so the bits do not depend on the GPU.
 *   x, y: bf16 [rows][128] device, 16-byte aligned; y == x rotates in place (other
 *   overlaps are not allowed). rows >= 0.
 * Asynchronous on `stream`. Errors: LBKV_EINVAL (null pointer, rows < 0),
 * LBKV_EUNSUPPORTED (head_dim != 128), LBKV_EALIGN, LBKV_ECUDA. */
LBKV_API int lbkv_rotate(const void* x, void* y, int64_t rows, int head_dim, lbkv_stream_t stream);

/* BF16 comparator: the same split-KV decode attention over a bf16 cache, without
 * quantization, so that the speedup that "FOSCAR: Accelerating Decode Attention over 2-
 * and 4-Bit KV Caches through Affine Folding" (abstract) reports over a BF16 decode
 * kernel can be measured on this GPU and pipeline.
 *   q: bf16 [B][Hq][D]; k, v: bf16 [B][Hkv][max_seq_len][D]; seq_lens: int32 [B] device;
 *   out: bf16 [B][Hq][D]. Softmax over the first L_b tokens (zero output when L_b == 0).
 * Uses desc's batch, heads, head_dim (128), max_seq_len, sm_scale and workspace (of at
 * least lbkv_bf16_workspace_bytes bytes, 256-byte aligned, first 256 bytes zeroed once:
 * the status word). Window fields and page_table must be NULL and rotation 0
 * (LBKV_EUNSUPPORTED).
 * Hq/Hkv <= 8.
 * Errors as for lbkv_decode_attn. Asynchronous on `stream`. */
LBKV_API size_t lbkv_bf16_workspace_bytes(const lbkv_desc* desc);
LBKV_API int lbkv_decode_bf16(const lbkv_desc* desc, const void* q, const void* k, const void* v,
                              const int32_t* seq_lens, void* out, lbkv_stream_t stream);

/* Same computation and arguments as lbkv_decode_attn, for callers that cannot
 * allocate device memory (an engine whose allocator owns all device memory, a
 * plugin that only receives its input and output buffers, a loop where an
 * allocation is not allowed). desc->workspace and desc->workspace_bytes are
 * ignored: the split-KV scratch is a fixed array of lbkv_noalloc_scratch_bytes()
 * bytes (16 MiB) inside this library, which every GPU that loads the library
 * keeps until the process exits. There is no counterpart on the pages; it only
 * changes where the scratch lives.
 *   - A call whose scratch (lbkv_workspace_bytes for the same arguments) would
 *     exceed that size returns LBKV_ESCRATCH before anything is launched.
 *   - The first call on each device looks the array's address up with that
 *     device current; make that first call before any stream capture.
 *   - Every call on a device shares the array and it keeps the last call's
 *     contents; the call clears the part that must start at zero. Calls that
 *     overlap on the GPU (other streams, other threads) race: order them.
 *   - The device status word (a bounded wait that ran out) lives in the same array
 *     and is cleared at the start of every call: lbkv_device_status cannot read it
 *     for these calls (it takes a caller's workspace).
 *   - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library call. */
LBKV_API int lbkv_decode_attn_noalloc(const lbkv_desc* desc, const void* q, const uint8_t* k_codes,
                                      const void* k_scale, const void* k_off, const uint8_t* v_codes,
                                      const void* v_scale, const void* v_off, const int32_t* seq_lens, int bits,
                                      int k_layout, int v_layout, int group, void* out, lbkv_stream_t stream);

/* Size in bytes of the fixed scratch array behind lbkv_decode_attn_noalloc. */
LBKV_API size_t lbkv_noalloc_scratch_bytes(void);

/* Reads and clears the device status word that kernels set instead of
 * hanging (a bounded wait that ran out). Synchronizes `stream`. Returns
 * LBKV_OK, LBKV_EDEVICE (the word was set; *code receives it when code is
 * not NULL) or LBKV_ECUDA / LBKV_EINVAL / LBKV_EWORKSPACE. */
LBKV_API int lbkv_device_status(const lbkv_desc* desc, lbkv_stream_t stream, int32_t* code);

/* Self-test of the bounded waits every kernel uses instead of spinning forever:
 * launches one warp that waits on an mbarrier nothing completes. The wait gives up
 * after limit_ns nanoseconds (0 < limit_ns <= 1e9), writes 1 (a consumer wait ran
 * out, the code the decode kernel uses) to status[0], and the warp then adds 1 to
 * status[1] and exits. status: device int32[2], 16-byte aligned, zeroed by the
 * caller. Asynchronous on `stream`. Returns LBKV_OK, LBKV_EINVAL, LBKV_EALIGN or
 * LBKV_ECUDA. (Not part of the method: a check that a failed wait reports instead
 * of hanging and leaves the context usable.) */
LBKV_API int lbkv_selftest_wait_timeout(void* status, uint64_t limit_ns, lbkv_stream_t stream);

/* Static English text for a status value. */
LBKV_API const char* lbkv_strerror(int status);

#ifdef __cplusplus
}
#endif
#endif /* LBKV_H */
