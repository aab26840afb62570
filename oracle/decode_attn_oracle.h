/*
 * decode_attn_oracle.h -- the float64 CPU oracle for single-query decode attention.
 *
 * TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / reference leg may load or call this code. The product path (the
 * CUDA library and its Python binding) never does. This header is the oracle's
 * own; it shares nothing with the CUDA library's sources or headers.
 *
 * What it computes is the plain definition, written out with no blocking, no
 * splitting and no unified constant:
 *   o = softmax(q K^T * scale) V   over the sequence's first N_b tokens,
 * read through the same logical -> physical token mapping the cache uses.
 * Sources: "Flash-Decoding: Mathematical Foundations, Split-KV Parallelism, Online
 * Softmax Reduction, and Serving Latency Optimization", section "The Single-Token
 * Generation Bottleneck"; "FlashAttention and inference kernels", sections
 * "PagedAttention" and "A paged decode attention kernel (with GQA)" (its float64
 * CPU reference and its GQA head mapping).
 */
#ifndef DECODE_ATTN_ORACLE_H
#define DECODE_ATTN_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element encodings the oracle reads exactly (bit for bit) from storage. ORACLE_E4M3 is
 * the 8-bit floating-point format with 4 exponent bits (bias 7) and 3 mantissa bits, no
 * infinities and S.1111.111 as NaN ("E4M3FN"); it is used only for K and V caches. */
enum { ORACLE_F32 = 0, ORACLE_F16 = 1, ORACLE_BF16 = 2, ORACLE_E4M3 = 3 };

typedef struct {
  int batch;                /* B */
  int num_q_heads;          /* H_q */
  int num_kv_heads;         /* H_kv, divides H_q */
  int head_dim;             /* d, any value >= 1 */
  int paged;                /* 1: caches are [num_physical_blocks, page_size, H_kv, d] */
                            /* 0: caches are [B, max_seq_len, H_kv, d]                  */
  int page_size;            /* tokens per physical block (paged only) */
  int max_blocks_per_seq;   /* block-table row length (paged only) */
  int max_seq_len;          /* token capacity per sequence (contiguous only) */
  int num_physical_blocks;  /* size of the paged pool (paged only) */
  int dtype;                /* ORACLE_F32 / ORACLE_F16 / ORACLE_BF16 for q, k and v */
  int kv_e4m3;              /* 1: k and v are ORACLE_E4M3 codes (q stays dtype), each */
  double k_scale;           /* element standing for code * k_scale / code * v_scale    */
  double v_scale;           /* ("FlashAttention and inference kernels": an FP8 KV cache, */
                            /* converted on read); 0: k, v in dtype, scales unused     */
} oracle_shape;

/* Exact value of element `index` of an array stored in `dtype`. */
double oracle_load(int dtype, const void* base, int64_t index);

/* Element offset of token t of (sequence b, KV head kvh) in the K (or V) cache, or
 * -1 when the block-table entry is outside [0, num_physical_blocks) or t is past the
 * table. */
int64_t oracle_kv_offset(const oracle_shape* s, const int32_t* block_table, int b, int kvh,
                         int64_t t);

/* offs[(b * H_kv + kvh) * T + t] for t < T, where T = max_blocks_per_seq * page_size
 * (paged) or max_seq_len (contiguous); -1 for t >= seq_lens[b]. */
int oracle_gather_offsets(const oracle_shape* s, const int32_t* block_table,
                          const int32_t* seq_lens, int64_t* offs);

/* The full decode attention, one row (b, h_q) at a time.
 *   rows   : row ids b * H_q + h_q to compute, or NULL for every row in order.
 *   out    : [nrows, d] float64;  lse : [nrows] natural-log log-sum-exp of the scaled
 *            logits;  row_flag : [nrows] 1 iff some scaled logit x has x - phi < lo or
 *            x - phi > hi;  margin : [nrows] |max_t dist_t| with
 *            dist_t = max(lo - (x_t - phi), (x_t - phi) - hi), the distance of the
 *            row's flag decision from flipping (+inf for an empty row).
 * Any of lse, row_flag, margin may be NULL. An empty row (seq_lens[b] == 0) gives
 * out = 0, lse = -inf, flag = 0. Returns 0, or -1 on a bad argument or a block-table
 * entry outside the pool. */
int oracle_decode_attn(const oracle_shape* s, const void* q, const void* k, const void* v,
                       const int32_t* block_table, const int32_t* seq_lens, double scale,
                       double phi, double range_lo, double range_hi, const int64_t* rows,
                       int64_t nrows, double* out, double* lse, uint8_t* row_flag,
                       double* margin, int nthreads);

/* One split's partial results for row (b, h_q) over an explicit list of token indices
 * (any subset, in any order): the split's scaled logits S, m = max S,
 * l = sum exp(S - m), the normalised partial output O = sum exp(S - m) v / l and
 * L = m + ln l. An empty list gives m = L = -inf, l = 0, O = 0. */
int oracle_split_partial(const oracle_shape* s, const void* q, const void* k, const void* v,
                         const int32_t* block_table, int b, int h, const int64_t* tokens,
                         int64_t ntok, double scale, double* o_s, double* m_s, double* l_s,
                         double* L_s);

/* Exact merge of S split partials, max-rescale form:
 *   m = max_s m_s,  l = sum_s l_s exp(m_s - m),  O = sum_s l_s exp(m_s - m) O_s / l,
 *   lse = m + ln l.  Splits with l_s == 0 are skipped; all empty -> O = 0, lse = -inf. */
int oracle_lse_merge(int S, int d, const double* o_s, const double* m_s, const double* l_s,
                     double* o, double* lse);

/* The same merge in log-sum-exp form: L = ln sum_s exp(L_s), O = sum_s exp(L_s - L) O_s. */
int oracle_lse_merge_alpha(int S, int d, const double* o_s, const double* L_s, double* o,
                           double* lse);

/* The unified-max ("asynchronised") form for row (b, h_q), split into consecutive
 * partitions of `split_tokens` tokens (0 = one partition): each partition accumulates
 * num = sum exp(x - phi) v and den = sum exp(x - phi) with no maximum; the result is
 * sum num / sum den. flag as for oracle_decode_attn; split_flags (nullable) receives
 * the number of partitions holding an out-of-range logit. */
int oracle_unified_row(const oracle_shape* s, const void* q, const void* k, const void* v,
                       const int32_t* block_table, const int32_t* seq_lens, int b, int h,
                       double scale, double phi, double range_lo, double range_hi,
                       int64_t split_tokens, double* out, double* lse, uint8_t* flag,
                       int64_t* split_flags);

/* The scaled logits x = scale * q[b,h_q] . k_t of every row, rows in order b * H_q + h_q
 * and tokens t < seq_lens[b] in order within a row, written to out (which holds
 * sum_b seq_lens[b] * H_q values): the pre-softmax values whose distribution
 * "FlashDecoding++" (Fig. 5, "The Overflow and Precision Problem: Choosing phi") reports.
 * Returns the number written, or -1 on a bad argument or block-table entry. */
int64_t oracle_logits(const oracle_shape* s, const void* q, const void* k,
                      const int32_t* block_table, const int32_t* seq_lens, double scale,
                      double* out);

#ifdef __cplusplus
}
#endif

#endif
