/*
 * decode_attn_oracle.c -- plain, slow, obviously correct float64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / reference leg, never by the product path. It shares no code, header,
 * table or helper with the CUDA library.
 *
 * Every function states the passage it follows. Sources (page title, then section):
 *   [FD]  "Flash-Decoding: Mathematical Foundations, Split-KV Parallelism, Online Softmax
 *         Reduction, and Serving Latency Optimization"
 *   [FDPP] "FlashDecoding++: Faster Large Language Model Inference on GPUs" (arXiv
 *         2311.01282 summary page)
 *   [HB]  "FlashAttention and inference kernels" (AI infra handbook, CUDA / advanced /
 *         attention)
 *
 * Pins (tests/test_oracle_pins.py, all -m "not gpu"): the handbook's worked online-softmax
 * example (Exercise 1), the FlashDecoding++ Fig. 6 flag example, an independent NumPy
 * brute force on tiny shapes, closed forms (constant V, uniform logits, one-hot large
 * logit through a shuffled block table), partition invariance of the merge, agreement of
 * the two merge forms, unified == synchronised on unflagged rows, IEEE decoding of
 * fp16 / bf16 against library conversions, and the GQA head mapping by a one-hot probe.
 * No function here is "parity unpinned".
 */
#include "decode_attn_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---- exact element decoding (IEEE 754 binary32 / binary16, and bfloat16 = the top
 * 16 bits of a binary32) ------------------------------------------------------------ */
static double decode_f16(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int e = (h >> 10) & 0x1f;
  const int m = h & 0x3ff;
  double mag;
  if (e == 0) {
    mag = ldexp((double)m, -24); /* subnormal: m * 2^-10 * 2^-14 */
  } else if (e == 31) {
    mag = m ? NAN : INFINITY;
  } else {
    mag = ldexp(1024.0 + (double)m, e - 25); /* (1 + m/1024) * 2^(e-15) */
  }
  return sign ? -mag : mag;
}

static double decode_bf16(uint16_t h) {
  const uint32_t bits = (uint32_t)h << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* E4M3 ("E4M3FN"): sign, 4-bit exponent e with bias 7, 3-bit mantissa m. e = 0 is
 * subnormal, m * 2^-9 (= m/8 * 2^-6); e = 15 with m = 7 is NaN; every other code is
 * (1 + m/8) * 2^(e - 7), up to 448. There are no infinities. */
static double decode_e4m3(uint8_t c) {
  const int sign = (c >> 7) & 1;
  const int e = (c >> 3) & 0xf;
  const int m = c & 0x7;
  double mag;
  if (e == 0xf && m == 0x7)
    mag = NAN;
  else if (e == 0)
    mag = ldexp((double)m, -9);
  else
    mag = ldexp(8.0 + (double)m, e - 10); /* (1 + m/8) * 2^(e-7) */
  return sign ? -mag : mag;
}

double oracle_load(int dtype, const void* base, int64_t index) {
  switch (dtype) {
    case ORACLE_F32: {
      float f;
      memcpy(&f, (const char*)base + index * 4, sizeof f);
      return (double)f;
    }
    case ORACLE_F16: {
      uint16_t h;
      memcpy(&h, (const char*)base + index * 2, sizeof h);
      return decode_f16(h);
    }
    case ORACLE_BF16: {
      uint16_t h;
      memcpy(&h, (const char*)base + index * 2, sizeof h);
      return decode_bf16(h);
    }
    case ORACLE_E4M3:
      return decode_e4m3(((const uint8_t*)base)[index]);
    default:
      return NAN;
  }
}

/* ---- shape checks ---------------------------------------------------------------- */
static int shape_ok(const oracle_shape* s) {
  if (!s || s->batch < 0 || s->num_q_heads <= 0 || s->num_kv_heads <= 0 || s->head_dim <= 0)
    return 0;
  if (s->num_q_heads % s->num_kv_heads) return 0;
  if (s->dtype < ORACLE_F32 || s->dtype > ORACLE_BF16) return 0;
  if (s->kv_e4m3 != 0 && s->kv_e4m3 != 1) return 0;
  if (s->kv_e4m3 && !(isfinite(s->k_scale) && isfinite(s->v_scale))) return 0;
  if (s->paged) {
    if (s->page_size <= 0 || s->max_blocks_per_seq < 0 || s->num_physical_blocks < 0) return 0;
  } else if (s->max_seq_len < 0) {
    return 0;
  }
  return 1;
}

static int64_t token_capacity(const oracle_shape* s) {
  return s->paged ? (int64_t)s->max_blocks_per_seq * s->page_size : (int64_t)s->max_seq_len;
}

/* [HB] "PagedAttention": token t of a sequence lives at slot t % page_size of physical
 * block block_table[t / page_size]; the cache is [num_blocks, page, H_kv, d]
 * ("A paged decode attention kernel (with GQA)"). The contiguous cache is
 * [B, max_seq_len, H_kv, d]. */
int64_t oracle_kv_offset(const oracle_shape* s, const int32_t* block_table, int b, int kvh,
                         int64_t t) {
  const int64_t H = s->num_kv_heads, d = s->head_dim;
  if (t < 0 || t >= token_capacity(s)) return -1;
  if (s->paged) {
    const int64_t logical_block = t / s->page_size;
    const int64_t slot = t % s->page_size;
    const int32_t phys = block_table[(int64_t)b * s->max_blocks_per_seq + logical_block];
    if (phys < 0 || phys >= s->num_physical_blocks) return -1;
    return (((int64_t)phys * s->page_size + slot) * H + kvh) * d;
  }
  return (((int64_t)b * s->max_seq_len + t) * H + kvh) * d;
}

int oracle_gather_offsets(const oracle_shape* s, const int32_t* block_table,
                          const int32_t* seq_lens, int64_t* offs) {
  if (!shape_ok(s) || !seq_lens || !offs || (s->paged && !block_table)) return -1;
  const int64_t T = token_capacity(s);
  for (int b = 0; b < s->batch; ++b)
    for (int kvh = 0; kvh < s->num_kv_heads; ++kvh)
      for (int64_t t = 0; t < T; ++t)
        offs[((int64_t)b * s->num_kv_heads + kvh) * T + t] =
            t < seq_lens[b] ? oracle_kv_offset(s, block_table, b, kvh, t) : -1;
  return 0;
}

/* Element `index` of the K / V cache: in q's encoding, or for an FP8 cache the code's
 * value times the tensor's scale ([HB] "A paged decode attention kernel (with GQA)": the
 * cache is "really BF16 or FP8", converted on read). */
static double load_k(const oracle_shape* s, const void* k, int64_t index) {
  return s->kv_e4m3 ? oracle_load(ORACLE_E4M3, k, index) * s->k_scale
                    : oracle_load(s->dtype, k, index);
}

static double load_v(const oracle_shape* s, const void* v, int64_t index) {
  return s->kv_e4m3 ? oracle_load(ORACLE_E4M3, v, index) * s->v_scale
                    : oracle_load(s->dtype, v, index);
}

/* [HB] "A paged decode attention kernel (with GQA)": several query heads share one KV
 * head, kv_head = head / (num_heads / num_kv_heads). */
static int kv_head_of(const oracle_shape* s, int h) {
  return h / (s->num_q_heads / s->num_kv_heads);
}

/* Scaled logit x_t = scale * <q[b,h,:], k_t> ([FD] "Mathematical Formulation of Split-KV
 * Parallelism": S = q K^T / sqrt(d), with the caller's scale in place of 1/sqrt(d)). */
static double logit(const oracle_shape* s, const void* q, const void* k, int b, int h,
                    int64_t koff, double scale) {
  const int64_t d = s->head_dim;
  const int64_t qoff = ((int64_t)b * s->num_q_heads + h) * d;
  double dot = 0.0;
  for (int64_t i = 0; i < d; ++i)
    dot += oracle_load(s->dtype, q, qoff + i) * load_k(s, k, koff + i);
  return scale * dot;
}

/* Distance of x - phi outside the closed interval [lo, hi] (positive = outside).
 * [FDPP] "The Overflow Fallback: Recomputation", Fig. 6: an element exactly on the
 * bound is in range (the worked example accepts 3 - 6 = -3 >= -3 and 9 - 6 = 3 <= 3);
 * only a strictly outside element triggers the recompute. */
static double outside_distance(double x, double phi, double lo, double hi) {
  const double y = x - phi;
  const double below = lo - y, above = y - hi;
  return below > above ? below : above;
}

/* One row of the plain definition: [FD] "The Single-Token Generation Bottleneck"
 * o = softmax(q K^T / sqrt(d)) V, evaluated as the max-shifted softmax of [FDPP]
 * "Asynchronized Softmax with Unified Max Value" (standard form, m = max x). */
static int one_row(const oracle_shape* s, const void* q, const void* k, const void* v,
                   const int32_t* block_table, const int32_t* seq_lens, double scale,
                   double phi, double lo, double hi, int64_t row, double* out, double* lse,
                   uint8_t* flag, double* margin) {
  const int64_t d = s->head_dim;
  const int b = (int)(row / s->num_q_heads), h = (int)(row % s->num_q_heads);
  const int kvh = kv_head_of(s, h);
  const int64_t n = seq_lens[b];
  for (int64_t i = 0; i < d; ++i) out[i] = 0.0;
  if (n < 0 || n > token_capacity(s)) return -1;
  if (n == 0) {
    if (lse) *lse = -INFINITY;
    if (flag) *flag = 0;
    if (margin) *margin = INFINITY;
    return 0;
  }
  double* x = (double*)malloc((size_t)n * sizeof(double));
  int64_t* off = (int64_t*)malloc((size_t)n * sizeof(int64_t));
  if (!x || !off) {
    free(x);
    free(off);
    return -1;
  }
  int rc = 0;
  double m = -INFINITY, worst = -INFINITY;
  for (int64_t t = 0; t < n; ++t) {
    off[t] = oracle_kv_offset(s, block_table, b, kvh, t);
    if (off[t] < 0) {
      rc = -1;
      break;
    }
    x[t] = logit(s, q, k, b, h, off[t], scale);
    if (x[t] > m) m = x[t];
    const double dist = outside_distance(x[t], phi, lo, hi);
    if (dist > worst) worst = dist;
  }
  if (rc == 0) {
    double l = 0.0;
    for (int64_t t = 0; t < n; ++t) l += exp(x[t] - m);
    for (int64_t t = 0; t < n; ++t) {
      const double p = exp(x[t] - m);
      for (int64_t i = 0; i < d; ++i) out[i] += p * load_v(s, v, off[t] + i);
    }
    for (int64_t i = 0; i < d; ++i) out[i] /= l;
    if (lse) *lse = m + log(l);
    if (flag) *flag = worst > 0.0 ? 1 : 0;
    if (margin) *margin = fabs(worst);
  }
  free(x);
  free(off);
  return rc;
}

int oracle_decode_attn(const oracle_shape* s, const void* q, const void* k, const void* v,
                       const int32_t* block_table, const int32_t* seq_lens, double scale,
                       double phi, double range_lo, double range_hi, const int64_t* rows,
                       int64_t nrows, double* out, double* lse, uint8_t* row_flag,
                       double* margin, int nthreads) {
  if (!shape_ok(s) || !q || !k || !v || !seq_lens || !out) return -1;
  if (s->paged && !block_table) return -1;
  const int64_t all = (int64_t)s->batch * s->num_q_heads;
  const int64_t count = rows ? nrows : all;
  if (rows)
    for (int64_t r = 0; r < count; ++r)
      if (rows[r] < 0 || rows[r] >= all) return -1;
  int failed = 0;
  (void)nthreads;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1) \
    reduction(| : failed)
  for (int64_t r = 0; r < count; ++r) {
    const int64_t row = rows ? rows[r] : r;
    if (one_row(s, q, k, v, block_table, seq_lens, scale, phi, range_lo, range_hi, row,
                out + r * s->head_dim, lse ? lse + r : NULL, row_flag ? row_flag + r : NULL,
                margin ? margin + r : NULL))
      failed = 1;
  }
  return failed ? -1 : 0;
}

/* [FD] "Mathematical Formulation of Split-KV Parallelism": for split s, the local logits
 * S^(s), the local maximum m^(s), the local sum l^(s) = sum exp(S^(s) - m^(s)), the
 * normalised partial output O^(s) = (1 / l^(s)) sum exp(S^(s) - m^(s)) V^(s), and
 * L^(s) = m^(s) + ln l^(s). [HB] Exercise 2: an empty segment has l = 0, m = -inf. */
int oracle_split_partial(const oracle_shape* s, const void* q, const void* k, const void* v,
                         const int32_t* block_table, int b, int h, const int64_t* tokens,
                         int64_t ntok, double scale, double* o_s, double* m_s, double* l_s,
                         double* L_s) {
  if (!shape_ok(s) || !q || !k || !v || !o_s || !m_s || !l_s || !L_s) return -1;
  if (b < 0 || b >= s->batch || h < 0 || h >= s->num_q_heads || ntok < 0) return -1;
  const int64_t d = s->head_dim;
  const int kvh = kv_head_of(s, h);
  for (int64_t i = 0; i < d; ++i) o_s[i] = 0.0;
  *m_s = -INFINITY;
  *l_s = 0.0;
  *L_s = -INFINITY;
  if (ntok == 0) return 0;
  double* x = (double*)malloc((size_t)ntok * sizeof(double));
  int64_t* off = (int64_t*)malloc((size_t)ntok * sizeof(int64_t));
  if (!x || !off) {
    free(x);
    free(off);
    return -1;
  }
  int rc = 0;
  double m = -INFINITY;
  for (int64_t j = 0; j < ntok; ++j) {
    off[j] = oracle_kv_offset(s, block_table, b, kvh, tokens[j]);
    if (off[j] < 0) {
      rc = -1;
      break;
    }
    x[j] = logit(s, q, k, b, h, off[j], scale);
    if (x[j] > m) m = x[j];
  }
  if (rc == 0) {
    double l = 0.0;
    for (int64_t j = 0; j < ntok; ++j) l += exp(x[j] - m);
    for (int64_t j = 0; j < ntok; ++j) {
      const double p = exp(x[j] - m);
      for (int64_t i = 0; i < d; ++i) o_s[i] += p * load_v(s, v, off[j] + i);
    }
    for (int64_t i = 0; i < d; ++i) o_s[i] /= l;
    *m_s = m;
    *l_s = l;
    *L_s = m + log(l);
  }
  free(x);
  free(off);
  return rc;
}

/* [FD] "The Rescaling and Online Softmax Reduction Algorithm" (first form):
 * m = max_s m^(s); l = sum_s l^(s) exp(m^(s) - m); O = (1/l) sum_s l^(s) exp(m^(s) - m) O^(s).
 * [HB] "Parallelism during decode: Flash-Decoding and split-K" states the same merge;
 * [HB] Exercise 2: segments with l = 0 (m = -inf) are skipped. */
int oracle_lse_merge(int S, int d, const double* o_s, const double* m_s, const double* l_s,
                     double* o, double* lse) {
  if (S < 0 || d <= 0 || !o || !lse || (S > 0 && (!o_s || !m_s || !l_s))) return -1;
  double m = -INFINITY;
  for (int s = 0; s < S; ++s)
    if (l_s[s] > 0.0 && m_s[s] > m) m = m_s[s];
  for (int i = 0; i < d; ++i) o[i] = 0.0;
  if (m == -INFINITY) {
    *lse = -INFINITY;
    return 0;
  }
  double l = 0.0;
  for (int s = 0; s < S; ++s) {
    if (!(l_s[s] > 0.0)) continue;
    const double w = l_s[s] * exp(m_s[s] - m);
    l += w;
    for (int i = 0; i < d; ++i) o[i] += w * o_s[(int64_t)s * d + i];
  }
  for (int i = 0; i < d; ++i) o[i] /= l;
  *lse = m + log(l);
  return 0;
}

/* [FD] "The Rescaling and Online Softmax Reduction Algorithm" (log-sum-exp form):
 * L = ln(sum_s exp(L^(s))), alpha^(s) = exp(L^(s) - L), O = sum_s alpha^(s) O^(s).
 * The sum of exponentials is evaluated shifted by max L^(s) so that it cannot
 * overflow; the shift cancels in L. */
int oracle_lse_merge_alpha(int S, int d, const double* o_s, const double* L_s, double* o,
                           double* lse) {
  if (S < 0 || d <= 0 || !o || !lse || (S > 0 && (!o_s || !L_s))) return -1;
  double top = -INFINITY;
  for (int s = 0; s < S; ++s)
    if (L_s[s] > top) top = L_s[s];
  for (int i = 0; i < d; ++i) o[i] = 0.0;
  if (top == -INFINITY) {
    *lse = -INFINITY;
    return 0;
  }
  double sum = 0.0;
  for (int s = 0; s < S; ++s)
    if (L_s[s] > -INFINITY) sum += exp(L_s[s] - top);
  const double L = top + log(sum);
  for (int s = 0; s < S; ++s) {
    if (!(L_s[s] > -INFINITY)) continue;
    const double alpha = exp(L_s[s] - L);
    for (int i = 0; i < d; ++i) o[i] += alpha * o_s[(int64_t)s * d + i];
  }
  *lse = L;
  return 0;
}

/* [FDPP] "Mathematical Reformulation: Unified Max Value" (Eq. 3): the softmax is
 * unchanged when every element is shifted by the same constant phi instead of by the
 * maximum. "Asynchronized Execution with Inner Product" (Eq. 4): each partition j
 * accumulates num^(j) = sum exp(x - phi) v and den^(j) = sum exp(x - phi); the output is
 * sum_j num^(j) / sum_j den^(j). "The Overflow Fallback: Recomputation": a partition with
 * an element outside [lo, hi] (closed, per Fig. 6) flags the whole row. */
int oracle_unified_row(const oracle_shape* s, const void* q, const void* k, const void* v,
                       const int32_t* block_table, const int32_t* seq_lens, int b, int h,
                       double scale, double phi, double range_lo, double range_hi,
                       int64_t split_tokens, double* out, double* lse, uint8_t* flag,
                       int64_t* split_flags) {
  if (!shape_ok(s) || !q || !k || !v || !seq_lens || !out || !lse || !flag) return -1;
  if (b < 0 || b >= s->batch || h < 0 || h >= s->num_q_heads || split_tokens < 0) return -1;
  const int64_t d = s->head_dim;
  const int kvh = kv_head_of(s, h);
  const int64_t n = seq_lens[b];
  if (n < 0 || n > token_capacity(s)) return -1;
  const int64_t part = split_tokens > 0 ? split_tokens : (n > 0 ? n : 1);
  double* num = (double*)calloc((size_t)d, sizeof(double));
  double* num_j = (double*)calloc((size_t)d, sizeof(double));
  if (!num || !num_j) {
    free(num);
    free(num_j);
    return -1;
  }
  double den = 0.0;
  int any = 0;
  int64_t flagged_parts = 0;
  int rc = 0;
  for (int64_t t0 = 0; t0 < n && rc == 0; t0 += part) {
    const int64_t t1 = t0 + part < n ? t0 + part : n;
    double den_j = 0.0;
    int flag_j = 0;
    for (int64_t i = 0; i < d; ++i) num_j[i] = 0.0;
    for (int64_t t = t0; t < t1; ++t) {
      const int64_t off = oracle_kv_offset(s, block_table, b, kvh, t);
      if (off < 0) {
        rc = -1;
        break;
      }
      const double x = logit(s, q, k, b, h, off, scale);
      if (outside_distance(x, phi, range_lo, range_hi) > 0.0) flag_j = 1;
      const double f = exp(x - phi);
      den_j += f;
      for (int64_t i = 0; i < d; ++i) num_j[i] += f * load_v(s, v, off + i);
    }
    den += den_j;
    for (int64_t i = 0; i < d; ++i) num[i] += num_j[i];
    flagged_parts += flag_j;
    any |= flag_j;
  }
  if (rc == 0) {
    for (int64_t i = 0; i < d; ++i) out[i] = n > 0 ? num[i] / den : 0.0;
    *lse = n > 0 ? phi + log(den) : -INFINITY;
    *flag = (uint8_t)any;
    if (split_flags) *split_flags = flagged_parts;
  }
  free(num);
  free(num_j);
  return rc;
}

int64_t oracle_logits(const oracle_shape* s, const void* q, const void* k,
                      const int32_t* block_table, const int32_t* seq_lens, double scale,
                      double* out) {
  if (!shape_ok(s) || !q || !k || !seq_lens || !out) return -1;
  if (s->paged && !block_table) return -1;
  int64_t n = 0;
  for (int b = 0; b < s->batch; ++b) {
    if (seq_lens[b] < 0) return -1;
    for (int h = 0; h < s->num_q_heads; ++h) {
      const int kvh = kv_head_of(s, h);
      for (int64_t t = 0; t < seq_lens[b]; ++t) {
        const int64_t off = oracle_kv_offset(s, block_table, b, kvh, t);
        if (off < 0) return -1;
        out[n++] = logit(s, q, k, b, h, off, scale);
      }
    }
  }
  return n;
}
