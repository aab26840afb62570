/*
 * decode_attn.h -- C ABI of the GB300 (sm_103a) single-query decode-attention library.
 *
 * Computes, for every sequence b and query head h of a decode step,
 *     o[b,h] = softmax(scale * q[b,h] . K_b^T) V_b          (natural exp)
 *     lse[b,h] = ln sum_t exp(scale * q[b,h] . k_t)
 * over the first seq_lens[b] tokens of the sequence's KV cache. Sources (page, section):
 *   - "Flash-Decoding: Mathematical Foundations, Split-KV Parallelism, Online Softmax
 *     Reduction, and Serving Latency Optimization": "The Single-Token Generation
 *     Bottleneck" (the operation), "Mathematical Formulation of Split-KV Parallelism"
 *     (split partials O, m, l, L), "The Rescaling and Online Softmax Reduction Algorithm"
 *     (exact merge), "Production Implementation Guidelines" (split heuristics).
 *   - "FlashAttention and inference kernels": "PagedAttention" (block table), "A paged
 *     decode attention kernel (with GQA)" (cache layout, kernel signature, GQA mapping
 *     kv_head = h / (H_q / H_kv)), Exercise 3 (one read of a KV head serves its group).
 *   - "FlashDecoding++: Faster Large Language Model Inference on GPUs": "Asynchronized
 *     Softmax with Unified Max Value" (Eq. 3, Eq. 4) and "The Overflow Fallback:
 *     Recomputation" (Fig. 6: range check, synchronised recompute of flagged rows).
 *
 * Conventions for every entry point:
 *   - Device pointers are CUDA device (or managed) addresses on the device that is
 *     current when the call is made; host pointers are plain host memory.
 *   - The caller owns every buffer: inputs, outputs and the workspace. The library owns
 *     only the host-side plan object. decode_attn_run allocates nothing.
 *   - Return value: DA_OK (0) or a negative DA_ERR_* code; decode_attn_strerror gives a
 *     message (for DA_ERR_CUDA it includes the CUDA error text of the failing call on
 *     this thread). No exception crosses the ABI. Argument errors are detected on the
 *     host before anything is enqueued.
 *   - Work is enqueued on the given cudaStream_t (NULL = legacy default stream) and the
 *     call returns without synchronising, unless the problem's `validate` flag is set
 *     or a stats struct is requested: then the call synchronises the stream and reports
 *     device-side findings (bad block-table entries, bad lengths, pipeline timeouts).
 *   - Thread safety: plans are read-only after creation and may be shared between
 *     threads; one workspace must not be used by two runs that can overlap on the GPU.
 */
#ifndef DECODE_ATTN_H
#define DECODE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DECODE_ATTN_ABI_VERSION 4

/* Largest bin count decode_attn_logit_histogram accepts. */
#define DECODE_ATTN_MAX_HIST_BINS 32768

typedef enum { DA_F32 = 0, DA_F16 = 1, DA_BF16 = 2 } da_dtype;

/* DA_SOFTMAX_SYNC: each split runs the online-softmax recurrence with its running
 *   maximum ("FlashAttention and inference kernels", "FlashAttention: tiling plus online
 *   softmax"; FlashDecoding++ Eq. 2).
 * DA_SOFTMAX_UNIFIED: every split exponentiates against the one constant phi =
 *   unified_max, with no maximum and no rescaling (FlashDecoding++ Eq. 3 and Eq. 4). A
 *   scaled logit x with x - phi < range_lo or x - phi > range_hi (the interval is
 *   closed: a value on a bound is in range, as in Fig. 6) flags its row; flagged rows are
 *   recomputed in DA_SOFTMAX_SYNC mode on the device, in the same call ("The Overflow
 *   Fallback: Recomputation").
 * DA_SOFTMAX_UNIFIED_LOCAL: as DA_SOFTMAX_UNIFIED, with the same row flags, but without the
 *   second pass: a unified partial whose logits were all in range is an exact online-softmax
 *   state with maximum phi, so on its first out-of-range logit each split rescales its state
 *   to the true maximum so far and continues with the synchronised recurrence, reading no
 *   KV twice. An extension of the FlashDecoding++ fallback (the outputs equal the plain
 *   softmax either way). */
typedef enum {
  DA_SOFTMAX_SYNC = 0,
  DA_SOFTMAX_UNIFIED = 1,
  DA_SOFTMAX_UNIFIED_LOCAL = 2
} da_softmax_mode;

enum {
  DA_OK = 0,
  DA_ERR_INVALID_ARG = -1,          /* a null, misaligned or inconsistent argument */
  DA_ERR_UNSUPPORTED = -2,          /* head_dim, dtype, group size or page size not built */
  DA_ERR_WORKSPACE_TOO_SMALL = -3,  /* workspace_bytes below the plan's requirement */
  DA_ERR_BAD_BLOCK_TABLE = -4,      /* validate: a used block-table entry outside the pool */
  DA_ERR_CUDA = -5,                 /* a CUDA runtime / driver call failed */
  DA_ERR_DEVICE_TIMEOUT = -6,       /* validate: a device pipeline wait ran out of time */
  DA_ERR_BAD_SEQ_LEN = -7,          /* validate: seq_lens[b] < 0 or above the capacity */
  DA_ERR_HISTOGRAM_RANGE = -8,      /* choose_phi: a coverage tail lies outside [lo, hi) */
  DA_ERR_RANGE_TOO_WIDE = -9        /* choose_phi: covered range wider than max_width */
};

typedef struct {
  int batch;                /* B >= 1 sequences */
  int num_q_heads;          /* H_q */
  int num_kv_heads;         /* H_kv; H_q % H_kv == 0; group G = H_q / H_kv in {1,2,4,8} */
  int head_dim;             /* d in {64, 128} */
  int paged;                /* 1: k/v caches are [num_physical_blocks, page_size, H_kv, d]
                               addressed through block_table (FlashAttention and inference
                               kernels, "PagedAttention");
                               0: k/v caches are [batch, max_seq_len, H_kv, d] */
  int page_size;            /* paged: tokens per physical block, a power of two in [8, 256] */
  int max_blocks_per_seq;   /* paged: block_table row length */
  int num_physical_blocks;  /* paged: pool size; num_physical_blocks * page_size < 2^31 */
  int max_seq_len;          /* contiguous: token capacity per sequence;
                               batch * max_seq_len < 2^31 */
  da_dtype qkv_dtype;       /* storage of q, k_cache and v_cache (q only when kv_fp8) */
  da_dtype out_dtype;       /* storage of out (rounded to nearest even from fp32) */
  da_softmax_mode mode;
  float unified_max;        /* phi (natural-log units of the scaled logits); UNIFIED modes */
  float range_lo;           /* closed in-range interval on x - phi; range_lo < range_hi */
  float range_hi;
  int validate;             /* 1: every run synchronises and reports device findings */
  int num_sms;              /* 0: plan for the current device's SM count; > 0: plan for
                               that many SMs without touching CUDA (host-side planning) */
  /* FP8 KV cache ("FlashAttention and inference kernels", "A paged decode attention kernel
   * (with GQA)": the cache is BF16 or FP8, converted to FP32 in registers on read).
   * kv_fp8 = 1: k_cache and v_cache hold one-byte E4M3 codes (sign, 4-bit exponent with
   * bias 7, 3-bit mantissa, no infinities, S.1111.111 = NaN; "E4M3FN"), element for element
   * in the layout above, and code c stands for c * k_scale (K) or c * v_scale (V), scales
   * finite and > 0; q stays qkv_dtype, which must be DA_BF16 (else DA_ERR_UNSUPPORTED).
   * With groups of 4 query heads over an even number of KV heads, the plan packs pairs of KV
   * heads into one group of the split kernel where the step is large (at least four packed
   * groups per SM, or a cache capacity of 128 MiB and more); da_plan_info reports it.
   * The codes convert exactly; k_scale enters the logits' FP32 scale factor and v_scale the
   * output's. P . V runs on f16, so in the unified modes each split keeps its p = exp(x - phi)
   * within f16's range by a power-of-two factor per head, which only changes when its largest
   * logit grows past the range (the outputs and flags are those of the unified softmax).
   * NaN codes are not detected (they read as finite values). kv_fp8 = 0: k_cache and v_cache
   * are qkv_dtype; the scales are not read. */
  int kv_fp8;
  float k_scale;
  float v_scale;
  /* Test hook, 0 in normal use. k > 0: in every run of the plan, CTA 0's copy producer neither
   * arms nor fills ring stage k - 1 (no copy is issued for it) and every pipeline wait gives up
   * after 2 ms instead of 2 s, so that the consumers waiting for that stage run out of time:
   * the device records DA_ERR_DEVICE_TIMEOUT, the producer issues nothing more and drains the
   * copies it issued, and the run ends with unspecified outputs (with validate set, the call
   * returns DA_ERR_DEVICE_TIMEOUT). This exercises the bounded-wait path without a fault. */
  int debug_stall_stage;
} da_problem;

typedef struct da_plan da_plan;   /* opaque, host-owned, immutable after creation */

/* What a plan chose (host-side, no CUDA call). */
typedef struct {
  int grid_ctas;            /* persistent CTAs per launch */
  int num_splits;           /* 0: balanced shares (one contiguous share per CTA);
                               > 0: uniform splits per sequence */
  int unit_tokens;          /* split boundaries fall on multiples of this many tokens */
  int stage_tokens;         /* tokens per shared-memory pipeline stage */
  int stages;               /* pipeline depth */
  int recompute_splits;     /* uniform splits per flagged group in the recompute pass */
  int max_splits;           /* largest num_splits a run may ask for with this workspace */
  size_t workspace_bytes;   /* device workspace the runs need */
  size_t smem_bytes;        /* dynamic shared memory per CTA */
  int split_tokens;         /* largest split (piece of one sequence's KV head, in tokens) of a
                               step whose sequences are all at capacity, under the plan's
                               default policy ("the split size" of Flash-Decoding) */
  int split_tokens_min;     /* smallest such split */
  int kv_heads_per_group;   /* KV heads one split-kernel group reads together: 2 where an FP8
                               cache's groups of 4 query heads are packed in pairs of KV heads
                               (8 query heads fill the tensor-core consumer; see kv_fp8), else
                               1. Splits, partials and the merge are then per pair. */
} da_plan_info;

/* Filled by decode_attn_run when requested (forces a stream synchronisation). */
typedef struct {
  int grid_ctas;
  int num_splits;           /* as in da_plan_info, for this run */
  long long rows_flagged;   /* UNIFIED: (b, h) rows whose range check failed */
  long long splits_flagged; /* UNIFIED: (split, h) partials whose range check failed */
  int recompute_launched;   /* 1 iff the recompute kernel was enqueued (DA_SOFTMAX_UNIFIED) */
  int split_tokens;         /* largest split of this run's first pass, in tokens (the split
                               the heuristic chose, as the device cut it from seq_lens) */
  int split_tokens_min;     /* smallest split of this run's first pass, in tokens */
} da_stats;

/* Validate a problem and choose the launch (grid, split policy, pipeline) for it.
 * num_splits: 0 = heuristic (one balanced share of the whole step's KV tokens per
 * persistent CTA, which splits a sequence exactly when the SMs would otherwise idle:
 * the Flash-Decoding rule of splitting only when B * H under-fills the GPU, applied to
 * the work itself); > 0 = exactly that many uniform splits per sequence, each of
 * roundup(ceil(N_b / num_splits), unit) tokens ("Mathematical Formulation of Split-KV
 * Parallelism"). *workspace_bytes_out receives the workspace size the runs need.
 * Owns: *plan_out (free with decode_attn_destroy). Errors: INVALID_ARG, UNSUPPORTED,
 * CUDA (only when num_sms == 0 and the device query fails). */
int decode_attn_plan(const da_problem* problem, int num_splits, da_plan** plan_out,
                     size_t* workspace_bytes_out);

/* Copy what the plan chose into *info. Errors: INVALID_ARG. */
int decode_attn_plan_info(const da_plan* plan, da_plan_info* info);

/* Zero the part of the workspace that runs expect at zero and leave at zero (counters and the
 * flagged list). Required once for a new workspace before its first run (a zero-filled
 * allocation needs no call), and again after a run reported DA_ERR_DEVICE_TIMEOUT. Enqueued
 * on `stream`.
 * Errors: INVALID_ARG, WORKSPACE_TOO_SMALL, CUDA. */
int decode_attn_workspace_init(const da_plan* plan, void* workspace, size_t workspace_bytes,
                               void* cuda_stream);

/* Run one decode step.
 *   q           device, [batch, H_q, d] in qkv_dtype, 16-byte aligned.
 *   k_cache,    device, layout per problem->paged (see da_problem), qkv_dtype (E4M3 codes
 *   v_cache     when kv_fp8), 16-byte aligned.
 *   block_table device int32 [batch, max_blocks_per_seq] when paged (entries for the
 *               pages a sequence uses must lie in [0, num_physical_blocks); the rest are
 *               ignored, -1 by convention); must be NULL when contiguous.
 *   seq_lens    device int32 [batch], 0 <= seq_lens[b] <= capacity (paged:
 *               max_blocks_per_seq * page_size; contiguous: max_seq_len).
 *   scale       multiplier of q . k (1/sqrt(d) for standard attention).
 *   num_splits  -1 = the plan's choice; 0 = balanced shares; > 0 = uniform splits
 *               (at most the plan's max_splits).
 *   out         device, [batch, H_q, d] in out_dtype. A sequence with seq_lens[b] == 0
 *               gets out = 0 ("FlashAttention and inference kernels", Exercise 2 skips
 *               empty segments; an empty row is this library's extension of it).
 *   out_lse     nullable device float [batch, H_q]: natural-log log-sum-exp of the
 *               scaled logits (-inf for an empty sequence).
 *   row_flags   nullable device uint8 [batch, H_q]: UNIFIED: 1 iff the row's range check
 *               failed (its out/out_lse then come from the synchronised recompute);
 *               SYNC: 0.
 *   workspace   device, at least the plan's workspace_bytes, 256-byte aligned, zeroed
 *               before first use (decode_attn_workspace_init); left reusable.
 *   cuda_stream cudaStream_t or NULL.
 *   stats       nullable; when given the call synchronises and fills it.
 * Errors: INVALID_ARG, WORKSPACE_TOO_SMALL, CUDA, and with validate (or stats):
 * BAD_BLOCK_TABLE, BAD_SEQ_LEN, DEVICE_TIMEOUT. A bad block-table entry never makes the
 * device read outside the cache: the page reads as zeros. */
int decode_attn_run(const da_plan* plan, const void* q, const void* k_cache,
                    const void* v_cache, const int32_t* block_table, const int32_t* seq_lens,
                    float scale, int num_splits, void* out, float* out_lse,
                    uint8_t* row_flags, void* workspace, size_t workspace_bytes,
                    void* cuda_stream, da_stats* stats);

/* All arguments of one run, for decode_attn_run_ex. Fields as for decode_attn_run, plus:
 *   split_event_begin, split_event_end: nullable cudaEvent_t handles recorded on the
 *   stream immediately before and immediately after the split kernel's launch (before the
 *   recompute kernel), so a caller can time the split kernel alone with
 *   cudaEventElapsedTime. Both or neither must be given. */
typedef struct {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_table;
  const int32_t* seq_lens;
  float scale;
  int num_splits;
  void* out;
  float* out_lse;
  uint8_t* row_flags;
  void* workspace;
  size_t workspace_bytes;
  void* cuda_stream;
  da_stats* stats;
  void* split_event_begin;
  void* split_event_end;
} da_run_args;

/* decode_attn_run with its arguments in a struct and optional timing events.
 * Errors: as decode_attn_run; INVALID_ARG also when only one event is given. */
int decode_attn_run_ex(const da_plan* plan, const da_run_args* args);

/* Size of the fixed scratch region that decode_attn_run_static uses (8 MiB per device). */
#define DECODE_ATTN_STATIC_SCRATCH_BYTES (8u << 20)

/* Run one decode step without a caller-provided workspace. The papers and pages this
 * library follows have no counterpart to this entry point; it exists for callers that
 * cannot allocate device memory for a workspace:
 *   - a server whose device memory is reserved up front for the KV-cache pool;
 *   - a process under a device-memory cap, where a new allocation can fail in mid-step;
 *   - a decode loop that cannot afford cudaMalloc / cudaFree, which may synchronise the
 *     whole device;
 *   - plain C code with no device allocator of its own.
 * In place of a workspace it uses one fixed region of DECODE_ATTN_STATIC_SCRATCH_BYTES per
 * device, which belongs to the library's device code and is reserved when that code is
 * loaded on the device. The call itself allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library routine.
 *   Arguments as for decode_attn_run, less workspace and workspace_bytes.
 *   First call in a CUDA context: it looks up the region's device address in the context
 *   current on the calling thread (which can load the library's device code there) and
 *   caches it under that context's unique ID; a device reset or a caller's own driver
 *   context therefore gets a lookup of its own. Make the first call in each context before
 *   any stream capture.
 *   Each call first clears, on `cuda_stream`, the part of the region the plan's run expects
 *   at zero (counters and the flagged list), so runs of different plans may follow one another
 *   on a stream.
 *   Overlapping calls race: all calls on one device share the one region, so two calls
 *   whose work can overlap on the GPU (other streams, other host threads, other plans)
 *   corrupt each other's results. Serialise them, or use decode_attn_run with separate
 *   workspaces.
 *   Device findings (bad block-table entries or lengths, pipeline timeouts) are reported
 *   only through `stats` or the problem's `validate` flag: the region's status word is
 *   cleared by the next call.
 * Errors: as decode_attn_run; WORKSPACE_TOO_SMALL also when the plan's workspace_bytes
 * exceeds DECODE_ATTN_STATIC_SCRATCH_BYTES (use decode_attn_run with a workspace of that
 * size instead). Argument errors, including a plan whose kernel is not built, are detected
 * before anything is enqueued. */
int decode_attn_run_static(const da_plan* plan, const void* q, const void* k_cache,
                           const void* v_cache, const int32_t* block_table,
                           const int32_t* seq_lens, float scale, int num_splits, void* out,
                           float* out_lse, uint8_t* row_flags, void* cuda_stream,
                           da_stats* stats);

/* Synchronise `stream`, then read and clear the device findings recorded in the
 * workspace by earlier runs. Returns DA_OK or the first finding's DA_ERR_* code. */
int decode_attn_check_status(const da_plan* plan, void* workspace, void* cuda_stream);

/* Test hook: the element offset (into k_cache / v_cache) from which the device reads
 * token t of (sequence b, KV head kvh), computed by the same device code the kernel's
 * loads use. offsets_out: device int64 [batch, H_kv, T] with T = max_blocks_per_seq *
 * page_size (paged) or max_seq_len (contiguous); -1 for t >= seq_lens[b] and for a
 * block-table entry outside the pool. Enqueued on `stream`. Errors: INVALID_ARG, CUDA. */
int decode_attn_debug_gather(const da_plan* plan, const int32_t* block_table,
                             const int32_t* seq_lens, int64_t* offsets_out, void* cuda_stream);

/* ---- Calibration: choosing phi from the logits of a step --------------------------------
 * "FlashDecoding++: Faster Large Language Model Inference on GPUs", "The Overflow and
 * Precision Problem: Choosing phi" and Fig. 5: the logits of a model's attention rows stay in
 * a narrow range, profiled as a histogram over many inputs; phi is set to the lower end of
 * the range that holds more than 99.99% of them, and where that range is too wide (OPT-6.7B
 * in Fig. 5) the unified max is not used. These two calls run that profile on the caller's
 * own steps: accumulate one histogram over as many steps as wanted, then read phi off it.
 * Neither is on the attention path. */

/* Histogram of the scaled logits x = scale * q[b,h] . k_t of one step, over every query head
 * h and every token t < seq_lens[b] of every sequence b, read through the plan's layout
 * (contiguous or block table, GQA mapping kv_head = h / G) as decode_attn_run reads them.
 *   plan: any plan of the problem shape; its softmax mode, phi and range are not used.
 *   q, k_cache, block_table, seq_lens, scale: as for decode_attn_run (device; k_cache
 *     16-byte aligned). v_cache is not read.
 *   lo, hi, nbins: nbins equal bins over [lo, hi), lo < hi finite, 1 <= nbins <=
 *     DECODE_ATTN_MAX_HIST_BINS. x falls in bin i = floor((x - lo) * (nbins / (hi - lo))),
 *     evaluated in fp32 from an fp32 dot product, so a logit within a few fp32 ulps of a bin
 *     edge may fall on either side of it.
 *   counts: device uint64 [nbins + 2], 8-byte aligned, ACCUMULATED into (zero it before the
 *     first step): counts[0] = values below lo, counts[1 + i] = bin i, counts[nbins + 1] =
 *     values at or above the top edge, and NaN.
 * A token whose block-table entry lies outside the pool, and tokens past the capacity, are
 * not counted: the counts then sum to less than H_q * sum_b min(seq_lens[b], capacity), which
 * the caller can check. Enqueued on `stream`; not synchronised.
 * For an FP8 cache (kv_fp8) the logits are scale * q . (code * k_scale), as decode_attn_run
 * forms them. Errors: INVALID_ARG (null or misaligned pointer, bad range or bin count),
 * UNSUPPORTED, CUDA. */
int decode_attn_logit_histogram(const da_plan* plan, const void* q, const void* k_cache,
                                const int32_t* block_table, const int32_t* seq_lens,
                                float scale, float lo, float hi, int nbins,
                                unsigned long long* counts, void* cuda_stream);

/* Host only: phi and the covered logit range from a histogram laid out as above.
 *   counts: HOST uint64 [nbins + 2]; nbins, lo, hi: those the histogram was taken with.
 *   coverage: the fraction of values the range must hold, in (0, 1] (0.9999 in Fig. 5).
 *     At most floor((1 - coverage) * total / 2) values are left out on each side, whole bins
 *     at a time, so the range is bin-aligned and holds at least that fraction.
 *   max_width: the widest covered range (x_hi - x_lo) for which the unified max is used.
 *   x_lo, x_hi (out): the covered range, bin edges rounded outwards to fp32.
 *   phi (out): x_lo, the pages' choice (the lower bound: a value below it underflows
 *     harmlessly, none in range overflows). With it, the in-range interval on x - phi of
 *     the covered values is [0, x_hi - x_lo]; da_problem's [range_lo, range_hi] may be set
 *     wider, to what fp32 tolerates, so that only values that would lose precision or
 *     overflow flag their rows.
 * Errors: INVALID_ARG (null pointer, empty histogram, bad coverage, range or max_width);
 * HISTOGRAM_RANGE (more than a tail's share of values lies below lo or at or above hi:
 * repeat the histogram over a wider [lo, hi); outputs not written); RANGE_TOO_WIDE (outputs
 * written, but x_hi - x_lo > max_width: the unified max does not apply to this data, use
 * DA_SOFTMAX_SYNC, as Fig. 5 does for OPT-6.7B). Touches no device. */
int decode_attn_choose_phi(const unsigned long long* counts, int nbins, float lo, float hi,
                           double coverage, float max_width, float* phi, float* x_lo,
                           float* x_hi);

void decode_attn_destroy(da_plan* plan);

const char* decode_attn_strerror(int code);

int decode_attn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DECODE_ATTN_H */
