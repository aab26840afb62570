// da_device.cuh -- launch parameters, shared-memory layout and sm_103a PTX helpers of the
// decode-attention kernels (TMA tensor loads, bulk copies, mbarriers, programmatic
// dependent launch, exp2 / log2, packed FP32 FMA).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace da {

// ---- fixed kernel geometry ------------------------------------------------------------
constexpr int kConsumerWarps = 8;                       // compute warps per CTA (2 warpgroups)
constexpr int kThreads = (kConsumerWarps + 4) * 32;     // + a producer warpgroup (1 working warp)
constexpr int kLaunchRegs = 168;                        // 65536 / 384, rounded to 8
constexpr int kConsumerRegs = 216;                      // after setmaxnreg.inc
constexpr int kProducerRegs = 72;                       // after setmaxnreg.dec
static_assert(kConsumerWarps * 32 * kConsumerRegs + 4 * 32 * kProducerRegs <=
                  (kConsumerWarps + 4) * 32 * kLaunchRegs,
              "the register split must fit the launch allocation");
constexpr int kTokensPerWarp = 8;                       // KV rows a consumer warp takes per stage
constexpr int kStageTokens = kConsumerWarps * kTokensPerWarp;   // 64 KV rows per stage
constexpr int kMaxStages = 8;
constexpr int kMaxBatchSmem = 2048;                     // balanced schedule keeps B lengths in smem
constexpr uint32_t kSmemLimit = 232448;                 // 227 KB opt-in per CTA
constexpr int kMinUnitsPerCta = 8;                      // no share below 8 units (128 tokens)
// Balanced shares charge every piece this many K+V bytes on top of its tokens: a piece ends
// with an in-CTA combine during which the CTA's copy stream stalls (about 2 us, measured as
// the end-time slope of CTAs over their piece counts), so CTAs whose share spans many short
// sequences would otherwise finish last.
constexpr int kPieceCostBytes = 96 * 1024;

// status bits recorded by the device in the workspace
constexpr int kStatusBadBlockTable = 1;
constexpr int kStatusBadSeqLen = 2;
constexpr int kStatusTimeout = 4;

// bound on any pipeline wait (ns); a healthy wait lasts microseconds
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
// the bound while the test hook that stalls a stage is on
constexpr unsigned long long kTestWaitLimitNs = 2000000ull;

enum Policy { kBalanced = 0, kUniform = 1 };
// Softmax modes, numbered as the C ABI's da_softmax_mode.
enum SoftmaxMode { kSoftmaxSync = 0, kSoftmaxUnified = 1, kSoftmaxUnifiedLocal = 2 };
enum OutType { kOutF32 = 0, kOutF16 = 1, kOutBF16 = 2 };

// FP8 storage of K and V: one E4M3 code per element (sign, 4-bit exponent with bias 7, 3-bit
// mantissa; no infinities), standing for code * k_scale or code * v_scale. q stays bf16.
// HP > 1: the split kernel's view of such a cache in which each group packs the query heads of
// HP consecutive KV heads (a TMA box then holds HP rows of every token, see Cfg::kHp).
template <int HP>
struct fp8e4m3_heads {
  uint8_t bits;
};
using fp8e4m3 = fp8e4m3_heads<1>;
template <typename T>
struct QOf {   // q's storage type for a K / V storage type
  using type = T;
};
template <int HP>
struct QOf<fp8e4m3_heads<HP>> {
  using type = __nv_bfloat16;
};
template <typename T>
struct KvHeads {   // KV heads per group of the split kernel, and whether the cache is FP8
  static constexpr int value = 1;
  static constexpr bool fp8 = false;
};
template <int HP>
struct KvHeads<fp8e4m3_heads<HP>> {
  static constexpr int value = HP;
  static constexpr bool fp8 = true;
};

struct Params {
  const void* q;                 // [B, Hq, D]
  const int32_t* block_table;    // [B, max_blocks] (paged)
  const int32_t* seq_lens;       // [B]
  void* out;                     // [B, Hq, D] out dtype
  float* out_lse;                // [B, Hq] or null
  uint8_t* row_flags;            // [B, Hq] or null
  int32_t* counters;             // [n_groups] arrivals per group (self-cleaning)
  int32_t* flag_list;            // [n_groups] flagged groups (unified mode)
  int32_t* list_state;           // unified: [0] flagged count, [1] recompute CTAs finished
                                 // (self-cleaning)
  int32_t* status;               // device findings
  unsigned long long* stats;     // [0] rows flagged, [1] split partials flagged, [2] largest
                                 // piece (tokens), [3] 2^31 - 1 - smallest piece (tokens)
  uint32_t* part_flags;          // [slots] range-check bits per head
  float* part_l;                 // [slots, G] log2-domain LSE of each partial
  float* part_o;                 // [slots, G, D] normalised partial outputs
  int64_t* debug_offsets;        // debug gather output
  int batch, hq, hkv, group, head_dim;
  int paged, page_size, max_blocks, num_blocks, max_seq_len;
  int capacity;                  // token capacity of one sequence
  int unit;                      // split boundaries fall on multiples of this many tokens
  int piece_units;               // balanced: cost units charged per group ahead of its tokens
  int box_tokens;                // KV rows per TMA box
  int out_dtype;
  int policy;                    // kBalanced / kUniform
  int num_splits;                // uniform: splits per group
  int recompute;                 // 1: the recompute launch (groups from the flagged list)
  int list_flags;                // 1: flagged groups go to the list (a recompute launch follows)
  int piece_stats;               // 1: record the largest and smallest piece in stats[2..3]
  unsigned long long wait_limit_ns;   // bound on every pipeline wait
  int stall_stage;               // test hook: 0, or k + 1: CTA 0's producer neither arms nor
                                 // fills ring stage k, so that its consumers' wait runs out
  int narrow;                    // 1: every product of the schedule's unit / item arithmetic
                                 // (index x CTA count) is below 2^31: 32-bit division suffices
  int n_groups;                  // B * Hkv
  int stages;                    // pipeline depth
  int batch_smem;                // lengths held in smem (balanced) or 0
  float qscale;                  // scale * log2(e) (* k_scale): logits in log2 units
  float v_scale;                 // FP8 V: the outputs' factor (1 otherwise)
  float phi2, lo2, hi2;          // unified constant and range bounds, log2 units
};

// ---- shared-memory layout (host and device compute it identically) ------------------------
struct Layout {
  uint32_t stage_bytes, k_off, v_off, q_off;
  uint32_t bar_off, wbuf_off, mm_off, ml_off, mflag_off, lens_off, prefix_off, misc_off;
  uint32_t total;
};

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// Split kernels whose consumers run on the tensor cores (see da_mma.cuh), in every softmax
// mode: bf16 or FP8 caches (es: K / V bytes per element), groups of 1, 2, 4 or 8 query heads.
// bf16 tiles are TMA-loaded with the 128-byte swizzle (4-D view: 64-element rows, d / 64 of
// them per token, heads, tokens); FP8 tiles as rows of d bytes (3-D view), with the 128-byte
// swizzle when d = 128. f16 caches keep the CUDA-core consumers: with P in f16 the unified
// phase needs a rescaled P . V per tile, which measured slower than the CUDA-core path on the
// MHA workload; f32 caches have no 16-bit MMA operand at all.
__host__ __device__ constexpr bool uses_mma(int es, bool is_f16, int G) {
  return (es == 1 || (es == 2 && !is_f16)) && (G == 1 || G == 2 || G == 4 || G == 8);
}

// Geometry of a consumer warp's logit transpose: a KV row of D elements of es bytes is split
// over lg_lanes lanes (16 bytes each); a warp has 32 / lg_lanes lane groups of 8 / that many
// rows, so each lane group produces v = G * rows partial-sum rows to transpose.
__host__ __device__ constexpr int tp_lanes(int D, int es) { return D / (16 / es); }
__host__ __device__ constexpr int tp_values(int D, int G, int es) {
  return G * (kTokensPerWarp / (32 / tp_lanes(D, es)));
}
__host__ __device__ constexpr int tp_row_stride(int D, int es) { return tp_lanes(D, es) + 4; }
// One lane group's block: v rows of row_stride floats, rounded to 32 floats, plus lg_lanes so
// that the groups' rows fall on different banks.
__host__ __device__ constexpr int tp_group_floats(int D, int G, int es) {
  return (tp_values(D, G, es) * tp_row_stride(D, es) + 31) / 32 * 32 + tp_lanes(D, es);
}
// Per-warp scratch (floats): the transpose, the (p, p) pairs and, at a piece's end, the
// warp's accumulators share it (they are never live at the same time).
__host__ __device__ constexpr int warp_scratch_floats(int D, int G, int es) {
  const int tp = (32 / tp_lanes(D, es)) * tp_group_floats(D, G, es);
  const int pairs = 2 * 2 * kTokensPerWarp * G;   // (p, p) pairs of two batches
  const int acc = G * D;
  const int m = tp > pairs ? (tp > acc ? tp : acc) : (pairs > acc ? pairs : acc);
  return (m + 3) / 4 * 4;
}

// es: q's bytes per element (also the consumer scratch geometry's); kv_es: K / V's (0: es);
// hp: KV heads per group, whose rows a stage holds for every token.
__host__ __device__ inline Layout make_layout(int D, int G, int es, int stages, int batch_smem,
                                              int kv_es = 0, int hp = 1) {
  Layout L;
  const uint32_t kv = (uint32_t)kStageTokens * D * (kv_es ? kv_es : es) * (uint32_t)hp;
  L.k_off = 0;
  L.v_off = kv;
  L.q_off = 2 * kv;
  L.stage_bytes = align_up(2 * kv + (uint32_t)G * D * es, 1024);   // swizzled tiles: 1 KB
  uint32_t off = (uint32_t)stages * L.stage_bytes;
  L.bar_off = off;
  off += 2u * stages * 8u;
  off = align_up(off, 16);
  L.wbuf_off = off;
  off += (uint32_t)kConsumerWarps * warp_scratch_floats(D, G, es) * 4u;
  L.mm_off = off;
  off += (uint32_t)kConsumerWarps * G * 4u;
  L.ml_off = off;
  off += (uint32_t)kConsumerWarps * G * 4u;
  L.mflag_off = off;
  off += (uint32_t)kConsumerWarps * 4u;
  off = align_up(off, 16);
  L.lens_off = off;
  off += (uint32_t)batch_smem * 4u;
  L.prefix_off = off;
  off += (uint32_t)(batch_smem + 1) * 4u;
  off = align_up(off, 16);
  L.misc_off = off;
  off += 16;
  L.total = off + 1024;   // slack for aligning the dynamic smem base to 1024 bytes
  return L;
}

#ifdef __CUDACC__
// ---- PTX helpers ---------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of `parity` to complete, for at most `limit_ns`. Returns false on
// timeout (the caller records it and degrades to a non-waiting completion).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ uint64_t make_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled TMA load of a box into shared memory, completing on `bar` by transaction bytes.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y, int z, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)),
      "l"(policy)
      : "memory");
}

// 4-D tiled TMA load (the swizzled [tokens, heads, d / 64, 64] view of a cache).
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y, int z, int w, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar)),
      "l"(policy)
      : "memory");
}

// Contiguous bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Atomic add with acquire-release semantics at GPU scope. After a CTA barrier, one thread's
// call releases every write the CTA made before the barrier and acquires every write that
// other CTAs released before their own calls on the same counter.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int32_t* addr, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(addr), "r"(v)
               : "memory");
  return old;
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two FP32 values held in one 64-bit register pair, operated on by the packed FP32
// instructions (fma/mul/add .f32x2). Keeping operands in this form end to end lets every
// packed instruction take its registers directly, with no packing moves.
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 f2_pack(float a, float b) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ f32x2 f2_pack_bits(uint32_t a, uint32_t b) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(f32x2 v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ void f2_fma(f32x2& d, f32x2 a, f32x2 b) {   // d = a * b + d
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}
__device__ __forceinline__ f32x2 f2_mul(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Two E4M3 codes (the low 16 bits of c; the lower code lands in the lower half) -> f16x2.
// Every E4M3 value is a normal binary16 number or zero, so the conversion is exact. (A NaN
// code converts to a NaN; caches hold none.)
// Four E4M3 codes (bytes 0..3 of c) -> two f16x2: lo from bytes 0, 1, hi from bytes 2, 3.
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t c, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, a;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(c));
}

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t c) {
  uint32_t h;
  asm("{\n\t.reg .b16 lo;\n\tcvt.u16.u32 lo, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
      : "=r"(h)
      : "r"(c));
  return h;
}

// ---- element conversion of one 16-byte chunk to FP32 ------------------------------------
template <typename T>
struct Elem;

template <>
struct Elem<float> {
  static constexpr int kPerChunk = 4;
  __device__ __forceinline__ static void to_pairs(const uint4 c, f32x2* f) {
    f[0] = f2_pack_bits(c.x, c.y);
    f[1] = f2_pack_bits(c.z, c.w);
  }
  __device__ __forceinline__ static void to_f32(const uint4 c, float* f) {
    f[0] = __uint_as_float(c.x);
    f[1] = __uint_as_float(c.y);
    f[2] = __uint_as_float(c.z);
    f[3] = __uint_as_float(c.w);
  }
};

template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kPerChunk = 8;
  __device__ __forceinline__ static void to_pairs(const uint4 c, f32x2* f) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = f2_pack_bits(w[i] << 16, w[i] & 0xffff0000u);
  }
  // bfloat16 is the upper half of a binary32: widening is a shift / mask.
  __device__ __forceinline__ static void to_f32(const uint4 c, float* f) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};

template <>
struct Elem<__half> {
  static constexpr int kPerChunk = 8;
  __device__ __forceinline__ static void to_pairs(const uint4 c, f32x2* f) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h;
      memcpy(&h, &w[i], 4);
      const float2 v = __half22float2(h);
      f[i] = f2_pack(v.x, v.y);
    }
  }
  __device__ __forceinline__ static void to_f32(const uint4 c, float* f) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h;
      memcpy(&h, &w[i], 4);
      const float2 v = __half22float2(h);
      f[2 * i] = v.x;
      f[2 * i + 1] = v.y;
    }
  }
};

__device__ __forceinline__ void store_out(void* out, int64_t idx, int type, float v) {
  if (type == kOutF32)
    static_cast<float*>(out)[idx] = v;
  else if (type == kOutF16)
    static_cast<__half*>(out)[idx] = __float2half_rn(v);
  else
    static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
}

// Token t of sequence b -> row coordinate z of the [tokens, Hkv, D] view of the cache
// ("FlashAttention and inference kernels", "PagedAttention": slot t % page of physical
// block block_table[t / page]). `entry` is the block-table entry for t's page (paged).
// Returns -1 for an entry outside the pool.
__device__ __forceinline__ int token_row(const Params& p, int b, int t, int entry) {
  if (p.paged) {
    if (entry < 0 || entry >= p.num_blocks) return -1;
    return entry * p.page_size + (t & (p.page_size - 1));
  }
  return b * p.max_seq_len + t;
}
#endif  // __CUDACC__

}  // namespace da
