// da_kernel.cuh -- the split-KV decode-attention kernel for sm_103a.
//
// One persistent CTA per SM walks a list of "pieces": (sequence b, KV head kvh, token
// range [t0, t1)); for an FP8 cache packed in pairs, kvh names a pair of KV heads (Cfg::kHp).
// A piece is one Flash-Decoding split ("Flash-Decoding: Mathematical
// Foundations, ...", "Mathematical Formulation of Split-KV Parallelism"): it yields the
// partial output O, the maximum m and the sum l for all G query heads of its KV head at
// once, so each KV row is read from HBM once for the whole group ("FlashAttention and
// inference kernels", Exercise 3).
//
// Warp roles (12 warps; `setmaxnreg` moves registers from the producer warpgroup to the
// consumers):
//   warps 8..11 producers: two (contiguous cache) or four (paged cache) of them TMA-load
//               64-row K and V tiles (and, per piece, the group's q) into a ring of
//               shared-memory stages; paged caches are gathered through the block table one
//               page per TMA box ("PagedAttention").
//   warps 0..7  consumers: each takes 8 rows of every stage. For bf16 and FP8 caches the
//               logits and P . V run on the tensor cores (da_mma.cuh). Otherwise a row of
//               d elements is split over a lane group (16 lanes for d = 128 in 16-bit types,
//               16-byte chunks per lane); q . k partial sums for all heads and rows of the
//               lane group are completed by a transpose-reduce through shared memory that
//               leaves whole (row, head) logits per lane. Softmax:
//                 SYNC    -- online softmax with the running maximum per head, rescaling
//                            the accumulators by exp(m_old - m_new) ("FlashAttention:
//                            tiling plus online softmax");
//                 UNIFIED -- exp(x - phi) against the one constant phi, no maximum, no
//                            rescaling, and a range check of x - phi against the closed
//                            interval [lo, hi] (FlashDecoding++, Eq. 3, Eq. 4, Fig. 6).
//               P . V then accumulates into per-lane FP32 registers.
// At a piece's end the 8 consumer warps' states are combined in shared memory into one
// partial (normalised O, L = m + log l). A group covered by a single piece is written out
// directly; otherwise the partial goes to the workspace and the CTA that completes the
// group's last piece (an atomic arrival counter, no waiting) performs the exact log-sum-exp
// merge ("The Rescaling and Online Softmax Reduction Algorithm").
//
// All exponentials are base 2: q is pre-multiplied by scale * log2(e), and log-sum-exps
// are converted back to natural log on output.
#pragma once

#include <type_traits>

#include "da_device.cuh"
#include "da_mma.cuh"

namespace da {

template <typename T, int D, int G>
struct Cfg {
  using Q = typename QOf<T>::type;                    // q's storage (bf16 over FP8 K / V)
  static constexpr bool kFp8 = KvHeads<T>::fp8;
  static constexpr int kHp = KvHeads<T>::value;         // KV heads per group (packed FP8: 2)
  static constexpr int kEs = sizeof(T);                 // K / V bytes per element
  static constexpr int kQEs = sizeof(Q);
  static constexpr int kEpl = 16 / kEs;               // elements per 16-byte chunk
  static constexpr int kLg = D / kEpl;                // lanes per KV row (lane group)
  static constexpr int kNlg = 32 / kLg;               // lane groups per warp
  static constexpr int kT = kTokensPerWarp / kNlg;    // rows per lane group per stage
  static constexpr int kV = G * kT;                   // logits per lane group per stage
  static constexpr int kNv = kV >= kLg ? kV / kLg : 1;    // complete logits per lane
  static constexpr int kRep = kV >= kLg ? 1 : kLg / kV;   // lanes that hold the same logit
  static constexpr int kRowBytes = D * kEs;             // one KV head's row of a token
  static constexpr int kTokBytes = kRowBytes * kHp;     // a token's rows in a stage tile
  static constexpr int kQBytes = G * D * kQEs;
  static_assert(kLg >= 1 && kLg <= 32 && (32 % kLg) == 0, "a row must span a lane group");
  static_assert((kTokensPerWarp % kNlg) == 0, "rows per warp must split over lane groups");
  static_assert((kV & (kV - 1)) == 0, "logit count must be a power of two");
  static_assert((kQBytes % 16) == 0, "q bulk copy must be a multiple of 16 bytes");
};

struct Piece {
  int g, b, kvh;
  int t0, t1;        // token range of this piece
  int nslots;        // pieces of the group (1: write the output directly)
  int slot_base;     // partial index of the group's first piece
  int slot;          // this piece's partial index
};

struct Sched {
  int policy;
  long long u, u1, W;    // balanced: unit cursor, end, total units
  int P, c;
  long long i, i1;       // uniform: item cursor, end
  int S;
  bool use_list;         // uniform: item i / S indexes the flagged list, not the groups
  bool first_phase;      // the step's first pass (flags, statistics, flagged list)
  const int* lens;       // balanced: clamped lengths (smem)
  const int* prefix;     // balanced: exclusive prefix of per-head units (cost + tokens) (smem)
};

__device__ __forceinline__ int clamp_len(const Params& p, int n) {
  return n < 0 ? 0 : (n > p.capacity ? p.capacity : n);
}

// CTA whose balanced share [floor(c W / P), floor((c + 1) W / P)) holds unit u. I is the
// integer type of the unit space: 32-bit when the host found every product below 2^31 (no
// calls to the 64-bit division routine on the paths that start the step), else 64-bit.
template <typename I>
__device__ __forceinline__ I cta_of(I u, I W, I P) {
  return ((u + 1) * P - 1) / W;
}

// Balanced shares. Group g of sequence b owns units [gs, ge) of the step's unit space:
// piece_units cost units, then one per `unit` tokens. A share that holds only cost units of a
// group has no piece of it.
template <typename I>
__device__ __forceinline__ bool sched_balanced(Sched& s, const Params& p, Piece& pc) {
  const I u1 = (I)s.u1, W = (I)s.W, P = (I)s.P, hkv = (I)p.hkv, pu = (I)p.piece_units;
  I u = (I)s.u;
  while (u < u1) {
    int lo = 0, hi = p.batch;   // invariant: hkv * prefix[lo] <= u < hkv * prefix[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (hkv * (I)s.prefix[mid] <= u) lo = mid; else hi = mid;
    }
    const int b = lo;
    const I nb = (I)(s.prefix[b + 1] - s.prefix[b]);
    const I base = hkv * (I)s.prefix[b];
    const int kvh = (int)((u - base) / nb);
    const I gs = base + (I)kvh * nb, ge = gs + nb;
    const I rs = gs + pu;   // the group's first token unit
    const I pe = u1 < ge ? u1 : ge;
    const I u_at = u;
    u = pe;
    if (pe <= rs) continue;
    s.u = (long long)u;
    const I n = (I)s.lens[b];
    pc.b = b;
    pc.kvh = kvh;
    pc.g = b * p.hkv + kvh;
    pc.t0 = (int)(((u_at > rs ? u_at : rs) - rs) * (I)p.unit);
    const I t1 = (pe - rs) * (I)p.unit;
    pc.t1 = (int)(t1 < n ? t1 : n);
    const I cf = cta_of<I>(rs, W, P), cl = cta_of<I>(ge - 1, W, P);
    pc.nslots = (int)(cl - cf + 1);
    pc.slot_base = (int)cf + pc.g;
    pc.slot = s.c + pc.g;
    return true;
  }
  s.u = (long long)u;
  return false;
}

__device__ __forceinline__ bool sched_next(Sched& s, const Params& p, Piece& pc) {
  if (s.policy == kBalanced)
    return p.narrow ? sched_balanced<unsigned>(s, p, pc) : sched_balanced<long long>(s, p, pc);
  if (s.i >= s.i1) return false;
  const long long i = s.i++;
  const int li = p.narrow ? (int)((unsigned)i / (unsigned)s.S) : (int)(i / s.S);
  const int sp = (int)(i - (long long)li * s.S);
  const int g = s.use_list ? __ldcg(p.flag_list + li) : li;
  const int b = g / p.hkv;
  const int n = clamp_len(p, __ldg(p.seq_lens + b));
  const int ts = n == 0 ? 0 : ((n + s.S - 1) / s.S + p.unit - 1) / p.unit * p.unit;
  const long long t0 = (long long)sp * ts < n ? (long long)sp * ts : n;
  const long long t1 = t0 + ts < n ? t0 + ts : n;
  pc.g = g;
  pc.b = b;
  pc.kvh = g - b * p.hkv;
  pc.t0 = (int)t0;
  pc.t1 = (int)t1;
  pc.nslots = s.S;
  pc.slot_base = g * s.S;
  pc.slot = g * s.S + sp;
  return true;
}

// ---- producer warps ------------------------------------------------------------------
// Copies are issued by two warps (part 0: K and q, part 1: V) for a contiguous cache and by
// four for a paged one (parts 2 and 3 take every other page box): one warp's TMA issue rate
// cannot keep up with a stage made of several small page boxes.
// `abort`: set by a consumer warp whose wait ran out; the producer then issues nothing more (a
// stage the consumers released without waiting for it may still have copies in flight into its
// slot) and leaves after draining the copies it issued.
template <typename T, int D, int G, bool SWZ>
__device__ __forceinline__ void run_producer(const Params& p, Sched s, uint8_t* stages,
                                             const Layout& L, uint64_t* full, uint64_t* empty,
                                             const CUtensorMap* tmk, const CUtensorMap* tmv,
                                             int lane, int part, const int* abort) {
  using C = Cfg<T, D, G>;
  const uint64_t pol = make_evict_first_policy();
  const uint32_t NS = (uint32_t)p.stages;
  const int nsub = p.paged ? 2 : 1;   // warps per tensor: K from even parts, V from odd
  uint32_t k = 0;
  bool dead = false;
  uint32_t issued = 0;   // one past the last stage this call issued copies for
  Piece pc;
  while (sched_next(s, p, pc)) {
    if (pc.t1 <= pc.t0) continue;
    const int32_t* trow = p.paged ? p.block_table + (long long)pc.b * p.max_blocks : nullptr;
    const char* qsrc = static_cast<const char*>(p.q) +
                       ((long long)pc.b * p.hq + (long long)pc.kvh * G) * D * C::kQEs;
    // Block-table entries of pages [wbase, wbase + 32) (win) and [wbase + 32, wbase + 64)
    // (wnext), one per lane; wnext is loaded a window ahead of its first use.
    int wbase = -(1 << 30);
    int32_t win = -1, wnext = -1;
    for (int ts = pc.t0, j = 0; ts < pc.t1; ts += kStageTokens, ++j, ++k) {
      const uint32_t slot = k % NS, ph = (k / NS) & 1u;
      if (!dead && !mbar_wait(&empty[slot], ph ^ 1u, p.wait_limit_ns)) {
        dead = true;
        if (lane == 0) atomicOr(p.status, kStatusTimeout);
      }
      if (!dead && *reinterpret_cast<const volatile int*>(abort) != 0) dead = true;
      dead = __any_sync(0xffffffffu, dead);   // several lanes issue copies: agree on it
      if (!dead) issued = k + 1;
      // test hook: this stage is neither armed nor filled
      const bool skip = dead || (p.stall_stage != 0 && blockIdx.x == 0 &&
                                 k == (uint32_t)(p.stall_stage - 1));
      const int n = min(kStageTokens, pc.t1 - ts);
      uint8_t* st = stages + slot * L.stage_bytes;
      if (p.paged) {
        // Lane l of this warp owns box l * nsub + part / 2 of the stage, if there is one (a
        // stage spans at most 64 / box pages, so every page of it lies in the two windows
        // once the first one does).
        const int box = p.box_tokens;
        const int nbox = (n + box - 1) / box;
        const int first = ts / p.page_size;   // warp-uniform
        if (first >= wbase + 64 || first < wbase) {
          wbase = first & ~31;
          const int i0 = wbase + lane, i1 = wbase + 32 + lane;
          win = i0 < p.max_blocks ? __ldg(trow + i0) : -1;
          wnext = i1 < p.max_blocks ? __ldg(trow + i1) : -1;
        } else if (first >= wbase + 32) {
          wbase += 32;
          win = wnext;
          const int i1 = wbase + 32 + lane;
          wnext = i1 < p.max_blocks ? __ldg(trow + i1) : -1;
        }
        const int bi = lane * nsub + (part >> 1);   // the box this lane issues, if < nbox
        const int mine = min(bi, nbox - 1);
        const int t = ts + mine * box;
        const int rel = t / p.page_size - wbase;   // 0 <= rel < 64
        const int e0 = __shfl_sync(0xffffffffu, win, rel & 31);
        const int e1 = __shfl_sync(0xffffffffu, wnext, rel & 31);
        int z = token_row(p, pc.b, t, rel < 32 ? e0 : e1);
        if (z < 0) {
          if (bi < nbox) atomicOr(p.status, kStatusBadBlockTable);
          z = p.num_blocks * p.page_size;   // past the pool: the box reads as zeros
        }
        if (part == 0 && lane == 0 && !skip) {
          const uint32_t bytes =
              (uint32_t)nbox * box * C::kTokBytes * 2u + (j == 0 ? (uint32_t)C::kQBytes : 0u);
          mbar_arrive_expect_tx(&full[slot], bytes);
          if (j == 0) bulk_load(st + L.q_off, qsrc, C::kQBytes, &full[slot]);
        }
        __syncwarp();
        if (bi < nbox && !skip) {
          const uint32_t off = ((part & 1) == 0 ? L.k_off : L.v_off) + bi * box * C::kTokBytes;
          const CUtensorMap* tm = (part & 1) == 0 ? tmk : tmv;
          if constexpr (SWZ)
            tma_load_4d(st + off, tm, &full[slot], 0, 0, pc.kvh, z, pol);
          else
            tma_load_3d(st + off, tm, &full[slot], 0, pc.kvh * C::kHp, z, pol);
        }
      } else if (lane == 0 && !skip) {
        const int z = pc.b * p.max_seq_len + ts;
        if (part == 0) {
          const uint32_t bytes =
              (uint32_t)kStageTokens * C::kTokBytes * 2u + (j == 0 ? (uint32_t)C::kQBytes : 0u);
          mbar_arrive_expect_tx(&full[slot], bytes);
          if (j == 0) bulk_load(st + L.q_off, qsrc, C::kQBytes, &full[slot]);
        }
        const uint32_t off = part == 0 ? L.k_off : L.v_off;
        const CUtensorMap* tm = part == 0 ? tmk : tmv;
        if constexpr (SWZ)
          tma_load_4d(st + off, tm, &full[slot], 0, 0, pc.kvh, z, pol);
        else
          tma_load_3d(st + off, tm, &full[slot], 0, pc.kvh * C::kHp, z, pol);
      }
      __syncwarp();
    }
  }
  // Never leave with copies in flight: wait (bounded) for the last issued stages to land,
  // after a timeout too.
  if (lane == 0) {
    const uint32_t first = issued > NS ? issued - NS : 0u;
    for (uint32_t kk = first; kk < issued; ++kk)
      mbar_wait(&full[kk % NS], (kk / NS) & 1u, p.wait_limit_ns);
  }
}

// ---- consumer warps ---------------------------------------------------------------------
// Per-lane constants of the logit layout after the transpose-reduce.
template <typename T, int D, int G>
struct LaneMap {
  using C = Cfg<T, D, G>;
  int lg, li, row0;              // lane group, lane in group, first stage row of the group
  int j[C::kNv], g[C::kNv];      // token (within the lane group) and head of each logit
  bool writer;                   // the lane that publishes a replicated logit
  __device__ __forceinline__ LaneMap(int warp, int lane) {
    lg = lane / C::kLg;
    li = lane % C::kLg;
    row0 = warp * kTokensPerWarp + lg * C::kT;
#pragma unroll
    for (int i = 0; i < C::kNv; ++i) {
      const int idx = C::kV >= C::kLg ? li * C::kNv + i : li / C::kRep;
      j[i] = idx / G;
      g[i] = idx % G;
    }
    writer = (li % C::kRep) == 0;
  }
  __device__ __forceinline__ int idx(int i) const { return j[i] * G + g[i]; }
};

// Two consecutive stages at once: the warp's 8 rows of each are two independent batches whose
// q . k and P . V chains interleave (when there is no second stage, n[1] == 0 masks every row
// of the second batch, which then reads stale but in-bounds shared memory). p values are
// published to shared memory as (p, p) pairs so that P . V takes its packed-FMA operands
// straight from a 16-byte load.
template <typename T, int D, int G, bool UNIFIED, bool LOCAL>
__device__ __forceinline__ void consume_stages(const Params& p, const LaneMap<T, D, G>& lm,
                                               const uint8_t* const (&ks)[2],
                                               const uint8_t* const (&vs)[2], const int (&n)[2],
                                               const f32x2 (&q2)[G][Cfg<T, D, G>::kEpl / 2],
                                               f32x2 (&acc2)[G][Cfg<T, D, G>::kEpl / 2],
                                               float (&dl)[Cfg<T, D, G>::kNv], float (&m)[G],
                                               float (&mt)[G], bool& sw, uint32_t& fmask,
                                               float* wscr) {
  using C = Cfg<T, D, G>;
  constexpr int E2 = C::kEpl / 2;
  constexpr int RS = tp_row_stride(D, C::kEs);
  constexpr int NB = 2;   // an absent second stage has n[1] == 0: all its rows are masked

  // q . k for the lane group's rows and all G heads: partial sums over this lane's chunk
  float part[NB][C::kV];
#pragma unroll
  for (int b = 0; b < NB; ++b) {
#pragma unroll
    for (int j = 0; j < C::kT; ++j) {
      const uint4 c =
          *reinterpret_cast<const uint4*>(ks[b] + (lm.row0 + j) * C::kRowBytes + lm.li * 16);
      f32x2 kp[E2];
      Elem<T>::to_pairs(c, kp);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        f32x2 s2 = f2_mul(q2[g][0], kp[0]);
#pragma unroll
        for (int e = 1; e < E2; ++e) f2_fma(s2, q2[g][e], kp[e]);
        float lo, hi;
        f2_unpack(s2, lo, hi);
        part[b][j * G + g] = lo + hi;
      }
    }
  }
  // Transpose-reduce through shared memory: lane li of the group stores its kV partial sums
  // as column li of a [kV][kLg] block (rows padded so that every 16-byte read of a row hits
  // its own banks), then each lane sums the kLg partials of its logit's row.
  float* tb = wscr + lm.lg * tp_group_floats(D, G, C::kEs);
  float sc[NB][C::kNv];
#pragma unroll
  for (int b = 0; b < NB; ++b) {
#pragma unroll
    for (int v = 0; v < C::kV; ++v) tb[v * RS + lm.li] = part[b][v];
    __syncwarp();
#pragma unroll
    for (int i = 0; i < C::kNv; ++i) {
      const float4* row = reinterpret_cast<const float4*>(tb + lm.idx(i) * RS);
      float4 acc4 = row[0];
#pragma unroll
      for (int c = 1; c < C::kLg / 4; ++c) {
        const float4 x = row[c];
        acc4.x += x.x;
        acc4.y += x.y;
        acc4.z += x.z;
        acc4.w += x.w;
      }
      sc[b][i] = (acc4.x + acc4.y) + (acc4.z + acc4.w);
    }
    __syncwarp();   // the block is reused by the next batch and for p below
  }

  // p pairs: batch b at pwarp + b * 8 * G, lane group lg at + lg * kV
  float2* pwarp = reinterpret_cast<float2*>(wscr);
  bool valid[NB][C::kNv];
#pragma unroll
  for (int b = 0; b < NB; ++b)
#pragma unroll
    for (int i = 0; i < C::kNv; ++i) valid[b][i] = lm.row0 + lm.j[i] < n[b];

  bool use_sync = !UNIFIED;
  if constexpr (LOCAL) {
    // Split-local fallback: while every logit so far was in range, the state is an exact
    // online-softmax state with m = phi. On the first tile with a logit out of range the warp
    // rescales it to each head's true maximum so far and continues with the synchronised
    // recurrence, so the split needs no second read of its KV.
    if (!sw) {
      bool out = false;
#pragma unroll
      for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int i = 0; i < C::kNv; ++i)
          if (valid[b][i]) {
            const float sv = sc[b][i];
            out = out || sv < p.lo2 || sv > p.hi2;
#pragma unroll
            for (int g = 0; g < G; ++g)
              if (lm.g[i] == g) mt[g] = fmaxf(mt[g], sv);
          }
      if (__any_sync(0xffffffffu, out)) {
        float alpha[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float mg = mt[g];
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1) mg = fmaxf(mg, __shfl_xor_sync(0xffffffffu, mg, o));
          alpha[g] = mg > -INFINITY ? fast_exp2(p.phi2 - mg) : 1.f;
          m[g] = mg;
          const f32x2 a2 = f2_pack(alpha[g], alpha[g]);
#pragma unroll
          for (int e = 0; e < E2; ++e) acc2[g][e] = f2_mul(acc2[g][e], a2);
        }
#pragma unroll
        for (int i = 0; i < C::kNv; ++i) {
          float ag = alpha[0];
#pragma unroll
          for (int g = 1; g < G; ++g)
            if (lm.g[i] == g) ag = alpha[g];
          dl[i] *= ag;
        }
        sw = true;
      }
    }
    use_sync = sw;
  }

  if (!use_sync) {
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      float2* pw = pwarp + b * kTokensPerWarp * G + lm.lg * C::kV;
#pragma unroll
      for (int i = 0; i < C::kNv; ++i) {
        const float s = sc[b][i];
        const float pr = valid[b][i] ? fast_exp2(s - p.phi2) : 0.f;
        if (valid[b][i] && (s < p.lo2 || s > p.hi2)) fmask |= 1u << lm.g[i];
        dl[i] += pr;
        if (lm.writer) pw[lm.idx(i)] = make_float2(pr, pr);
      }
    }
  } else {
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      float2* pw = pwarp + b * kTokensPerWarp * G + lm.lg * C::kV;
#pragma unroll
      for (int i = 0; i < C::kNv; ++i) {
        const float s = valid[b][i] ? sc[b][i] : -INFINITY;
        if (UNIFIED && valid[b][i] && (s < p.lo2 || s > p.hi2)) fmask |= 1u << lm.g[i];
        if (lm.writer) pw[lm.idx(i)] = make_float2(s, s);
      }
    }
    __syncwarp();
    // per-head maximum over the warp's rows of both stages, then one online update
    float tm[G];
#pragma unroll
    for (int g = 0; g < G; ++g) tm[g] = -INFINITY;
#pragma unroll
    for (int r = 0; r < NB * kTokensPerWarp; ++r)
#pragma unroll
      for (int g = 0; g < G; ++g) tm[g] = fmaxf(tm[g], pwarp[r * G + g].x);
    float alpha[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float mn = fmaxf(m[g], tm[g]);
      alpha[g] = mn == -INFINITY ? 1.f : fast_exp2(m[g] - mn);
      m[g] = mn;
      const f32x2 a2 = f2_pack(alpha[g], alpha[g]);
#pragma unroll
      for (int e = 0; e < E2; ++e) acc2[g][e] = f2_mul(acc2[g][e], a2);
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < C::kNv; ++i) {
      float mg = m[0], ag = alpha[0];
#pragma unroll
      for (int g = 1; g < G; ++g)
        if (lm.g[i] == g) {
          mg = m[g];
          ag = alpha[g];
        }
      dl[i] *= ag;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const float pr = valid[b][i] ? fast_exp2(sc[b][i] - mg) : 0.f;
        dl[i] += pr;
        float2* pw = pwarp + b * kTokensPerWarp * G + lm.lg * C::kV;
        if (lm.writer) pw[lm.idx(i)] = make_float2(pr, pr);
      }
    }
  }
  __syncwarp();

  // P . V: every lane of the group accumulates its chunk of d for all heads
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const float2* pw = pwarp + b * kTokensPerWarp * G + lm.lg * C::kV;
#pragma unroll
    for (int j = 0; j < C::kT; ++j) {
      if (lm.row0 + j < n[b]) {
        const uint4 c =
            *reinterpret_cast<const uint4*>(vs[b] + (lm.row0 + j) * C::kRowBytes + lm.li * 16);
        f32x2 vp[E2];
        Elem<T>::to_pairs(c, vp);
        f32x2 pp[G];
        const f32x2* pwj = reinterpret_cast<const f32x2*>(pw + j * G);
        if constexpr (G == 1) {
          pp[0] = pwj[0];
        } else {
#pragma unroll
          for (int g = 0; g < G; g += 2) {
            const ulonglong2 two2 = *reinterpret_cast<const ulonglong2*>(pwj + g);
            pp[g] = two2.x;
            pp[g + 1] = two2.y;
          }
        }
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int e = 0; e < E2; ++e) f2_fma(acc2[g][e], pp[g], vp[e]);
      }
    }
  }
  __syncwarp();
}

// ---- consumer warps: end of a piece ---------------------------------------------------
// Publish a CUDA-core warp's piece state to the shared scratch: m, l per head and the
// accumulators as [warp][G][D].
template <typename T, int D, int G>
__device__ __forceinline__ void publish_cuda(const LaneMap<T, D, G>& lm,
                                             float (&acc)[G][Cfg<T, D, G>::kEpl],
                                             const float (&dl)[Cfg<T, D, G>::kNv],
                                             const float (&m)[G], uint32_t fmask, float* mm,
                                             float* ml, uint32_t* mflag, float* wbuf, int warp,
                                             int lane) {
  using C = Cfg<T, D, G>;
  constexpr int E = C::kEpl;
  constexpr int W = warp_scratch_floats(D, G, C::kEs);
  // the warp's denominators: each head's p values are spread over the lanes holding it
  float den[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < C::kNv; ++i)
      if (lm.writer && lm.g[i] == g) s += dl[i];
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    den[g] = s;
  }
  // combine the warp's lane groups (same d-chunk, disjoint rows)
#pragma unroll
  for (int o = C::kLg; o < 32; o <<= 1)
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < E; ++e) acc[g][e] += __shfl_xor_sync(0xffffffffu, acc[g][e], o);
  const uint32_t fm = __reduce_or_sync(0xffffffffu, fmask);
  if (lm.lg == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < E; ++e) wbuf[warp * W + g * D + lm.li * E + e] = acc[g][e];
  }
  if (lane == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      mm[warp * G + g] = m[g];
      ml[warp * G + g] = den[g];
    }
    mflag[warp] = fm;
  }
}

// Publish a tensor-core warp's piece state (same scratch format as publish_cuda): the lane
// holds O^T elements (d = 16 mt + lane / 4 and d + 8) of heads hp = 2 (lane % 4) and hp + 1,
// and its share of those heads' denominators; the 8 lanes sharing lane % 4 complete a head.
template <typename T, int D, int G>
__device__ __forceinline__ void publish_mma(const MmaState<D, G>& st, float m0, float m1,
                                            uint32_t fmask, float* mm, float* ml,
                                            uint32_t* mflag, float* wbuf, int warp, int lane) {
  constexpr int W = warp_scratch_floats(D, G, Cfg<T, D, G>::kQEs);
  const int hp = 2 * (lane & 3), dr = lane >> 2;
  float den0 = st.den[0], den1 = st.den[1];
#pragma unroll
  for (int o = 4; o <= 16; o <<= 1) {
    den0 += __shfl_xor_sync(0xffffffffu, den0, o);
    den1 += __shfl_xor_sync(0xffffffffu, den1, o);
  }
  const uint32_t fm = __reduce_or_sync(0xffffffffu, fmask);
  float* w0 = wbuf + warp * W + hp * D;
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    // the O^T rows this lane holds: d and d + 8 (bf16 tiles), d and d + 1 (FP8 tiles)
    const int d = Cfg<T, D, G>::kFp8 ? (D / 8) * dr + 2 * mt : mt * 16 + dr;
    const int d2 = Cfg<T, D, G>::kFp8 ? d + 1 : d + 8;
    if (hp < G) {
      w0[d] = st.o[mt][0];
      w0[d2] = st.o[mt][2];
    }
    if (hp + 1 < G) {
      w0[D + d] = st.o[mt][1];
      w0[D + d2] = st.o[mt][3];
    }
  }
  if (lane < 4) {
    if (hp < G) {
      mm[warp * G + hp] = m0;
      ml[warp * G + hp] = den0;
    }
    if (hp + 1 < G) {
      mm[warp * G + hp + 1] = m1;
      ml[warp * G + hp + 1] = den1;
    }
  }
  if (lane == 0) mflag[warp] = fm;
}

// Each consumer thread owns EPT consecutive output elements of one head in the combine and
// merge steps (e0 = thread * EPT; threads with e0 >= G * D own none).
template <int D, int G>
struct CombineMap {
  static constexpr int kCT = kConsumerWarps * 32;
  static constexpr int EPT = G * D >= 4 * kCT ? 4 : (G * D >= 2 * kCT ? 2 : 1);
  int e0, g, d0;
  bool owns;
  __device__ __forceinline__ explicit CombineMap(int ctid) {
    e0 = ctid * EPT;
    owns = e0 < G * D;
    g = owns ? e0 / D : 0;
    d0 = e0 - g * D;
  }
};

template <int N>
__device__ __forceinline__ void load_smem_vec(const float* src, float (&v)[N]) {
  if constexpr (N == 4) {
    const float4 x = *reinterpret_cast<const float4*>(src);
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  } else if constexpr (N == 2) {
    const float2 x = *reinterpret_cast<const float2*>(src);
    v[0] = x.x; v[1] = x.y;
  } else {
    v[0] = src[0];
  }
}

// The last piece of a group to finish merges it (recompute pass): the partial goes to the
// workspace, a release-acquire arrival count picks the last piece, which loads all partials
// and forms L = log2 sum_s 2^L_s, O = sum_s 2^(L_s - L) O_s.
template <typename T, int D, int G>
__device__ __forceinline__ void merge_last_arriver(const Params& p, const Piece& pc,
                                                   bool first_phase,
                                                   const float (&o)[CombineMap<D, G>::EPT],
                                                   float L2, uint32_t fl, float* mm, float* ml,
                                                   float* wbuf, int* misc, int warp, int lane,
                                                   int ctid) {
  using CM = CombineMap<D, G>;
  constexpr int kCT = CM::kCT, EPT = CM::EPT;
  constexpr float kLn2 = 0.6931471805599453f;
  const CM cm(ctid);
  const long long row0 = (long long)pc.b * p.hq + (long long)pc.kvh * G;
  if (cm.owns) {
    float* dst = p.part_o + ((long long)pc.slot * G + cm.g) * D + cm.d0;
#pragma unroll
    for (int i = 0; i < EPT; ++i) __stcg(dst + i, o[i]);
    if (cm.d0 == 0) __stcg(p.part_l + (long long)pc.slot * G + cm.g, L2);
  }
  if (ctid == 0) __stcg(p.part_flags + pc.slot, fl);
  // Arrival: the barrier orders the CTA's partial writes before thread 0's release-acquire
  // count; the last piece's count also acquires the other pieces' partials.
  named_bar_sync(1, kCT);
  if (ctid == 0) {
    const int old = atom_add_acq_rel_gpu(p.counters + pc.g, 1);
    misc[0] = old == pc.nslots - 1;
    misc[1] = 0;
  }
  named_bar_sync(1, kCT);
  if (!misc[0]) return;
  // Last piece of the group: merge all its partials; each thread issues the loads of up to 64
  // partial values at once, together with the LSEs, so a group of up to 64 / EPT pieces pays
  // the L2 latency once.
  const int S = pc.nslots;
  float* wts = wbuf;              // [S, G] weights (scratch reused; S <= 8 * D)
  float* hsum = mm;               // [G] sum of weights
  float* hmax = ml;               // [G] maximum partial LSE
  constexpr int SB = 16;   // partials per round of loads (a small block keeps this rarely run code short)
  const float* po = p.part_o + (long long)pc.slot_base * G * D + (cm.owns ? cm.e0 : 0);
  float ob[SB][EPT];
  auto load_block = [&](int s0) {
#pragma unroll
    for (int j = 0; j < SB; ++j) {
      const bool ok = cm.owns && s0 + j < S;
      const float* src = po + (long long)(s0 + j) * G * D;
#pragma unroll
      for (int i = 0; i < EPT; ++i) ob[j][i] = ok ? __ldcg(src + i) : 0.f;
    }
  };
  load_block(0);
  const float* pl = p.part_l + (long long)pc.slot_base * G;
  for (int i = ctid; i < S * G; i += kCT) wts[i] = __ldcg(pl + i);
  uint32_t rf = 0;
  for (int s = ctid; s < S; s += kCT) rf |= __ldcg(p.part_flags + pc.slot_base + s);
  rf = __reduce_or_sync(0xffffffffu, rf);
  if (lane == 0 && rf) atomicOr(reinterpret_cast<unsigned int*>(misc + 1), rf);
  named_bar_sync(1, kCT);
  if (warp < G) {
    const int g = warp;
    float M = -INFINITY;
    for (int s = lane; s < S; s += 32) M = fmaxf(M, wts[s * G + g]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float sum = 0.f;
    for (int s = lane; s < S; s += 32) {
      const float L = wts[s * G + g];
      const float f = L > -INFINITY ? fast_exp2(L - M) : 0.f;
      wts[s * G + g] = f;
      sum += f;
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane == 0) {
      hsum[g] = sum;
      hmax[g] = M;
    }
  }
  named_bar_sync(1, kCT);
  float num[EPT];
#pragma unroll
  for (int i = 0; i < EPT; ++i) num[i] = 0.f;
  for (int s0 = 0; s0 < S; s0 += SB) {
    if (s0 > 0) load_block(s0);
#pragma unroll
    for (int j = 0; j < SB; ++j) {
      if (s0 + j < S) {
        const float w = wts[(s0 + j) * G + cm.g];
#pragma unroll
        for (int i = 0; i < EPT; ++i) num[i] += w * ob[j][i];
      }
    }
  }
  const uint32_t rfa = (uint32_t)misc[1];
  if (cm.owns) {
    const float sum = hsum[cm.g];
#pragma unroll
    for (int i = 0; i < EPT; ++i)
      store_out(p.out, (row0 + cm.g) * D + cm.d0 + i, p.out_dtype,
                sum > 0.f ? num[i] / sum * p.v_scale : 0.f);
    if (cm.d0 == 0) {
      if (p.out_lse)
        p.out_lse[row0 + cm.g] = sum > 0.f ? (hmax[cm.g] + fast_log2(sum)) * kLn2 : -INFINITY;
      if (p.row_flags && first_phase) p.row_flags[row0 + cm.g] = (uint8_t)((rfa >> cm.g) & 1u);
    }
  }
  if (ctid == 0) {
    p.counters[pc.g] = 0;   // leave the counter ready for the next run
    if (first_phase && rfa) {
      atomicAdd(p.stats + 0, (unsigned long long)__popc(rfa));
      if (p.list_flags) {
        const int at = atomicAdd(p.list_state, 1);
        if (at < p.n_groups) p.flag_list[at] = pc.g;
      }
    }
  }
}

// The 8 consumer warps' published states -> one partial of the piece (or the output, when the
// piece is its group's only one), then the group's merge where this piece takes part in it
// (the split-KV log-sum-exp merge, "The Rescaling and Online Softmax Reduction Algorithm").
// `first_phase`: the piece belongs to the step's first pass, which records flags, statistics
// and the flagged list.
template <typename T, int D, int G>
__device__ __forceinline__ void combine_piece(const Params& p, const Piece& pc, bool first_phase,
                                              float* mm, float* ml, uint32_t* mflag,
                                              float* wbuf, int* misc, int warp, int lane,
                                              int ctid) {
  using CM = CombineMap<D, G>;
  constexpr int kCT = CM::kCT, EPT = CM::EPT;
  constexpr float kLn2 = 0.6931471805599453f;
  constexpr int W = warp_scratch_floats(D, G, Cfg<T, D, G>::kQEs);
  named_bar_sync(1, kCT);

  uint32_t fl = 0;
#pragma unroll
  for (int w = 0; w < kConsumerWarps; ++w) fl |= mflag[w];
  const bool direct = pc.nslots == 1;
  const long long row0 = (long long)pc.b * p.hq + (long long)pc.kvh * G;
  const CM cm(ctid);

  // the 8 warps' (m, l, acc) -> this piece's partial for the thread's elements (max-rescale)
  float o[EPT], L2 = -INFINITY;
#pragma unroll
  for (int i = 0; i < EPT; ++i) o[i] = 0.f;
  if (cm.owns) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w)
      if (ml[w * G + cm.g] > 0.f) M = fmaxf(M, mm[w * G + cm.g]);
    float num[EPT], sum = 0.f;
#pragma unroll
    for (int i = 0; i < EPT; ++i) num[i] = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float lw = ml[w * G + cm.g];
      if (lw > 0.f) {
        const float f = fast_exp2(mm[w * G + cm.g] - M);
        float a[EPT];
        load_smem_vec<EPT>(wbuf + w * W + cm.g * D + cm.d0, a);
        sum += f * lw;
#pragma unroll
        for (int i = 0; i < EPT; ++i) num[i] += f * a[i];
      }
    }
#pragma unroll
    for (int i = 0; i < EPT; ++i) o[i] = sum > 0.f ? num[i] / sum : 0.f;
    L2 = sum > 0.f ? M + fast_log2(sum) : -INFINITY;
  }

  if (ctid == 0 && first_phase) {
    if (fl) {
      atomicAdd(p.stats + 1, (unsigned long long)__popc(fl));
      if (direct) {
        atomicAdd(p.stats + 0, (unsigned long long)__popc(fl));
        if (p.list_flags) {
          const int at = atomicAdd(p.list_state, 1);
          if (at < p.n_groups) p.flag_list[at] = pc.g;
        }
      }
    }
    if (p.piece_stats) {
      const unsigned long long t = (unsigned long long)(pc.t1 - pc.t0);
      atomicMax(p.stats + 2, t);
      atomicMax(p.stats + 3, 0x7fffffffull - t);
    }
  }

  if (direct) {
    if (cm.owns) {
#pragma unroll
      for (int i = 0; i < EPT; ++i)
        store_out(p.out, (row0 + cm.g) * D + cm.d0 + i, p.out_dtype, o[i] * p.v_scale);
      if (cm.d0 == 0) {
        if (p.out_lse) p.out_lse[row0 + cm.g] = L2 * kLn2;
        if (p.row_flags && first_phase) p.row_flags[row0 + cm.g] = (uint8_t)((fl >> cm.g) & 1u);
      }
    }
  } else {
    merge_last_arriver<T, D, G>(p, pc, first_phase, o, L2, fl, mm, ml, wbuf, misc, warp, lane,
                                ctid);
  }
  named_bar_sync(1, kCT);   // shared scratch is free for the next piece
}

template <typename T, int D, int G, bool UNIFIED, bool LOCAL>
__device__ __forceinline__ void run_consumers(const Params& p, Sched s, uint8_t* stages,
                                              const Layout& L, uint64_t* full, uint64_t* empty,
                                              uint8_t* smem, int warp, int lane) {
  using C = Cfg<T, D, G>;
  constexpr int E = C::kEpl;
  const uint32_t NS = (uint32_t)p.stages;
  float* wbuf = reinterpret_cast<float*>(smem + L.wbuf_off);
  float* wscr = wbuf + warp * warp_scratch_floats(D, G, C::kEs);
  float* mm = reinterpret_cast<float*>(smem + L.mm_off);
  float* ml = reinterpret_cast<float*>(smem + L.ml_off);
  uint32_t* mflag = reinterpret_cast<uint32_t*>(smem + L.mflag_off);
  int* misc = reinterpret_cast<int*>(smem + L.misc_off);
  const LaneMap<T, D, G> lm(warp, lane);
  const int ctid = warp * 32 + lane;
  Piece pc;
  constexpr int E2 = E / 2;
  uint32_t k = 0;
  bool dead = false, gave_up = false;
  while (sched_next(s, p, pc)) {
    float dl[C::kNv], m[G], mt[G];
    bool sw = false;
    f32x2 acc2[G][E2], q2[G][E2];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m[g] = UNIFIED ? p.phi2 : -INFINITY;
      mt[g] = -INFINITY;
#pragma unroll
      for (int e = 0; e < E2; ++e) {
        acc2[g][e] = 0ull;   // +0.0f in both halves
        q2[g][e] = 0ull;
      }
    }
#pragma unroll
    for (int i = 0; i < C::kNv; ++i) dl[i] = 0.f;
    uint32_t fmask = 0;
    const int nst = (pc.t1 - pc.t0 + kStageTokens - 1) / kStageTokens;
    for (int j = 0; j < nst; j += 2) {
      const bool pair = j + 1 < nst;
      const uint32_t s0 = k % NS, s1 = (k + 1) % NS;
      if (!dead && !mbar_wait(&full[s0], (k / NS) & 1u, p.wait_limit_ns)) dead = true;
      if (pair && !dead && !mbar_wait(&full[s1], ((k + 1) / NS) & 1u, p.wait_limit_ns))
        dead = true;
      if (dead && lane == 0 && !gave_up) {
        gave_up = true;
        atomicOr(p.status, kStatusTimeout);
        atomicExch(misc + 3, 1);   // the producer stops issuing
      }
      const uint8_t* st0 = stages + s0 * L.stage_bytes;
      const uint8_t* st1 = stages + s1 * L.stage_bytes;
      if (j == 0) {
        const f32x2 qs = f2_pack(p.qscale, p.qscale);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const uint4 c =
              *reinterpret_cast<const uint4*>(st0 + L.q_off + g * C::kRowBytes + lm.li * 16);
          Elem<T>::to_pairs(c, q2[g]);
#pragma unroll
          for (int e = 0; e < E2; ++e) q2[g][e] = f2_mul(q2[g][e], qs);
        }
      }
      const int ts = pc.t0 + j * kStageTokens;
      const int n[2] = {min(kStageTokens, pc.t1 - ts),
                        pair ? min(kStageTokens, pc.t1 - ts - kStageTokens) : 0};
      const uint8_t* const kss[2] = {st0 + L.k_off, st1 + L.k_off};
      const uint8_t* const vss[2] = {st0 + L.v_off, st1 + L.v_off};
      if (!dead)
        consume_stages<T, D, G, UNIFIED, LOCAL>(p, lm, kss, vss, n, q2, acc2, dl, m, mt, sw,
                                                fmask, wscr);
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&empty[s0]);
        if (pair) mbar_arrive(&empty[s1]);
      }
      k += pair ? 2u : 1u;
    }
    float acc[G][E];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < E2; ++e) f2_unpack(acc2[g][e], acc[g][2 * e], acc[g][2 * e + 1]);
    publish_cuda<T, D, G>(lm, acc, dl, m, fmask, mm, ml, mflag, wbuf, warp, lane);
    combine_piece<T, D, G>(p, pc, s.first_phase, mm, ml, mflag, wbuf, misc, warp, lane, ctid);
  }
}

// Tensor-core consumers (bf16 or FP8 caches, every softmax mode): same stage-pair loop as
// run_consumers, the math in mma_consume / mma_consume_fp8.
template <typename T, int D, int G, bool UNIFIED, bool LOCAL>
__device__ __forceinline__ void run_consumers_mma(const Params& p, Sched s, uint8_t* stages,
                                                  const Layout& L, uint64_t* full,
                                                  uint64_t* empty, uint8_t* smem, int warp,
                                                  int lane) {
  const uint32_t NS = (uint32_t)p.stages;
  float* wbuf = reinterpret_cast<float*>(smem + L.wbuf_off);
  float* mm = reinterpret_cast<float*>(smem + L.mm_off);
  float* ml = reinterpret_cast<float*>(smem + L.ml_off);
  uint32_t* mflag = reinterpret_cast<uint32_t*>(smem + L.mflag_off);
  int* misc = reinterpret_cast<int*>(smem + L.misc_off);
  const int ctid = warp * 32 + lane;
  const int row0 = warp * kTokensPerWarp;
  constexpr bool kFp8 = Cfg<T, D, G>::kFp8;
  const std::conditional_t<kFp8, NoMmaLane, MmaLane<D>> mlane(row0, lane);
  Piece pc;
  uint32_t k = 0;
  bool dead = false, gave_up = false;
  while (sched_next(s, p, pc)) {
    MmaState<D, G> st;
#pragma unroll
    for (int j = 0; j < D / 16; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) st.o[j][i] = 0.f;
    st.den[0] = st.den[1] = 0.f;
    st.m[0] = st.m[1] = -INFINITY;
    st.sw = false;
    st.qmul = p.qscale;   // FP8 tiles: reset with q's scale when q is loaded
    uint32_t fmask = 0;
    const int nst = (pc.t1 - pc.t0 + kStageTokens - 1) / kStageTokens;
    for (int j = 0; j < nst; j += 2) {
      const bool pair = j + 1 < nst;
      const uint32_t s0 = k % NS, s1 = (k + 1) % NS;
      if (!dead && !mbar_wait(&full[s0], (k / NS) & 1u, p.wait_limit_ns)) dead = true;
      if (pair && !dead && !mbar_wait(&full[s1], ((k + 1) / NS) & 1u, p.wait_limit_ns))
        dead = true;
      if (dead && lane == 0 && !gave_up) {
        gave_up = true;
        atomicOr(p.status, kStatusTimeout);
        atomicExch(misc + 3, 1);   // the producer stops issuing
      }
      const uint8_t* st0 = stages + s0 * L.stage_bytes;
      const uint8_t* st1 = stages + s1 * L.stage_bytes;
      if (j == 0) {
        if constexpr (kFp8)
          mma_load_q_fp8<D, G>(p, st, st0 + L.q_off, lane);
        else
          mma_load_q<D, G>(st, st0 + L.q_off, lane);
      }
      const int ts = pc.t0 + j * kStageTokens;
      const int n[2] = {min(kStageTokens, pc.t1 - ts),
                        pair ? min(kStageTokens, pc.t1 - ts - kStageTokens) : 0};
      const uint8_t* const st1m = pair ? st1 : st0;   // no second stage: read stage 0 again
      const uint32_t kt[2] = {smem_u32(st0 + L.k_off), smem_u32(st1m + L.k_off)};
      const uint32_t vt[2] = {smem_u32(st0 + L.v_off), smem_u32(st1m + L.v_off)};
      if (!dead) {
        if constexpr (kFp8)
          mma_consume_fp8<D, G, Cfg<T, D, G>::kHp, UNIFIED, LOCAL>(p, st, kt, vt, n, row0, lane,
                                                                    fmask);
        else
          mma_consume<D, G, UNIFIED, LOCAL>(p, st, mlane, kt, vt, n, row0, lane, fmask);
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&empty[s0]);
        if (pair) mbar_arrive(&empty[s1]);
      }
      k += pair ? 2u : 1u;
    }
    // the state is relative to phi (bf16 tiles, unified phase) or to st.m (FP8 tiles, whose
    // unified phase keeps its own power-of-two reference there)
    const bool at_phi = UNIFIED && !kFp8 && !(LOCAL && st.sw);
    publish_mma<T, D, G>(st, at_phi ? p.phi2 : st.m[0], at_phi ? p.phi2 : st.m[1], fmask, mm, ml,
                         mflag, wbuf, warp, lane);
    combine_piece<T, D, G>(p, pc, s.first_phase, mm, ml, mflag, wbuf, misc, warp, lane, ctid);
  }
}

// The dynamic shared memory, aligned to 1024 bytes (the 128-byte swizzle's period).
__device__ __forceinline__ uint8_t* smem_base() {
  extern __shared__ uint8_t smem_raw[];
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                    ~static_cast<uintptr_t>(1023));
}

// The launch's schedule for this CTA, from the parameters and what the prologue left in shared
// memory (lengths and prefix for balanced shares, the flagged count for a recompute launch).
// The roles rebuild it after the register split, so that nothing but the parameters stays live
// across it: the producer warps' small register budget then holds only their own state.
__device__ __forceinline__ Sched launch_sched(const Params& p, const int* lens, const int* prefix,
                                              const int* misc) {
  Sched s;
  s.policy = p.policy;
  s.P = gridDim.x;
  s.c = blockIdx.x;
  s.lens = lens;
  s.prefix = prefix;
  s.u = s.u1 = s.W = 0;
  s.i = s.i1 = 0;
  s.S = p.num_splits > 0 ? p.num_splits : 1;
  s.use_list = p.recompute != 0;
  s.first_phase = p.recompute == 0;
  if (p.recompute || p.policy != kBalanced) {
    const long long ni = (long long)(p.recompute ? misc[2] : p.n_groups) * s.S;
    if (p.narrow) {
      s.i = (unsigned)blockIdx.x * (unsigned)ni / gridDim.x;
      s.i1 = ((unsigned)blockIdx.x + 1u) * (unsigned)ni / gridDim.x;
    } else {
      s.i = (long long)blockIdx.x * ni / gridDim.x;
      s.i1 = ((long long)blockIdx.x + 1) * ni / gridDim.x;
    }
  } else {
    s.W = (long long)p.hkv * prefix[p.batch];
    // The grid is sized from the cache capacity; when the step holds fewer units than CTAs,
    // only the first W CTAs take shares, so that every share is non-empty and a group's
    // pieces sit on consecutive CTAs (its piece count is then cl - cf + 1).
    s.P = (int)(s.W < (long long)gridDim.x ? s.W : (long long)gridDim.x);
    if ((int)blockIdx.x < s.P) {
      if (p.narrow) {
        s.u = (unsigned)blockIdx.x * (unsigned)s.W / (unsigned)s.P;
        s.u1 = ((unsigned)blockIdx.x + 1u) * (unsigned)s.W / (unsigned)s.P;
      } else {
        s.u = (long long)blockIdx.x * s.W / s.P;
        s.u1 = ((long long)blockIdx.x + 1) * s.W / s.P;
      }
    }
  }
  return s;
}

// A consumer warp's role over the launch's pieces.
template <typename T, int D, int G, int MODE>
__device__ __forceinline__ void consumer_role(const Params& p, int warp, int lane) {
  constexpr bool UNIFIED = MODE != kSoftmaxSync, LOCAL = MODE == kSoftmaxUnifiedLocal;
  using C = Cfg<T, D, G>;
  constexpr bool kMma = uses_mma(sizeof(T), std::is_same<T, __half>::value, G);
  uint8_t* smem = smem_base();
  const Layout L = make_layout(D, G, C::kQEs, p.stages, p.batch_smem, C::kEs, C::kHp);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  uint64_t* empty = full + p.stages;
  const Sched s = launch_sched(p, reinterpret_cast<const int*>(smem + L.lens_off),
                               reinterpret_cast<const int*>(smem + L.prefix_off),
                               reinterpret_cast<const int*>(smem + L.misc_off));
  if constexpr (kMma)
    run_consumers_mma<T, D, G, UNIFIED, LOCAL>(p, s, smem, L, full, empty, smem, warp, lane);
  else
    run_consumers<T, D, G, UNIFIED, LOCAL>(p, s, smem, L, full, empty, smem, warp, lane);
}

// A producer-warpgroup warp's role (two warps issue copies for a contiguous cache, four for a
// paged one; the others have nothing to do).
template <typename T, int D, int G>
__device__ __forceinline__ void producer_role(const Params& p, const CUtensorMap* tmk,
                                              const CUtensorMap* tmv, int warp, int lane) {
  using C = Cfg<T, D, G>;
  constexpr bool kMma = uses_mma(sizeof(T), std::is_same<T, __half>::value, G);
  constexpr bool k4d = kMma && !C::kFp8;   // bf16 tensor-core tiles: the 4-D swizzled view
  if (warp >= kConsumerWarps + (p.paged ? 4 : 2)) return;
  uint8_t* smem = smem_base();
  const Layout L = make_layout(D, G, C::kQEs, p.stages, p.batch_smem, C::kEs, C::kHp);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  uint64_t* empty = full + p.stages;
  const Sched s = launch_sched(p, reinterpret_cast<const int*>(smem + L.lens_off),
                               reinterpret_cast<const int*>(smem + L.prefix_off),
                               reinterpret_cast<const int*>(smem + L.misc_off));
  run_producer<T, D, G, k4d>(p, s, smem, L, full, empty, tmk, tmv, lane, warp - kConsumerWarps,
                              reinterpret_cast<const int*>(smem + L.misc_off) + 3);
}

// The split kernel. A step's first launch computes every group with the step's softmax mode
// (balanced shares, or uniform splits of every group); the last piece of each group to finish
// merges the group. In unified mode a second launch of the synchronised kernel follows as a
// programmatic dependent (`recompute`): it waits for the first launch's results, reads the
// list of groups whose range check failed and recomputes them with the synchronised softmax
// as uniform splits ("The Overflow Fallback: Recomputation"); with nothing flagged it exits
// at once.
template <typename T, int D, int G, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    decode_split_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv) {
  using C = Cfg<T, D, G>;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (p.recompute) {
    // the first launch's flagged list is complete and visible after this wait; with nothing
    // flagged the recompute launch has no work (and nothing to reset)
    pdl_wait();
    if (min(__ldcg(p.list_state), p.n_groups) == 0) return;
  }
  {
    uint8_t* smem = smem_base();
    const Layout L = make_layout(D, G, C::kQEs, p.stages, p.batch_smem, C::kEs, C::kHp);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_off);
    uint64_t* empty = full + p.stages;
    int* lens = reinterpret_cast<int*>(smem + L.lens_off);
    int* prefix = reinterpret_cast<int*>(smem + L.prefix_off);
    int* misc = reinterpret_cast<int*>(smem + L.misc_off);
    if (tid == 0) {
      for (int s = 0; s < p.stages; ++s) {
        mbar_init(&full[s], 1);
        mbar_init(&empty[s], kConsumerWarps);
      }
      fence_mbar_init();
      if (p.recompute) misc[2] = min(__ldcg(p.list_state), p.n_groups);
      misc[3] = 0;   // set when a consumer's wait runs out
    }
    if (warp == kConsumerWarps && lane == 0) {
      prefetch_tensormap(&tmk);
      prefetch_tensormap(&tmv);
    }
    if (!p.recompute && p.policy == kBalanced) {
      if (p.batch <= 32) {
        // One warp (not thread 0, which initialises the barriers meanwhile) loads the lengths
        // and builds the unit prefix with shuffles: one CTA barrier in the whole prologue.
        if (warp == 1) {
          int n = 0;
          if (lane < p.batch) {
            const int raw = __ldg(p.seq_lens + lane);
            n = clamp_len(p, raw);
            if (n != raw && blockIdx.x == 0) atomicOr(p.status, kStatusBadSeqLen);
            lens[lane] = n;
          }
          const int units = n ? (n + p.unit - 1) / p.unit + p.piece_units : 0;
          int incl = units;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
          }
          if (lane < p.batch) prefix[lane] = incl - units;
          if (lane == p.batch - 1) prefix[p.batch] = incl;
        }
        __syncthreads();
      } else {
        for (int b = tid; b < p.batch; b += blockDim.x) {
          const int raw = __ldg(p.seq_lens + b);
          const int n = clamp_len(p, raw);
          if (n != raw && blockIdx.x == 0) atomicOr(p.status, kStatusBadSeqLen);
          lens[b] = n;
        }
        __syncthreads();
        if (warp == 0) {
          const int per = (p.batch + 31) / 32;
          const int beg = min(p.batch, lane * per), end = min(p.batch, beg + per);
          int local = 0;
          for (int b = beg; b < end; ++b)
            local += lens[b] ? (lens[b] + p.unit - 1) / p.unit + p.piece_units : 0;
          int incl = local;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
          }
          int run = incl - local;
          for (int b = beg; b < end; ++b) {
            prefix[b] = run;
            run += lens[b] ? (lens[b] + p.unit - 1) / p.unit + p.piece_units : 0;
          }
          if (lane == 31) prefix[p.batch] = incl;
        }
        __syncthreads();
      }
      // sequences with no tokens have no piece: out = 0, lse = -inf, flag = 0
      for (int b = blockIdx.x; b < p.batch; b += gridDim.x) {
        if (lens[b] != 0) continue;
        const long long r0 = (long long)b * p.hq;
        for (int e = tid; e < p.hq * D; e += blockDim.x)
          store_out(p.out, r0 * D + e, p.out_dtype, 0.f);
        for (int h = tid; h < p.hq; h += blockDim.x) {
          if (p.out_lse) p.out_lse[r0 + h] = -INFINITY;
          if (p.row_flags) p.row_flags[r0 + h] = 0;
        }
      }
    } else {
      __syncthreads();   // the barriers are initialised
    }
  }
  // a dependent launch (the recompute) may start its launch while this grid runs
  if (!p.recompute) pdl_launch_dependents();

  // Registers move from the producer warpgroup (two or four working warps) to the two
  // consumer warpgroups: 8 * 32 * kConsumerRegs + 4 * 32 * kProducerRegs equals the launch's
  // 12 * 32 * 168 (checked on the host before the first launch).
  if (warp < kConsumerWarps) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kConsumerRegs));
    consumer_role<T, D, G, MODE>(p, warp, lane);
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProducerRegs));
    producer_role<T, D, G>(p, &tmk, &tmv, warp, lane);
  }

  if (p.recompute) {
    // the recompute launch's last CTA resets the flagged list for the next step
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      if (atomicAdd(p.list_state + 1, 1) == (int)gridDim.x - 1) {
        p.list_state[0] = 0;
        p.list_state[1] = 0;
      }
    }
  }
}

template <typename T, int D, int G>
inline const void* pick_mode(int mode) {
  return mode == kSoftmaxSync      ? (const void*)&decode_split_kernel<T, D, G, 0>
         : mode == kSoftmaxUnified ? (const void*)&decode_split_kernel<T, D, G, 1>
                                   : (const void*)&decode_split_kernel<T, D, G, 2>;
}

template <typename T, int D>
inline const void* pick_kernel(int G, int mode) {
  switch (G) {
    case 1: return pick_mode<T, D, 1>(mode);
    case 2: return pick_mode<T, D, 2>(mode);
    case 4: return pick_mode<T, D, 4>(mode);
    case 8: return pick_mode<T, D, 8>(mode);
    default: return nullptr;
  }
}


}  // namespace da
