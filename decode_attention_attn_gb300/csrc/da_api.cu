// da_api.cu -- host side of the C ABI declared in include/decode_attn.h: problem validation,
// the launch plan (split policy, grid, pipeline depth, workspace layout), TMA tensor maps,
// kernel launches, error reporting and the debug gather hook; and the logit-histogram kernels
// of the phi calibration pass.
#include "decode_attn.h"

#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <set>
#include <string>
#include <utility>

#include "da_device.cuh"
#include "da_mma.cuh"
#include "da_scratch_cache.h"

namespace da {
const void* kernel_f32(int head_dim, int group, int mode);
const void* kernel_f16(int head_dim, int group, int mode);
const void* kernel_bf16(int head_dim, int group, int mode);
const void* kernel_fp8(int head_dim, int group, int mode, int kv_heads);

// The element offset the kernel reads token t of (b, kvh) from: the same token_row() the
// producer warp uses for its TMA box coordinates.
__global__ void debug_gather_kernel(const __grid_constant__ Params p) {
  const long long T = p.capacity;
  const long long total = (long long)p.batch * p.hkv * T;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(i % T);
    const int kvh = (int)((i / T) % p.hkv);
    const int b = (int)(i / T / p.hkv);
    long long off = -1;
    const int raw = p.seq_lens[b];
    const int n = raw < 0 ? 0 : (raw > p.capacity ? p.capacity : raw);
    if (t < n) {
      const int entry = p.paged ? p.block_table[(long long)b * p.max_blocks + t / p.page_size] : 0;
      const int z = token_row(p, b, t, entry);
      if (z >= 0) off = ((long long)z * p.hkv + kvh) * p.head_dim;
    }
    p.debug_offsets[i] = off;
  }
}

// ---- logit histogram: the calibration pass behind the choice of phi ----------------------
// "FlashDecoding++", Fig. 5 and "The Overflow and Precision Problem: Choosing phi": the
// distribution of the scaled logits x = scale * q[b, h] . K[b, t, h / G] over every row and
// token of a step, from which phi and the covered range are read. Not on the attention path:
// a plain memory-bound pass over K (one read of every used K row; q from L2 into registers).

constexpr int kHistThreads = 256;
constexpr int kHistWarps = kHistThreads / 32;
constexpr int kHistItemTokens = 64;   // tokens of one (b, kv head) per warp work item

// Bin of x: i = floor((x - lo) * inv_w) in fp32 gives counts[1 + i] for 0 <= i < nbins,
// counts[0] below lo, counts[nbins + 1] at or above the top edge and for NaN.
__device__ __forceinline__ int hist_bin(float x, float lo, float inv_w, int nbins) {
  if (x != x) return nbins + 1;
  if (x < lo) return 0;
  const float f = floorf((x - lo) * inv_w);
  return f >= (float)nbins ? nbins + 1 : 1 + (int)f;
}

// How a lane reads its share of a K row: 16-byte chunks of q's own storage type, or for an
// FP8 cache 8-byte chunks of E4M3 codes (so that a lane's q, bf16, stays 8 elements) with q
// read as bf16.
template <typename T>
struct HistIO {
  using Q = T;
  using KChunk = uint4;
  static constexpr int kEpc = Elem<T>::kPerChunk;
  __device__ __forceinline__ static void k_pairs(const uint4& c, f32x2* f) {
    Elem<T>::to_pairs(c, f);
  }
};
template <>
struct HistIO<fp8e4m3> {
  using Q = __nv_bfloat16;
  using KChunk = uint2;
  static constexpr int kEpc = 8;
  __device__ __forceinline__ static void k_pairs(const uint2& c, f32x2* f) {
    const uint32_t w[2] = {c.x, c.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t v = e4m3x2_to_f16x2(h ? w[i] >> 16 : w[i]);
        __half2 hv;
        memcpy(&hv, &v, 4);
        const float2 x = __half22float2(hv);
        f[2 * i + h] = f2_pack(x.x, x.y);
      }
    }
  }
};

// One warp per work item (64 tokens of one sequence and KV head); a K row is split over C
// lanes, 16 bytes each, so a warp reads R = 32 / C rows per load and U loads per lane are in
// flight before any arithmetic. The pass is latency-bound per warp, so the number of resident
// warps matters more than U: registers are capped for 4 blocks of 8 warps per SM (2-3 for
// G = 8, whose q takes up to 64 registers); on the bf16 GQA shapes U = 2 at 4 blocks streams
// K 1.5x faster than U = 8 at 2. The G query heads of the KV head sit in registers as fp32
// pairs. The C lanes' G partial dot products are summed by a transposing butterfly: each of
// the first log2 G exchange steps hands half of a lane's heads to its partner, so a row costs
// G - 1 + log2(C / G) shuffles instead of G log2 C; afterwards the top log2 G bits of the
// lane's index within its row name the head it holds the sum for.
template <typename T, int D, int G>
__global__ void __launch_bounds__(kHistThreads, G == 8 ? (sizeof(T) == 4 ? 3 : 2) : 4)
    logit_histogram_kernel(const __grid_constant__ Params p, const T* __restrict__ kc,
                           float scale, float lo, float inv_w, int nbins,
                           unsigned long long* __restrict__ counts) {
  extern __shared__ unsigned hist[];   // [nbins + 2]
  using IO = HistIO<T>;
  using Q = typename IO::Q;
  using KChunk = typename IO::KChunk;
  constexpr int EPC = IO::kEpc;             // K elements per lane chunk (16 or 8 bytes)
  constexpr int NP = EPC / 2;               // fp32 pairs per chunk
  constexpr int C = D / EPC;                // lanes per K row: 8, 16 or 32
  constexpr int R = 32 / C;                 // K rows per warp load
  constexpr int U = 2;                      // loads in flight per lane
  constexpr int LG = G == 1 ? 0 : (G == 2 ? 1 : (G == 4 ? 2 : 3));
  static_assert(G <= C, "a row's lanes must cover its heads");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / C, c = lane % C;
  const bool binner = (c % (C / G)) == 0;   // one lane of the C / G holding each head's sum

  for (int i = threadIdx.x; i < nbins + 2; i += kHistThreads) hist[i] = 0;
  __syncthreads();

  const int chunks = (p.capacity + kHistItemTokens - 1) / kHistItemTokens;
  const long long items = (long long)p.batch * p.hkv * chunks;
  for (long long it = (long long)blockIdx.x * kHistWarps + warp; it < items;
       it += (long long)gridDim.x * kHistWarps) {
    const int ch = (int)(it % chunks);
    const int kvh = (int)((it / chunks) % p.hkv);
    const int b = (int)(it / chunks / p.hkv);
    const int raw = p.seq_lens[b];
    const int n = raw < 0 ? 0 : (raw > p.capacity ? p.capacity : raw);
    const int t0 = ch * kHistItemTokens;
    if (t0 >= n) continue;                  // the same for the whole warp
    const int t1 = min(n, t0 + kHistItemTokens);

    f32x2 qp[G][NP];
    const Q* qg = static_cast<const Q*>(p.q) + ((long long)b * p.hq + (long long)kvh * G) * D;
#pragma unroll
    for (int g = 0; g < G; ++g)   // q's chunk c: EPC elements of Q, 16 bytes
      Elem<Q>::to_pairs(__ldg(reinterpret_cast<const uint4*>(qg + g * D) + c), qp[g]);

    for (int tb = t0; tb < t1; tb += R * U) {
      KChunk kr[U];
      bool ok[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int t = tb + u * R + sub;
        int z = -1;
        if (t < t1) {
          const int entry =
              p.paged ? p.block_table[(long long)b * p.max_blocks + t / p.page_size] : 0;
          z = token_row(p, b, t, entry);
        }
        ok[u] = z >= 0;
        kr[u] = KChunk{};
        if (ok[u])
          kr[u] = __ldg(reinterpret_cast<const KChunk*>(kc + ((long long)z * p.hkv + kvh) * D) + c);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        f32x2 kf[NP];
        IO::k_pairs(kr[u], kf);
        float v[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          f32x2 a = f2_mul(qp[g][0], kf[0]);
#pragma unroll
          for (int j = 1; j < NP; ++j) f2_fma(a, qp[g][j], kf[j]);
          float x0, x1;
          f2_unpack(a, x0, x1);
          v[g] = x0 + x1;
        }
#pragma unroll
        for (int s = 0; s < LG; ++s) {          // transposing steps: offsets C/2, C/4, ...
          const int o = C >> (s + 1);
          const int half = G >> (s + 1);
          const bool upper = (lane & o) != 0;
#pragma unroll
          for (int i = 0; i < half; ++i) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
          }
        }
#pragma unroll
        for (int o = C >> (LG + 1); o > 0; o >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
        if (ok[u] && binner) atomicAdd(&hist[hist_bin(scale * v[0], lo, inv_w, nbins)], 1u);
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < nbins + 2; i += kHistThreads)
    if (hist[i]) atomicAdd(&counts[i], (unsigned long long)hist[i]);
}

// ---- the histogram pass on the tensor cores (bf16 and FP8 caches) -------------------------
// Persistent CTAs, up to four per SM: a producer warp TMA-loads each work item's K rows (64
// tokens of one sequence and KV head, laid out and swizzled as the split kernel's tiles) and
// the group's q into a ring of stages; 4 consumer warps form S^T = K q^T for 8 rows of each
// 32-row half with the split kernel's MMAs (mma_logits, mma_logits_fp8), so a row's G logits
// cost a few MMA instructions instead of the CUDA-core pass's per-lane dot products and
// butterflies. The producer looks up the next item's pages while the current one waits for its
// stage; rows a bad block-table entry would have supplied are masked. Every wait is bounded: on
// a timeout the CTA stops, having counted less.
constexpr int kHmConsumerWarps = 4;
constexpr int kHmThreads = (kHmConsumerWarps + 1) * 32;   // + one producer warp
// an item: two halves of 8 rows per consumer warp, 16 rows = one MMA's tokens per warp
constexpr int kHmHalfTokens = kHmConsumerWarps * kTokensPerWarp;   // 32
constexpr int kHmItemTokens = 2 * kHmHalfTokens;                    // 64
constexpr int kHmMaxStages = 8;
constexpr int kHmMaxBatchSmem = 4096;                      // lengths kept in shared memory

struct HmLayout {
  uint32_t bar_off, flag_off, lens_off, stage_off, stage_bytes, q_off, mask_off, total;
};
// es: K bytes per element; lens: sequence lengths held in shared memory
__host__ __device__ inline HmLayout hm_layout(int D, int G, int es, int nbins, int stages,
                                              int lens) {
  HmLayout L;
  L.bar_off = align_up((uint32_t)(nbins + 2) * 4u, 16);
  L.flag_off = L.bar_off + 2u * stages * 8u;
  L.lens_off = L.flag_off + 16u;
  L.stage_off = align_up(L.lens_off + (uint32_t)lens * 4u, 1024);
  L.q_off = (uint32_t)kHmItemTokens * D * es;
  L.mask_off = L.q_off + align_up((uint32_t)G * D * 2u, 16);
  L.stage_bytes = align_up(L.mask_off + 16u, 1024);
  L.total = L.stage_off + (uint32_t)stages * L.stage_bytes + 1024;   // + aligning the base
  return L;
}

// Bits [lo, hi) of a 64-bit word (both clamped to [0, 64]).
__device__ __forceinline__ unsigned long long bit_range(int lo, int hi) {
  lo = max(lo, 0);
  hi = min(hi, 64);
  if (hi <= lo) return 0ull;
  const unsigned long long up = hi == 64 ? ~0ull : (1ull << hi) - 1ull;
  return up & ~((1ull << lo) - 1ull);
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(kHmThreads, 4)
    logit_histogram_mma_kernel(const __grid_constant__ Params p,
                               const __grid_constant__ CUtensorMap tmk, float lo, float inv_w,
                               int nbins, unsigned long long* __restrict__ counts, int stages) {
  extern __shared__ uint8_t hm_raw[];
  constexpr bool kFp8 = std::is_same<T, fp8e4m3>::value;
  constexpr uint32_t kRowBytes = (uint32_t)D * sizeof(T);
  constexpr uint32_t kQBytes = (uint32_t)G * D * 2u;   // bf16 q
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nlens = p.batch <= kHmMaxBatchSmem ? p.batch : 0;
  const HmLayout L = hm_layout(D, G, sizeof(T), nbins, stages, nlens);
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(hm_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned* hist = reinterpret_cast<unsigned*>(sm);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L.bar_off);
  uint64_t* empty = full + stages;
  int& abort_flag = *reinterpret_cast<int*>(sm + L.flag_off);
  int* lens = reinterpret_cast<int*>(sm + L.lens_off);
  uint8_t* ring = sm + L.stage_off;

  for (int i = tid; i < nbins + 2; i += kHmThreads) hist[i] = 0;
  for (int i = tid; i < nlens; i += kHmThreads) {
    const int raw = __ldg(p.seq_lens + i);
    lens[i] = raw < 0 ? 0 : (raw > p.capacity ? p.capacity : raw);
  }
  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kHmConsumerWarps);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // Items it = (b * H_kv + kvh) * chunks + ch (fewer than 2^31, checked on the host); this
  // CTA's are blockIdx.x, + gridDim.x, ...; next_item() skips those past their sequence's end.
  const int chunks = (p.capacity + kHmItemTokens - 1) / kHmItemTokens;
  const int items = p.batch * p.hkv * chunks;
  auto seq_len = [&](int b) {
    if (nlens) return lens[b];
    const int raw = __ldg(p.seq_lens + b);
    return raw < 0 ? 0 : (raw > p.capacity ? p.capacity : raw);
  };
  auto next_item = [&](int it) {
    for (; it < items; it += gridDim.x)
      if ((it % chunks) * kHmItemTokens < seq_len(it / chunks / p.hkv)) break;
    return it < items ? it : items;
  };
  const uint32_t NS = (uint32_t)stages;
  uint32_t k = 0;   // stages used so far (the same count in every warp)
  if (warp == kHmConsumerWarps) {
    const uint64_t pol = make_evict_first_policy();
    const int box = p.box_tokens;
    auto lookup = [&](int it) {   // the cache row of box `lane` of item it (-1: none or bad)
      if (it >= items) return -1;
      const int ch = it % chunks, b = it / chunks / p.hkv;
      const int t0 = ch * kHmItemTokens, t1 = min(seq_len(b), t0 + kHmItemTokens);
      const int t = t0 + lane * box;
      if (t >= t1) return -1;
      const int entry =
          p.paged ? __ldg(p.block_table + (long long)b * p.max_blocks + t / p.page_size) : 0;
      return token_row(p, b, t, entry);
    };
    uint32_t issued = 0;
    int it = next_item(blockIdx.x);
    int z = lookup(it);
    while (it < items) {
      const int nxt = next_item(it + gridDim.x);
      const int z_next = lookup(nxt);   // in flight while this item waits for its stage
      const int ch = it % chunks, kvh = (it / chunks) % p.hkv, b = it / chunks / p.hkv;
      const int t0 = ch * kHmItemTokens, t1 = min(seq_len(b), t0 + kHmItemTokens);
      const uint32_t slot = k % NS, ph = (k / NS) & 1u;
      ++k;
      bool stop = !mbar_wait(&empty[slot], ph ^ 1u, p.wait_limit_ns) ||
                  *reinterpret_cast<volatile int*>(&abort_flag) != 0;
      stop = __any_sync(0xffffffffu, stop);
      if (stop) {
        if (lane == 0) atomicExch(&abort_flag, 1);
        break;
      }
      uint8_t* st = ring + slot * L.stage_bytes;
      const int nbox = (t1 - t0 + box - 1) / box;   // lane i loads box i: rows [i box, (i+1) box)
      const unsigned bad = __ballot_sync(0xffffffffu, lane < nbox && z < 0);
      if (lane == 0) {
        // the tile rows below t1, less the boxes of bad entries (rare)
        unsigned long long m0 = bit_range(0, t1 - t0), m1 = bit_range(0, t1 - t0 - 64);
        for (unsigned rest = bad; rest != 0u; rest &= rest - 1u) {
          const int i = __ffs(rest) - 1;
          m0 &= ~bit_range(i * box, (i + 1) * box);
          m1 &= ~bit_range(i * box - 64, (i + 1) * box - 64);
        }
        reinterpret_cast<unsigned long long*>(st + L.mask_off)[0] = m0;
        reinterpret_cast<unsigned long long*>(st + L.mask_off)[1] = m1;
        mbar_arrive_expect_tx(&full[slot], (uint32_t)nbox * box * kRowBytes + kQBytes);
        const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(p.q) +
                                  ((long long)b * p.hq + (long long)kvh * G) * D;
        bulk_load(st + L.q_off, qg, kQBytes, &full[slot]);
      }
      __syncwarp();
      if (lane < nbox) {
        // a bad entry reads past the pool (zero fill); its rows are masked
        const int zz = z >= 0 ? z : p.num_blocks * p.page_size;
        uint8_t* dst = st + (uint32_t)lane * box * kRowBytes;
        if constexpr (kFp8)
          tma_load_3d(dst, &tmk, &full[slot], 0, kvh, zz, pol);
        else
          tma_load_4d(dst, &tmk, &full[slot], 0, 0, kvh, zz, pol);
      }
      issued = k;
      __syncwarp();
      it = nxt;
      z = z_next;
    }
    // never leave with copies in flight
    if (lane == 0) {
      const uint32_t first = issued > NS ? issued - NS : 0u;
      for (uint32_t kk = first; kk < issued; ++kk)
        mbar_wait(&full[kk % NS], (kk / NS) & 1u, p.wait_limit_ns);
    }
  } else {
    // consumers: rows row0 .. row0 + 7 of each 64-row half, as a split-kernel warp
    const int row0 = warp * kTokensPerWarp;
    const std::conditional_t<kFp8, NoMmaLane, MmaLane<D>> ml(row0, lane);
    const int hp = 2 * (lane & 3), tr = row0 + (lane >> 2);
    for (int it = next_item(blockIdx.x); it < items; it = next_item(it + gridDim.x)) {
      const uint32_t slot = k % NS, ph = (k / NS) & 1u;
      ++k;
      bool stop = !mbar_wait(&full[slot], ph, p.wait_limit_ns);
      stop = __any_sync(0xffffffffu, stop);
      if (stop) {
        if (lane == 0) atomicExch(&abort_flag, 1);
        break;
      }
      const uint8_t* st = ring + slot * L.stage_bytes;
      const unsigned long long* mask =
          reinterpret_cast<const unsigned long long*>(st + L.mask_off);
      const uint32_t kt[2] = {smem_u32(st), smem_u32(st + kHmHalfTokens * kRowBytes)};
      MmaState<D, G> ms;
      float sa[4], sb[4];
      if constexpr (kFp8) {
        mma_load_q_fp8<D, G>(p, ms, st + L.q_off, lane);   // qmul: the logit scale * 2^-s
        mma_logits_fp8<D, G, 1>(ms, kt, row0, lane, sa, sb);
      } else {
        mma_load_q<D, G>(ms, st + L.q_off, lane);
        ms.qmul = p.qscale;
        mma_logits<D, G>(ms, ml, kt, sa, sb);
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {   // token tr of half c / 2, head hp + c % 2
        const int h = hp + (c & 1);
        const int row = (c >> 1) * kHmHalfTokens + tr;   // tile row
        const bool ok = h < G && ((mask[row >> 6] >> (row & 63)) & 1ull);
        if (ok) atomicAdd(&hist[hist_bin((sa[c] + sb[c]) * ms.qmul, lo, inv_w, nbins)], 1u);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }
  }
  __syncthreads();
  for (int i = tid; i < nbins + 2; i += kHmThreads)
    if (hist[i]) atomicAdd(&counts[i], (unsigned long long)hist[i]);
}

template <typename T, int D>
const void* histogram_mma_kernel_for_d(int G) {
  switch (G) {
    case 1: return reinterpret_cast<const void*>(&logit_histogram_mma_kernel<T, D, 1>);
    case 2: return reinterpret_cast<const void*>(&logit_histogram_mma_kernel<T, D, 2>);
    case 4: return reinterpret_cast<const void*>(&logit_histogram_mma_kernel<T, D, 4>);
    case 8: return reinterpret_cast<const void*>(&logit_histogram_mma_kernel<T, D, 8>);
    default: return nullptr;
  }
}

template <typename T>
const void* histogram_mma_kernel_for(int D, int G) {
  return D == 64 ? histogram_mma_kernel_for_d<T, 64>(G)
                 : (D == 128 ? histogram_mma_kernel_for_d<T, 128>(G) : nullptr);
}

template <typename T, int D>
const void* histogram_kernel_for_d(int G) {
  switch (G) {
    case 1: return reinterpret_cast<const void*>(&logit_histogram_kernel<T, D, 1>);
    case 2: return reinterpret_cast<const void*>(&logit_histogram_kernel<T, D, 2>);
    case 4: return reinterpret_cast<const void*>(&logit_histogram_kernel<T, D, 4>);
    case 8: return reinterpret_cast<const void*>(&logit_histogram_kernel<T, D, 8>);
    default: return nullptr;
  }
}

template <typename T>
const void* histogram_kernel_for(int D, int G) {
  return D == 64 ? histogram_kernel_for_d<T, 64>(G)
                 : (D == 128 ? histogram_kernel_for_d<T, 128>(G) : nullptr);
}
}  // namespace da

using namespace da;

struct da_plan {
  da_problem prob;
  int num_sms;
  int group, es, unit, box_tokens, capacity, n_groups, piece_units;
  int kv_es;                    // K / V bytes per element (1: FP8 E4M3 cache; else es)
  int hp;                       // KV heads per split-kernel group (2: packed FP8 pairs)
  int sgroup;                   // query heads per split-kernel group (group * hp)
  int policy, num_splits;       // the plan's default split choice
  int narrow;                   // the device schedule's arithmetic fits 32 bits
  int grid;                     // balanced grid (or the default uniform grid)
  int recompute_splits, max_splits;
  int stages, batch_smem;
  size_t smem_bytes;
  long long slots;
  size_t off_counters, off_list, off_list_state, off_status, off_stats;
  size_t off_part_flags, off_part_l, off_part_o, zero_bytes, ws_bytes;
};

namespace {

thread_local std::string g_cuda_error;

int cuda_fail(cudaError_t e, const char* what) {
  g_cuda_error = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return DA_ERR_CUDA;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Grid for `items` equal uniform-split items: the fewest CTAs that still give every CTA the
// smallest possible number of items (512 items on 152 SMs: 128 CTAs of 4 rather than a mix
// of 3 and 4, whose slowest CTAs would set the step time).
int uniform_grid(long long items, int sms) {
  if (items <= 0) return 1;
  const long long per = (items + sms - 1) / sms;
  return (int)((items + per - 1) / per);
}

int elem_size(int dt) { return dt == DA_F32 ? 4 : 2; }

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int validate_problem(const da_problem& p) {
  if (p.batch < 1 || p.num_q_heads < 1 || p.num_kv_heads < 1) return DA_ERR_INVALID_ARG;
  if (p.num_q_heads % p.num_kv_heads) return DA_ERR_INVALID_ARG;
  const int G = p.num_q_heads / p.num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return DA_ERR_UNSUPPORTED;
  if (p.head_dim != 64 && p.head_dim != 128) return DA_ERR_UNSUPPORTED;
  if (p.qkv_dtype < DA_F32 || p.qkv_dtype > DA_BF16) return DA_ERR_UNSUPPORTED;
  if (p.out_dtype < DA_F32 || p.out_dtype > DA_BF16) return DA_ERR_UNSUPPORTED;
  if (p.mode != DA_SOFTMAX_SYNC && p.mode != DA_SOFTMAX_UNIFIED &&
      p.mode != DA_SOFTMAX_UNIFIED_LOCAL)
    return DA_ERR_INVALID_ARG;
  if (p.num_sms < 0) return DA_ERR_INVALID_ARG;
  if (p.paged) {
    if (!is_pow2(p.page_size) || p.page_size < 8 || p.page_size > 256) return DA_ERR_UNSUPPORTED;
    if (p.max_blocks_per_seq < 1 || p.num_physical_blocks < 1) return DA_ERR_INVALID_ARG;
    if ((long long)p.num_physical_blocks * p.page_size >= (1ll << 31)) return DA_ERR_INVALID_ARG;
    if ((long long)p.max_blocks_per_seq * p.page_size >= (1ll << 31)) return DA_ERR_INVALID_ARG;
  } else {
    if (p.max_seq_len < 1) return DA_ERR_INVALID_ARG;
    if ((long long)p.batch * p.max_seq_len >= (1ll << 31)) return DA_ERR_INVALID_ARG;
  }
  if (p.kv_fp8 != 0 && p.kv_fp8 != 1) return DA_ERR_INVALID_ARG;
  if (p.debug_stall_stage < 0) return DA_ERR_INVALID_ARG;
  if (p.kv_fp8) {
    // FP8 caches run on the tensor-core consumers with bf16 q
    if (p.qkv_dtype != DA_BF16) return DA_ERR_UNSUPPORTED;
    if (!std::isfinite(p.k_scale) || !std::isfinite(p.v_scale) || !(p.k_scale > 0.f) ||
        !(p.v_scale > 0.f))
      return DA_ERR_INVALID_ARG;
  }
  if (p.mode != DA_SOFTMAX_SYNC) {
    if (!std::isfinite(p.unified_max) || !std::isfinite(p.range_lo) ||
        !std::isfinite(p.range_hi) || !(p.range_lo < p.range_hi))
      return DA_ERR_INVALID_ARG;
  }
  return DA_OK;
}

const void* kernel_for(const da_plan& pl, int mode) {
  if (pl.prob.kv_fp8) return kernel_fp8(pl.prob.head_dim, pl.sgroup, mode, pl.hp);
  switch (pl.prob.qkv_dtype) {
    case DA_F32: return kernel_f32(pl.prob.head_dim, pl.sgroup, mode);
    case DA_F16: return kernel_f16(pl.prob.head_dim, pl.sgroup, mode);
    case DA_BF16: return kernel_bf16(pl.prob.head_dim, pl.sgroup, mode);
  }
  return nullptr;
}

std::mutex g_attr_mu;
std::set<std::pair<int, const void*>> g_attr_done;

int ensure_smem_attr(const void* fn, size_t smem) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lk(g_attr_mu);
  if (g_attr_done.count({dev, fn})) return DA_OK;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimit);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
  if (smem > 0) {
    // The split kernels redistribute registers with setmaxnreg; that is only safe when every
    // thread was launched with kLaunchRegs registers.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncGetAttributes");
    if (fa.numRegs != kLaunchRegs || fa.maxThreadsPerBlock < kThreads) {
      g_cuda_error = "split kernel built with " + std::to_string(fa.numRegs) +
                     " registers per thread; the register split needs " +
                     std::to_string(kLaunchRegs);
      return DA_ERR_CUDA;
    }
  }
  g_attr_done.insert({dev, fn});
  return DA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// [tokens, Hkv, D] view of a K or V cache; one box = box_tokens rows of one KV head. The
// bf16 tensor-core kernels read the tile with ldmatrix and need the 128-byte swizzle, whose
// rows are at most 128 bytes: for them the view is 4-D, [tokens, Hkv, D / 64, 64]. FP8 tiles
// keep the 3-D view (a row of D = 64 or 128 bytes), 128-byte-swizzled when D = 128.
int make_kv_map(const da_plan& pl, const void* base, bool swizzled, int hp,
                CUtensorMap* map) {
  auto fn = encode_fn();
  if (!fn) {
    g_cuda_error = "cuTensorMapEncodeTiled is not available from the driver";
    return DA_ERR_CUDA;
  }
  const da_problem& p = pl.prob;
  const cuuint64_t tokens = p.paged ? (cuuint64_t)p.num_physical_blocks * p.page_size
                                    : (cuuint64_t)p.batch * p.max_seq_len;
  const cuuint64_t dims[3] = {(cuuint64_t)p.head_dim, (cuuint64_t)p.num_kv_heads, tokens};
  const int es = pl.kv_es;
  const cuuint64_t strides[2] = {(cuuint64_t)p.head_dim * es,
                                 (cuuint64_t)p.num_kv_heads * p.head_dim * es};
  // a box holds the rows of hp KV heads (a split-kernel group) of box_tokens tokens
  const cuuint32_t box[3] = {(cuuint32_t)p.head_dim, (cuuint32_t)hp, (cuuint32_t)pl.box_tokens};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  // L2 fills no wider than a KV row: with a wider promotion every box row also pulls in the
  // neighbouring head's row, which a paged gather seldom reads before it is evicted (FP8 rows
  // of 128 bytes under 256-byte promotion: 1.48x the algorithmic DRAM bytes on the paged
  // batch)
  const long long row_bytes = (long long)p.head_dim * es;
  const CUtensorMapL2promotion l2p = row_bytes >= 256   ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                                     : row_bytes >= 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                                        : CU_TENSOR_MAP_L2_PROMOTION_L2_64B;
  const CUtensorMapDataType dt = es == 4   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : es == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                                           : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUresult r;
  if (swizzled && es == 2) {
    const cuuint64_t dims4[4] = {64u, (cuuint64_t)p.head_dim / 64u, (cuuint64_t)p.num_kv_heads,
                                 tokens};
    const cuuint64_t strides4[3] = {64u * es, (cuuint64_t)p.head_dim * es,
                                    (cuuint64_t)p.num_kv_heads * p.head_dim * es};
    const cuuint32_t box4[4] = {64u, (cuuint32_t)p.head_dim / 64u, 1u,
                                (cuuint32_t)pl.box_tokens};
    const cuuint32_t estr4[4] = {1u, 1u, 1u, 1u};
    r = fn(map, dt, 4, const_cast<void*>(base), dims4, strides4, box4, estr4,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           l2p, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    const bool swz8 = swizzled && es == 1 && p.head_dim == 128;
    r = fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, swz8 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
           l2p, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) {
    g_cuda_error = "cuTensorMapEncodeTiled failed with CUresult " + std::to_string((int)r);
    return DA_ERR_CUDA;
  }
  return DA_OK;
}

void fill_common(const da_plan& pl, Params& k, const int32_t* block_table,
                 const int32_t* seq_lens, void* ws) {
  const da_problem& p = pl.prob;
  std::memset(&k, 0, sizeof k);
  char* w = static_cast<char*>(ws);
  k.block_table = block_table;
  k.seq_lens = seq_lens;
  if (w) {
    k.counters = reinterpret_cast<int32_t*>(w + pl.off_counters);
    k.flag_list = reinterpret_cast<int32_t*>(w + pl.off_list);
    k.list_state = reinterpret_cast<int32_t*>(w + pl.off_list_state);
    k.status = reinterpret_cast<int32_t*>(w + pl.off_status);
    k.stats = reinterpret_cast<unsigned long long*>(w + pl.off_stats);
    k.part_flags = reinterpret_cast<uint32_t*>(w + pl.off_part_flags);
    k.part_l = reinterpret_cast<float*>(w + pl.off_part_l);
    k.part_o = reinterpret_cast<float*>(w + pl.off_part_o);
  }
  k.batch = p.batch;
  k.hq = p.num_q_heads;
  k.hkv = p.num_kv_heads;
  k.group = pl.group;
  k.head_dim = p.head_dim;
  k.paged = p.paged ? 1 : 0;
  k.page_size = p.paged ? p.page_size : 1;
  k.max_blocks = p.paged ? p.max_blocks_per_seq : 0;
  k.num_blocks = p.paged ? p.num_physical_blocks : 0;
  k.max_seq_len = p.paged ? 0 : p.max_seq_len;
  k.capacity = pl.capacity;
  k.unit = pl.unit;
  k.piece_units = pl.piece_units;
  k.box_tokens = pl.box_tokens;
  k.out_dtype = p.out_dtype;
  k.v_scale = 1.f;
  k.n_groups = pl.n_groups;
  k.stages = pl.stages;
  k.batch_smem = pl.batch_smem;
  k.narrow = pl.narrow;
  k.stall_stage = p.debug_stall_stage;
  k.wait_limit_ns = p.debug_stall_stage ? kTestWaitLimitNs : kWaitLimitNs;
}

int status_to_error(int s) {
  if (s & kStatusBadBlockTable) return DA_ERR_BAD_BLOCK_TABLE;
  if (s & kStatusBadSeqLen) return DA_ERR_BAD_SEQ_LEN;
  if (s & kStatusTimeout) return DA_ERR_DEVICE_TIMEOUT;
  return DA_OK;
}

}  // namespace

extern "C" {

int decode_attn_abi_version(void) { return DECODE_ATTN_ABI_VERSION; }

const char* decode_attn_strerror(int code) {
  switch (code) {
    case DA_OK: return "success";
    case DA_ERR_INVALID_ARG: return "invalid argument";
    case DA_ERR_UNSUPPORTED: return "unsupported head_dim, group size, dtype or page size";
    case DA_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than the plan requires";
    case DA_ERR_BAD_BLOCK_TABLE: return "a used block-table entry lies outside the page pool";
    case DA_ERR_CUDA: return g_cuda_error.empty() ? "CUDA error" : g_cuda_error.c_str();
    case DA_ERR_DEVICE_TIMEOUT: return "a device pipeline wait ran out of time";
    case DA_ERR_BAD_SEQ_LEN: return "a sequence length is negative or above the cache capacity";
    case DA_ERR_HISTOGRAM_RANGE:
      return "a tail of the requested coverage lies outside the histogram's range";
    case DA_ERR_RANGE_TOO_WIDE:
      return "the covered logit range is wider than allowed: use DA_SOFTMAX_SYNC";
    default: return "unknown error code";
  }
}

int decode_attn_plan(const da_problem* problem, int num_splits, da_plan** plan_out,
                     size_t* workspace_bytes_out) {
  if (!problem || !plan_out || num_splits < 0) return DA_ERR_INVALID_ARG;
  *plan_out = nullptr;
  const int v = validate_problem(*problem);
  if (v != DA_OK) return v;
  da_plan* pl = new (std::nothrow) da_plan();
  if (!pl) return DA_ERR_INVALID_ARG;
  pl->prob = *problem;
  const da_problem& p = pl->prob;
  int sms = p.num_sms;
  if (sms == 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
      delete pl;
      return cuda_fail(e, "querying the SM count");
    }
  }
  pl->num_sms = sms;
  pl->group = p.num_q_heads / p.num_kv_heads;
  pl->es = elem_size(p.qkv_dtype);
  pl->kv_es = p.kv_fp8 ? 1 : pl->es;
  pl->unit = p.paged ? std::max(16, p.page_size) : 16;
  pl->box_tokens = p.paged ? std::min(p.page_size, kStageTokens) : kStageTokens;
  pl->capacity = p.paged ? p.max_blocks_per_seq * p.page_size : p.max_seq_len;
  // FP8 caches with groups of 4 query heads over pairs of KV heads: the split kernel can take
  // a pair at once (8 query heads, all of the tensor-core consumer's columns, and one 256-byte
  // read of a token's two rows at d = 128). It does where the step is large: four packed
  // groups per SM or more, or a cache of 128 MiB and more. On a smaller step spread over many
  // CTAs per group, merging twice the partials of twice the heads costs more than the faster
  // stream saves (batch 1, 8 KV heads: 6 us slower at 8K tokens, 10 us faster at 128K).
  pl->hp = 1;
  if (p.kv_fp8 && pl->group == 4 && p.num_kv_heads % 2 == 0) {
    const long long packed = (long long)p.batch * (p.num_kv_heads / 2);
    const long long cache_bytes =
        2LL * p.batch * pl->capacity * p.num_kv_heads * p.head_dim;   // K + V, one byte each
    if (packed * 4 >= sms || cache_bytes >= (128LL << 20)) pl->hp = 2;
  }
  pl->sgroup = pl->group * pl->hp;
  pl->n_groups = p.batch * (p.num_kv_heads / pl->hp);
  {
    // K + V of one unit of a group
    const long long unit_bytes = 2LL * pl->unit * p.head_dim * pl->kv_es * pl->hp;
    pl->piece_units = (int)((kPieceCostBytes + unit_bytes / 2) / unit_bytes);
  }
  const long long units_max = (pl->capacity + pl->unit - 1) / pl->unit;
  const long long w_max = (long long)pl->n_groups * units_max;
  pl->batch_smem = p.batch <= kMaxBatchSmem ? p.batch : 0;

  // the merge stages one weight per (split, head) in 8 * d * G floats of shared memory
  const int split_cap = kConsumerWarps * p.head_dim;
  if (num_splits > split_cap) {
    delete pl;
    return DA_ERR_UNSUPPORTED;
  }
  if (num_splits > 0) {
    pl->policy = kUniform;
    pl->num_splits = num_splits;
  } else if (pl->batch_smem > 0) {
    // Balanced shares: every persistent CTA gets the same number of KV tokens. A sequence
    // is split only where a CTA boundary falls inside it, so small batches split finely and
    // batches that fill the SMs on their own barely split.
    pl->policy = kBalanced;
    pl->num_splits = 0;
  } else {
    pl->policy = kUniform;
    pl->num_splits = (int)std::min<long long>(units_max, std::max(1, (sms + pl->n_groups - 1) / pl->n_groups));
  }
  const long long min_ctas = (w_max + kMinUnitsPerCta - 1) / kMinUnitsPerCta;
  pl->grid = pl->policy == kBalanced
                 ? (int)std::max<long long>(1, std::min<long long>(sms, min_ctas))
                 : uniform_grid((long long)pl->n_groups * pl->num_splits, sms);
  pl->recompute_splits = (int)std::min<long long>(
      units_max, std::max(1, (sms + pl->n_groups - 1) / pl->n_groups));
  const long long need_uniform =
      (long long)pl->n_groups * std::max(pl->recompute_splits, pl->policy == kUniform ? pl->num_splits : 1);
  pl->slots = std::max<long long>((long long)sms + pl->n_groups, need_uniform);
  pl->max_splits = (int)std::min<long long>(split_cap, pl->slots / pl->n_groups);
  {
    // the largest unit index (balanced) or item count (uniform splits, any num_splits up to
    // max_splits, and the recompute pass) times the CTA count must stay below 2^31 for the
    // device's 32-bit schedule arithmetic
    const long long units = (long long)pl->n_groups * (units_max + pl->piece_units);
    const long long items = (long long)pl->n_groups * std::max(pl->max_splits, pl->recompute_splits);
    const long long ctas = std::max<long long>(sms, 1);
    pl->narrow = (units + 1) * ctas < (1ll << 31) && (items + 1) * ctas < (1ll << 31) ? 1 : 0;
  }

  // deepest pipeline that fits the per-CTA shared memory limit
  pl->stages = 0;
  for (int s = kMaxStages; s >= 2; --s) {
    const Layout L =
        make_layout(p.head_dim, pl->sgroup, pl->es, s, pl->batch_smem, pl->kv_es, pl->hp);
    if (L.total <= kSmemLimit) {
      pl->stages = s;
      pl->smem_bytes = L.total;
      break;
    }
  }
  if (pl->stages == 0) {
    delete pl;
    return DA_ERR_UNSUPPORTED;
  }

  // Workspace: the counters, the flagged list, status and statistics (zeroed once, left at
  // zero by every run), then the partials (no initial value needed).
  const int G = pl->sgroup, D = p.head_dim;
  size_t off = 0;
  pl->off_counters = off;
  off = align256(off + (size_t)pl->n_groups * 4);
  pl->off_list = off;
  off = align256(off + (size_t)pl->n_groups * 4);
  pl->off_list_state = off;      // 2 x int32
  pl->off_status = off + 16;     // int32
  pl->off_stats = off + 24;      // 4 x uint64
  off = align256(off + 56);
  pl->zero_bytes = off;
  pl->off_part_flags = off;
  off = align256(off + (size_t)pl->slots * 4);
  pl->off_part_l = off;
  off = align256(off + (size_t)pl->slots * G * 4);
  pl->off_part_o = off;
  off = align256(off + (size_t)pl->slots * G * D * 4);
  pl->ws_bytes = off;

  *plan_out = pl;
  if (workspace_bytes_out) *workspace_bytes_out = pl->ws_bytes;
  return DA_OK;
}

// Largest and smallest piece (tokens) of a step whose sequences are all at capacity, under
// the plan's default policy: the host-side image of the device's schedule.
void full_step_pieces(const da_plan& pl, int* mx, int* mn) {
  const long long cap = pl.capacity, unit = pl.unit;
  long long hi = 0, lo = 0;
  if (pl.policy == kUniform) {
    const long long S = pl.num_splits;
    const long long ts = ((cap + S - 1) / S + unit - 1) / unit * unit;
    hi = std::min(ts, cap);
    lo = cap - (S - 1) * ts > 0 ? std::min(hi, cap - (S - 1) * ts) : 0;
    for (long long sp = 0; sp < S; ++sp) {   // splits past the end are empty
      const long long t0 = std::min(cap, sp * ts), t1 = std::min(cap, t0 + ts);
      lo = sp == 0 ? t1 - t0 : std::min(lo, t1 - t0);
    }
  } else {
    const long long per = (cap + unit - 1) / unit + pl.piece_units;
    const long long W = (long long)pl.n_groups * per;
    const long long P = std::min<long long>(pl.grid, W);
    lo = cap;
    for (long long c = 0; c < P; ++c) {
      const long long u0 = c * W / P, u1 = (c + 1) * W / P;
      for (long long g = u0 / per; g * per < u1 && g < pl.n_groups; ++g) {
        const long long rs = g * per + pl.piece_units, ge = (g + 1) * per;
        const long long a = std::max(u0, rs), b = std::min(u1, ge);
        if (b <= a) continue;
        const long long t = std::min(cap, (b - rs) * unit) - (a - rs) * unit;
        hi = std::max(hi, t);
        lo = std::min(lo, t);
      }
    }
  }
  *mx = (int)hi;
  *mn = (int)lo;
}

int decode_attn_plan_info(const da_plan* plan, da_plan_info* info) {
  if (!plan || !info) return DA_ERR_INVALID_ARG;
  full_step_pieces(*plan, &info->split_tokens, &info->split_tokens_min);
  info->grid_ctas = plan->grid;
  info->num_splits = plan->policy == kBalanced ? 0 : plan->num_splits;
  info->unit_tokens = plan->unit;
  info->stage_tokens = kStageTokens;
  info->stages = plan->stages;
  info->recompute_splits = plan->recompute_splits;
  info->max_splits = plan->max_splits;
  info->workspace_bytes = plan->ws_bytes;
  info->smem_bytes = plan->smem_bytes;
  info->kv_heads_per_group = plan->hp;
  return DA_OK;
}

void decode_attn_destroy(da_plan* plan) { delete plan; }

int decode_attn_workspace_init(const da_plan* plan, void* workspace, size_t workspace_bytes,
                               void* cuda_stream) {
  if (!plan || !workspace || !aligned(workspace, 256)) return DA_ERR_INVALID_ARG;
  if (workspace_bytes < plan->ws_bytes) return DA_ERR_WORKSPACE_TOO_SMALL;
  const cudaError_t e =
      cudaMemsetAsync(workspace, 0, plan->zero_bytes, static_cast<cudaStream_t>(cuda_stream));
  return e == cudaSuccess ? DA_OK : cuda_fail(e, "cudaMemsetAsync(workspace)");
}

int decode_attn_run(const da_plan* plan, const void* q, const void* k_cache,
                    const void* v_cache, const int32_t* block_table, const int32_t* seq_lens,
                    float scale, int num_splits, void* out, float* out_lse,
                    uint8_t* row_flags, void* workspace, size_t workspace_bytes,
                    void* cuda_stream, da_stats* stats) {
  da_run_args a;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.scale = scale;
  a.num_splits = num_splits;
  a.out = out;
  a.out_lse = out_lse;
  a.row_flags = row_flags;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.cuda_stream = cuda_stream;
  a.stats = stats;
  a.split_event_begin = nullptr;
  a.split_event_end = nullptr;
  return decode_attn_run_ex(plan, &a);
}

int decode_attn_run_ex(const da_plan* plan, const da_run_args* args) {
  if (!plan || !args) return DA_ERR_INVALID_ARG;
  const void* q = args->q;
  const void* k_cache = args->k_cache;
  const void* v_cache = args->v_cache;
  const int32_t* block_table = args->block_table;
  const int32_t* seq_lens = args->seq_lens;
  const float scale = args->scale;
  const int num_splits = args->num_splits;
  void* out = args->out;
  float* out_lse = args->out_lse;
  uint8_t* row_flags = args->row_flags;
  void* workspace = args->workspace;
  const size_t workspace_bytes = args->workspace_bytes;
  void* cuda_stream = args->cuda_stream;
  da_stats* stats = args->stats;
  if ((args->split_event_begin == nullptr) != (args->split_event_end == nullptr))
    return DA_ERR_INVALID_ARG;
  const da_plan& pl = *plan;
  const da_problem& p = pl.prob;
  if (!q || !k_cache || !v_cache || !seq_lens || !out || !workspace) return DA_ERR_INVALID_ARG;
  if (p.paged ? !block_table : block_table != nullptr) return DA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(workspace, 256) || !aligned(seq_lens, 4) || !aligned(out, 16) ||
      (out_lse && !aligned(out_lse, 4)) || (block_table && !aligned(block_table, 4)))
    return DA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return DA_ERR_INVALID_ARG;
  if (num_splits < -1) return DA_ERR_INVALID_ARG;
  if (workspace_bytes < pl.ws_bytes) return DA_ERR_WORKSPACE_TOO_SMALL;
  int policy = pl.policy, S = pl.num_splits;
  if (num_splits == 0) {
    if (pl.batch_smem == 0) return DA_ERR_UNSUPPORTED;
    policy = kBalanced;
    S = 0;
  } else if (num_splits > 0) {
    if (num_splits > pl.max_splits) return DA_ERR_WORKSPACE_TOO_SMALL;
    policy = kUniform;
    S = num_splits;
  }
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  const bool unified = p.mode == DA_SOFTMAX_UNIFIED;   // the recompute launch follows

  // tensor-core kernels (both modes, so the recompute pass too) read 128-byte-swizzled tiles
  const bool mma = uses_mma(pl.kv_es, p.qkv_dtype == DA_F16, pl.sgroup);
  CUtensorMap tmk, tmv;
  int rc = make_kv_map(pl, k_cache, mma, pl.hp, &tmk);
  if (rc == DA_OK) rc = make_kv_map(pl, v_cache, mma, pl.hp, &tmv);
  if (rc != DA_OK) return rc;

  Params kp;
  fill_common(pl, kp, block_table, seq_lens, workspace);
  kp.hkv = p.num_kv_heads / pl.hp;   // the split kernel's groups (packed FP8: KV head pairs)
  kp.group = pl.sgroup;
  kp.q = q;
  kp.out = out;
  kp.out_lse = out_lse;
  kp.row_flags = row_flags;
  kp.policy = policy;
  kp.num_splits = S;
  kp.list_flags = unified ? 1 : 0;
  const double log2e = 1.4426950408889634;
  kp.qscale = (float)((double)scale * log2e * (p.kv_fp8 ? (double)p.k_scale : 1.0));
  kp.v_scale = p.kv_fp8 ? p.v_scale : 1.f;
  kp.phi2 = (float)((double)p.unified_max * log2e);
  kp.lo2 = (float)(((double)p.unified_max + p.range_lo) * log2e);
  kp.hi2 = (float)(((double)p.unified_max + p.range_hi) * log2e);
  const int grid = policy == kBalanced
                       ? pl.grid
                       : uniform_grid((long long)pl.n_groups * S, pl.num_sms);

  const bool sync_after = stats != nullptr || p.validate;
  kp.piece_stats = stats != nullptr ? 1 : 0;
  char* ws = static_cast<char*>(workspace);
  cudaError_t e;
  if (sync_after) {
    e = cudaMemsetAsync(ws + pl.off_status, 0, 40, stream);   // status + stats counters
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(status)");
  }

  // The split kernel computes the step; the last piece of each group merges it in-kernel.
  const void* fn = kernel_for(pl, p.mode);
  if (!fn) return DA_ERR_UNSUPPORTED;
  rc = ensure_smem_attr(fn, pl.smem_bytes);
  if (rc != DA_OK) return rc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = pl.smem_bytes;
  cfg.stream = stream;
  void* kargs[3] = {&kp, &tmk, &tmv};
  if (args->split_event_begin) {
    e = cudaEventRecord(static_cast<cudaEvent_t>(args->split_event_begin), stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord(split_event_begin)");
  }
  e = cudaLaunchKernelExC(&cfg, fn, kargs);
  if (e != cudaSuccess) return cuda_fail(e, "launching the split kernel");
  if (args->split_event_end) {
    e = cudaEventRecord(static_cast<cudaEvent_t>(args->split_event_end), stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord(split_event_end)");
  }

  if (unified) {
    // Synchronised recompute of flagged groups ("The Overflow Fallback: Recomputation"),
    // always enqueued, as a programmatic dependent of the split kernel, so that no host round
    // trip is needed; it exits at once when nothing was flagged.
    Params rp = kp;
    rp.policy = kUniform;
    rp.num_splits = pl.recompute_splits;
    rp.recompute = 1;
    rp.piece_stats = 0;
    const void* rfn = kernel_for(pl, DA_SOFTMAX_SYNC);
    rc = ensure_smem_attr(rfn, pl.smem_bytes);
    if (rc != DA_OK) return rc;
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t rcfg = cfg;
    rcfg.gridDim = dim3((unsigned)uniform_grid((long long)pl.n_groups * pl.recompute_splits,
                                                pl.num_sms));
    rcfg.attrs = pdl;
    rcfg.numAttrs = 1;
    void* rargs[3] = {&rp, &tmk, &tmv};   // same consumer kind, same tile layout
    e = cudaLaunchKernelExC(&rcfg, rfn, rargs);
    if (e != cudaSuccess) return cuda_fail(e, "launching the recompute kernel");
  }

  if (sync_after) {
    int32_t st = 0;
    unsigned long long counts[4] = {0, 0, 0, 0};
    e = cudaMemcpyAsync(&st, ws + pl.off_status, 4, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(counts, ws + pl.off_stats, 32, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device status");
    if (stats) {
      stats->grid_ctas = grid;
      stats->num_splits = policy == kBalanced ? 0 : S;
      stats->rows_flagged = (long long)counts[0];
      stats->splits_flagged = (long long)counts[1];
      stats->recompute_launched = unified ? 1 : 0;
      stats->split_tokens = (int)counts[2];
      stats->split_tokens_min = counts[3] ? (int)(0x7fffffffull - counts[3]) : 0;
    }
    const int err = status_to_error(st);
    if (err != DA_OK) return err;
  }
  return DA_OK;
}

int decode_attn_check_status(const da_plan* plan, void* workspace, void* cuda_stream) {
  if (!plan || !workspace) return DA_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  char* ws = static_cast<char*>(workspace);
  int32_t st = 0;
  cudaError_t e = cudaMemcpyAsync(&st, ws + plan->off_status, 4, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws + plan->off_status, 0, 4, stream);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status");
  return status_to_error(st);
}

int decode_attn_debug_gather(const da_plan* plan, const int32_t* block_table,
                             const int32_t* seq_lens, int64_t* offsets_out, void* cuda_stream) {
  if (!plan || !seq_lens || !offsets_out) return DA_ERR_INVALID_ARG;
  if (plan->prob.paged ? !block_table : block_table != nullptr) return DA_ERR_INVALID_ARG;
  Params kp;
  fill_common(*plan, kp, block_table, seq_lens, nullptr);
  kp.debug_offsets = reinterpret_cast<int64_t*>(offsets_out);
  debug_gather_kernel<<<std::max(1, std::min(4096, plan->num_sms * 8)), 256, 0,
                        static_cast<cudaStream_t>(cuda_stream)>>>(kp);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DA_OK : cuda_fail(e, "launching the debug gather kernel");
}

int decode_attn_logit_histogram(const da_plan* plan, const void* q, const void* k_cache,
                                const int32_t* block_table, const int32_t* seq_lens,
                                float scale, float lo, float hi, int nbins,
                                unsigned long long* counts, void* cuda_stream) {
  if (!plan || !q || !k_cache || !seq_lens || !counts) return DA_ERR_INVALID_ARG;
  const da_plan& pl = *plan;
  if (pl.prob.paged ? !block_table : block_table != nullptr) return DA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(seq_lens, 4) ||
      !aligned(counts, 8) || (block_table && !aligned(block_table, 4)))
    return DA_ERR_INVALID_ARG;
  if (nbins < 1 || nbins > DECODE_ATTN_MAX_HIST_BINS) return DA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !std::isfinite(lo) || !std::isfinite(hi) || !(lo < hi))
    return DA_ERR_INVALID_ARG;
  const float inv_w = (float)((double)nbins / ((double)hi - (double)lo));
  if (!std::isfinite(inv_w) || !(inv_w > 0.f)) return DA_ERR_INVALID_ARG;

  // an FP8 cache's codes stand for code * k_scale: fold it into the logit scale
  float xscale = pl.prob.kv_fp8 ? (float)((double)scale * (double)pl.prob.k_scale) : scale;
  const int D = pl.prob.head_dim, G = pl.group;
  if (pl.prob.kv_fp8 || pl.prob.qkv_dtype == DA_BF16) {
    // bf16 and FP8 caches: the tensor-core pass
    const void* fn = pl.prob.kv_fp8 ? histogram_mma_kernel_for<fp8e4m3>(D, G)
                                    : histogram_mma_kernel_for<__nv_bfloat16>(D, G);
    if (!fn) return DA_ERR_UNSUPPORTED;
    const long long items = (long long)pl.prob.batch * pl.prob.num_kv_heads *
                            ((pl.capacity + kHmItemTokens - 1) / kHmItemTokens);
    if (items >= (1ll << 31) - pl.num_sms) return DA_ERR_UNSUPPORTED;   // 32-bit item indices
    const int nlens = pl.prob.batch <= kHmMaxBatchSmem ? pl.prob.batch : 0;
    // As many CTAs per SM as fit, up to 4, each with the deepest ring that then fits: a CTA
    // turns its items around one at a time, so several of them keep more of each SM busy than
    // one deeper ring.
    constexpr size_t kSmSmem = 233472, kBlockReserve = 1024;   // per SM; reserved per CTA
    int stages = 0, per_sm = 1;
    size_t smem = 0;
    for (int target = 4; target >= 1 && stages == 0; --target)
      for (int st = kHmMaxStages; st >= 2 && stages == 0; --st) {
        const size_t bytes = hm_layout(D, G, pl.kv_es, nbins, st, nlens).total;
        if (bytes <= kSmemLimit && (size_t)target * (bytes + kBlockReserve) <= kSmSmem) {
          stages = st;
          smem = bytes;
          per_sm = target;
        }
      }
    if (stages == 0) return DA_ERR_UNSUPPORTED;
    cudaError_t e =
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(histogram smem)");
    int fit = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, fn, kHmThreads, smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    per_sm = std::max(1, std::min(per_sm, fit));
    CUtensorMap tmk;   // the split kernel's tiles of one KV head
    const int rc = make_kv_map(pl, k_cache, true, 1, &tmk);
    if (rc != DA_OK) return rc;
    Params kp;
    fill_common(pl, kp, block_table, seq_lens, nullptr);
    kp.q = q;
    kp.qscale = xscale;
    const int grid = (int)std::max(1ll, std::min(items, (long long)pl.num_sms * per_sm));
    void* args[7] = {&kp, &tmk, &lo, const_cast<float*>(&inv_w), &nbins, &counts, &stages};
    e = cudaLaunchKernel(fn, dim3((unsigned)grid), dim3(kHmThreads), args, smem,
                         static_cast<cudaStream_t>(cuda_stream));
    return e == cudaSuccess ? DA_OK : cuda_fail(e, "launching the logit histogram kernel");
  }

  const void* fn = nullptr;
  if (pl.prob.kv_fp8) fn = histogram_kernel_for<fp8e4m3>(pl.prob.head_dim, pl.group);
  else switch (pl.prob.qkv_dtype) {
    case DA_F32: fn = histogram_kernel_for<float>(pl.prob.head_dim, pl.group); break;
    case DA_F16: fn = histogram_kernel_for<__half>(pl.prob.head_dim, pl.group); break;
    default: fn = histogram_kernel_for<__nv_bfloat16>(pl.prob.head_dim, pl.group); break;
  }
  if (!fn) return DA_ERR_UNSUPPORTED;
  const size_t smem = ((size_t)nbins + 2) * 4;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(histogram smem)");
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kHistThreads, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
  const long long items = (long long)pl.prob.batch * pl.prob.num_kv_heads *
                          ((pl.capacity + kHistItemTokens - 1) / kHistItemTokens);
  const long long blocks = (items + kHistWarps - 1) / kHistWarps;
  const int grid =
      (int)std::max(1ll, std::min(blocks, (long long)pl.num_sms * std::max(1, per_sm)));

  Params kp;
  fill_common(pl, kp, block_table, seq_lens, nullptr);
  kp.q = q;
  void* args[7] = {&kp, &k_cache, &xscale, &lo, const_cast<float*>(&inv_w), &nbins, &counts};
  e = cudaLaunchKernel(fn, dim3((unsigned)grid), dim3(kHistThreads), args, smem,
                       static_cast<cudaStream_t>(cuda_stream));
  return e == cudaSuccess ? DA_OK : cuda_fail(e, "launching the logit histogram kernel");
}

int decode_attn_choose_phi(const unsigned long long* counts, int nbins, float lo, float hi,
                           double coverage, float max_width, float* phi, float* x_lo,
                           float* x_hi) {
  if (!counts || !phi || !x_lo || !x_hi || nbins < 1) return DA_ERR_INVALID_ARG;
  if (!(coverage > 0.0 && coverage <= 1.0) || !(max_width > 0.f)) return DA_ERR_INVALID_ARG;
  if (!std::isfinite(lo) || !std::isfinite(hi) || !(lo < hi)) return DA_ERR_INVALID_ARG;
  double total = 0.0;
  for (int i = 0; i < nbins + 2; ++i) total += (double)counts[i];
  if (total == 0.0) return DA_ERR_INVALID_ARG;
  // At most `tail` values may lie outside the range on each side, so that the range holds
  // at least the fraction `coverage` of them.
  const double tail = std::floor((1.0 - coverage) * total / 2.0);
  const double under = (double)counts[0], over = (double)counts[nbins + 1];
  if (under > tail || over > tail) return DA_ERR_HISTOGRAM_RANGE;
  int first = 0;                 // first kept bin
  double below = under;
  while (first < nbins && below + (double)counts[1 + first] <= tail)
    below += (double)counts[1 + first++];
  int last = nbins - 1;          // last kept bin
  double above = over;
  while (last >= 0 && above + (double)counts[1 + last] <= tail)
    above += (double)counts[1 + last--];
  // first <= last: otherwise every value would be among the <= 2 * tail < total dropped.
  const double w = ((double)hi - (double)lo) / nbins;
  const double e_lo = (double)lo + first * w, e_hi = (double)lo + (last + 1) * w;
  float f_lo = (float)e_lo, f_hi = (float)e_hi;   // rounded outwards to fp32
  if ((double)f_lo > e_lo) f_lo = std::nextafter(f_lo, -INFINITY);
  if ((double)f_hi < e_hi) f_hi = std::nextafter(f_hi, INFINITY);
  *x_lo = f_lo;
  *x_hi = f_hi;
  *phi = f_lo;   // phi = the lower bound of the covered range
  return (double)f_hi - (double)f_lo > (double)max_width ? DA_ERR_RANGE_TOO_WIDE : DA_OK;
}

}  // extern "C"

// ---- decode_attn_run_static: the library's own fixed scratch in place of a workspace ----
// One region per device, part of the library's device code: it is reserved (and zero-filled)
// when that code is loaded on a device, never by a call.
static __device__ __align__(256) unsigned char g_static_scratch[DECODE_ATTN_STATIC_SCRATCH_BYTES];

namespace {

SymbolAddressCache<64> g_static_cache;

// Unique ID of the calling thread's current CUDA context (0 when none is current yet).
int current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 4000, cudaEnableDefault, &q1) ==
            cudaSuccess && q1 == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &q2) ==
            cudaSuccess && q2 == cudaDriverEntryPointSuccess) {
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(a);
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(b);
    }
  });
  if (!get_current || !get_id) {
    g_cuda_error = "cuCtxGetCurrent / cuCtxGetId are not available from the driver";
    return DA_ERR_CUDA;
  }
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) {
    g_cuda_error = "cuCtxGetCurrent failed";
    return DA_ERR_CUDA;
  }
  *id = 0;
  if (ctx && get_id(ctx, id) != CUDA_SUCCESS) {
    g_cuda_error = "cuCtxGetId failed";
    return DA_ERR_CUDA;
  }
  return DA_OK;
}

// Device address of the scratch region in the calling thread's current context. Looked up
// (cudaGetSymbolAddress, which loads the library's device code into the context if needed)
// on the first call in each context and cached under the context's unique ID, so a device
// reset or a caller's own driver context gets its own lookup.
int static_scratch(void** addr) {
  auto resolve = [](void** out) -> int {
    const cudaError_t e = cudaGetSymbolAddress(out, g_static_scratch);
    return e == cudaSuccess ? DA_OK : cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
  };
  unsigned long long id = 0;
  int rc = current_context_id(&id);
  if (rc != DA_OK) return rc;
  if (id == 0) {
    // no context is current yet: the lookup makes the device's primary context current
    rc = resolve(addr);
    if (rc != DA_OK) return rc;
    rc = current_context_id(&id);
    if (rc != DA_OK) return rc;
    if (id == 0) return DA_OK;   // (not cached)
  }
  return g_static_cache.get(id, resolve, addr);
}

// decode_attn_run's host-side argument checks, made before the scratch is cleared so that
// an argument error enqueues nothing.
int static_args_ok(const da_plan& pl, const void* q, const void* k_cache, const void* v_cache,
                   const int32_t* block_table, const int32_t* seq_lens, float scale,
                   int num_splits, const void* out, const float* out_lse) {
  if (!q || !k_cache || !v_cache || !seq_lens || !out) return DA_ERR_INVALID_ARG;
  if (pl.prob.paged ? !block_table : block_table != nullptr) return DA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(seq_lens, 4) || !aligned(out, 16) || (out_lse && !aligned(out_lse, 4)) ||
      (block_table && !aligned(block_table, 4)))
    return DA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || num_splits < -1) return DA_ERR_INVALID_ARG;
  if (num_splits == 0 && pl.batch_smem == 0) return DA_ERR_UNSUPPORTED;
  if (num_splits > pl.max_splits) return DA_ERR_WORKSPACE_TOO_SMALL;
  if (!kernel_for(pl, pl.prob.mode)) return DA_ERR_UNSUPPORTED;
  if (pl.prob.mode == DA_SOFTMAX_UNIFIED && !kernel_for(pl, DA_SOFTMAX_SYNC))
    return DA_ERR_UNSUPPORTED;
  return DA_OK;
}

}  // namespace

extern "C" {

int decode_attn_run_static(const da_plan* plan, const void* q, const void* k_cache,
                           const void* v_cache, const int32_t* block_table,
                           const int32_t* seq_lens, float scale, int num_splits, void* out,
                           float* out_lse, uint8_t* row_flags, void* cuda_stream,
                           da_stats* stats) {
  if (!plan) return DA_ERR_INVALID_ARG;
  if (plan->ws_bytes > (size_t)DECODE_ATTN_STATIC_SCRATCH_BYTES) return DA_ERR_WORKSPACE_TOO_SMALL;
  int rc = static_args_ok(*plan, q, k_cache, v_cache, block_table, seq_lens, scale, num_splits,
                          out, out_lse);
  if (rc != DA_OK) return rc;
  void* scratch = nullptr;
  rc = static_scratch(&scratch);
  if (rc != DA_OK) return rc;
  // The counters the kernels expect at zero: the region may hold another plan's layout.
  rc = decode_attn_workspace_init(plan, scratch, DECODE_ATTN_STATIC_SCRATCH_BYTES, cuda_stream);
  if (rc != DA_OK) return rc;
  return decode_attn_run(plan, q, k_cache, v_cache, block_table, seq_lens, scale, num_splits,
                         out, out_lse, row_flags, scratch, DECODE_ATTN_STATIC_SCRATCH_BYTES,
                         cuda_stream, stats);
}

}  // extern "C"
