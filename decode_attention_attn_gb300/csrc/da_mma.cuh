// da_mma.cuh -- tensor-core consumer for groups of 1 to 8 query heads over bf16 or FP8
// (E4M3) caches, in every softmax mode (FP8 tiles: f16 MMAs, see the end of the file).
//
// Per KV tile the group's work is two contractions (the logits of G heads against the tile's
// tokens, and P . V). On CUDA cores they made the split kernel issue-bound on GB300 (the
// consumers alone, with no HBM traffic, took about as long as the whole kernel), so they run
// on the tensor cores with warp-level m16n8k16 bf16 MMAs, in transposed form so that the 16
// rows of the MMA are never wasted on a small group:
//   S^T = K q^T: A = the warp's 16 K rows (8 of each of two stages) read with ldmatrix from
//   the 128-byte-swizzled TMA tile, B = q^T (k = d, n = heads; unscaled bf16 so the operand is
//   exact, the scale applied to the FP32 logits), 8 MMAs for d = 128;
//   O^T += V^T P^T: A = V^T read with ldmatrix.trans (rows = d), B = P^T, which movmatrix
//   transposes out of the S^T accumulator layout in registers; 8 m-tiles for d = 128.
// The MMA's n = 8 head columns beyond the group are zero in q and masked in the softmax, so a
// group of 1 or 2 heads costs the same instructions per KV byte as a group of 8.
// O accumulates in the MMA registers across the whole piece. With one constant phi
// (FlashDecoding++ Eq. 3 / Eq. 4) the accumulators are never rescaled. In the synchronised
// mode each warp keeps a running maximum per head (the online-softmax recurrence of
// "FlashAttention: tiling plus online softmax"); when one of them grows the warp rescales its
// accumulators and denominators by 2^(m_old - m_new), which after the first tiles is rare.
// P enters the MMA as a bf16 pair p_hi + p_lo (p_lo = bf16 of the rounding residual), which
// keeps P exact to ~2^-17; the softmax denominators are summed from the FP32 p.
#pragma once

#include <type_traits>

#include "da_device.cuh"

namespace da {

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A (16x16) * B (16x8), bf16 inputs, FP32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D += A (16x16) * B (16x8), f16 inputs, FP32 accumulators.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 matrix of 16-bit values held in the warp's fragment layout.
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

// Two FP32 values -> f16x2 (round to nearest even); `hi_elem` lands in the upper half.
__device__ __forceinline__ uint32_t f16x2_rn(float lo_elem, float hi_elem) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi_elem), "f"(lo_elem));
  return r;
}
__device__ __forceinline__ float f16_lo(uint32_t h) {
  return __half2float(__ushort_as_half((unsigned short)(h & 0xffffu)));
}
__device__ __forceinline__ float f16_hi(uint32_t h) {
  return __half2float(__ushort_as_half((unsigned short)(h >> 16)));
}

// Two FP32 values -> bf16x2 (round to nearest even); `hi_elem` lands in the upper half.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo_elem, float hi_elem) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi_elem), "f"(lo_elem));
  return r;
}

// ---- FP8 (E4M3) tiles ----------------------------------------------------------------------
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// Bytes of {b, a} picked by the selector's nibbles (byte i of the result = byte s_i).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Byte offset of 16-byte chunk c of row r in an FP8 tile of rows of D bytes (row t * HP + h
// holds KV head h of token t), as the TMA box writes it: with the 128-byte swizzle for
// D = 128 (chunk c of row r at chunk c ^ (r mod 8)), unswizzled for D = 64.
template <int D>
__device__ __forceinline__ uint32_t fp8_off(int r, int c) {
  if constexpr (D == 128)
    return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
  else
    return (uint32_t)(r * D + c * 16);
}

// Byte offset of element e (a multiple of 8) of row t in a tile written by a TMA box of
// 64-element (128-byte) rows with the 128-byte swizzle: 128-byte row r = t * (D / 64) + e / 64
// stores its 16-byte chunk c at chunk c ^ (r mod 8). Tile bases are 1024-aligned.
template <int D>
__device__ __forceinline__ uint32_t swz_off(int t, int e) {
  const int r = t * (D / 64) + e / 64;
  const int c = (e >> 3) & 7;
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

// Per-lane constants of the warp's ldmatrix reads: lane l addresses row l % 8 of matrix l / 8.
template <int D>
struct MmaLane {
  static constexpr int KS = D / 16;
  uint32_t koff[KS];   // K tile, k-step kk: matrices (stage 0, d+0), (stage 1, d+0), (0, +8), (1, +8)
  uint32_t voff[KS];   // V tile, m-tile mt: matrices (stage 0, d+0), (stage 0, +8), (1, +0), (1, +8)
  int kst, vst;        // stage whose tile this lane's K / V row address lies in
  __device__ __forceinline__ MmaLane(int row0, int lane) {
    const int lmat = lane >> 3, t = row0 + (lane & 7);
#pragma unroll
    for (int i = 0; i < KS; ++i) {
      koff[i] = swz_off<D>(t, i * 16 + (lmat >> 1) * 8);
      voff[i] = swz_off<D>(t, i * 16 + (lmat & 1) * 8);
    }
    kst = lmat & 1;
    vst = lmat >> 1;
  }
};

// FP8 tiles need no ldmatrix addresses.
struct NoMmaLane {
  __device__ __forceinline__ NoMmaLane(int, int) {}
};

template <int D, int G>
struct MmaState {
  static constexpr int KS = D / 16;     // k-steps of the logits / m-tiles of the output
  uint32_t qb[KS][2];                   // B fragments of q^T (k = d, n = head); heads >= G zero
  float o[KS][4];                       // O^T: [0] (d, head hp), [1] (d, hp + 1), [2] (d', hp),
                                        // [3] (d', hp + 1) with d = 16 mt + lane / 4, d' = d + 8
                                        // (FP8 tiles: d = (D/8)(lane / 4) + 2 mt, d' = d + 1)
  float den[2];                         // this lane's share of heads hp, hp + 1 denominators
  float m[2];                           // synchronised recurrence: their running maxima
                                        // (FP8 tiles, unified phase: the reference r)
  float qmul;                           // logit factor: scale * log2 e (FP8 tiles: times 2^-s,
                                        // s the power of two q was scaled by)
  bool sw;                              // split-local fallback: the warp has switched to the
                                        // synchronised recurrence
};

// Load the group's q^T fragments from the stage's q area (G x D bf16, row-major, unscaled).
template <int D, int G>
__device__ __forceinline__ void mma_load_q(MmaState<D, G>& st, const uint8_t* qsm, int lane) {
  const int head = lane >> 2, kq = 2 * (lane & 3);
  const bool hv = head < G;
#pragma unroll
  for (int k = 0; k < MmaState<D, G>::KS; ++k) {
    const __nv_bfloat16* qr = reinterpret_cast<const __nv_bfloat16*>(qsm) + head * D + k * 16 + kq;
    st.qb[k][0] = hv ? *reinterpret_cast<const uint32_t*>(qr) : 0u;
    st.qb[k][1] = hv ? *reinterpret_cast<const uint32_t*>(qr + 8) : 0u;
  }
}

// One stage pair's softmax step, shared by the bf16 and FP8 consumers: the logits from the
// two S^T accumulator chains sa, sb (token lane/4 of stage 0 in [0], [1], of stage 1 in
// [2], [3]; heads hp, hp + 1), the range check, the running maxima of the synchronised
// recurrence, p, the denominators, and P^T as hi / lo B fragments (bh*, bl*): bf16, or f16
// when F16. f16 holds only p <= 2^15 and keeps 11 bits only above 2^-14, so in the unified
// phase the F16 step takes p = 2^(x - r) against a reference r = phi + 16 k per head and warp,
// with k the smallest integer that puts the largest logit so far in (r - 1, r + 15]. k starts
// from the first logits and only grows, in steps that rescale the state by 2^-16 each, so p
// stays exactly the unified 2^(x - phi) up to one power of two per warp and head, and no stage
// pair is rescaled on its own. The state is then relative to r (kept in st.m), not to phi.
template <int D, int G, bool UNIFIED, bool LOCAL, bool F16>
__device__ __forceinline__ void mma_softmax(const Params& p, MmaState<D, G>& st,
                                            const float (&sa)[4], const float (&sb)[4],
                                            const int (&n)[2], int row0, int lane,
                                            uint32_t& fmask, uint32_t& bh0, uint32_t& bh1,
                                            uint32_t& bl0, uint32_t& bl1) {
  constexpr int KS = MmaState<D, G>::KS;
  // The lane's logits: [0], [1] = token lane/4 of stage 0 for heads hp, hp + 1; [2], [3] = the
  // same row of stage 1. A head's 16 logits sit in the 8 lanes that share lane % 4.
  const int hp = 2 * (lane & 3), tr = row0 + (lane >> 2);
  float x[4];
  bool valid[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    x[c] = (sa[c] + sb[c]) * st.qmul;
    valid[c] = hp + (c & 1) < G && tr < n[c >> 1];
  }
  float ref0 = p.phi2, ref1 = p.phi2;
  if constexpr (LOCAL) {
    // Split-local fallback: while every logit so far was in range, the state is an exact
    // online-softmax state with m = phi. On the first tile with a logit out of range the warp
    // rescales it to the true maximum so far and continues with the synchronised recurrence,
    // so the split needs no second read of its KV.
    if (!st.sw) {
      bool out = false;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (valid[c]) out = out || x[c] < p.lo2 || x[c] > p.hi2;
      if constexpr (F16) {
        // f16 P: the state is already relative to the warp's reference r = st.m, which lies
        // within 15 below the largest logit so far at most; the synchronised recurrence
        // continues from it
        if (__any_sync(0xffffffffu, out)) st.sw = true;
      } else if (__any_sync(0xffffffffu, out)) {
        // The new reference must bound every logit so far from above. With bf16 P a bound
        // within log2(tokens) of the maximum is as good as the maximum, and the state gives
        // one for free: its denominators are sums of 2^(x - phi) over in-range logits, so
        // phi + log2(sum) lies between the maximum and the maximum plus log2 of the warp's
        // token count.
        float m0 = st.den[0], m1 = st.den[1];
#pragma unroll
        for (int o = 4; o <= 16; o <<= 1) {
          m0 += __shfl_xor_sync(0xffffffffu, m0, o);
          m1 += __shfl_xor_sync(0xffffffffu, m1, o);
        }
        m0 = m0 > 0.f ? p.phi2 + fast_log2(m0) : -INFINITY;
        m1 = m1 > 0.f ? p.phi2 + fast_log2(m1) : -INFINITY;
        const float al0 = m0 > -INFINITY ? fast_exp2(p.phi2 - m0) : 1.f;
        const float al1 = m1 > -INFINITY ? fast_exp2(p.phi2 - m1) : 1.f;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          st.o[mt][0] *= al0;
          st.o[mt][1] *= al1;
          st.o[mt][2] *= al0;
          st.o[mt][3] *= al1;
        }
        st.den[0] *= al0;
        st.den[1] *= al1;
        st.m[0] = m0;
        st.m[1] = m1;
        st.sw = true;
      }
    }
  }
  if (!UNIFIED || (LOCAL && st.sw)) {
    float m0 = fmaxf(valid[0] ? x[0] : -INFINITY, valid[2] ? x[2] : -INFINITY);
    float m1 = fmaxf(valid[1] ? x[1] : -INFINITY, valid[3] ? x[3] : -INFINITY);
#pragma unroll
    for (int o = 4; o <= 16; o <<= 1) {
      m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
      m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
    }
    const float n0 = fmaxf(st.m[0], m0), n1 = fmaxf(st.m[1], m1);
    if (__any_sync(0xffffffffu, n0 > st.m[0] || n1 > st.m[1])) {
      const float al0 = n0 > st.m[0] ? fast_exp2(st.m[0] - n0) : 1.f;   // 0 from -inf
      const float al1 = n1 > st.m[1] ? fast_exp2(st.m[1] - n1) : 1.f;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        st.o[mt][0] *= al0;
        st.o[mt][1] *= al1;
        st.o[mt][2] *= al0;
        st.o[mt][3] *= al1;
      }
      st.den[0] *= al0;
      st.den[1] *= al1;
      st.m[0] = n0;
      st.m[1] = n1;
    }
    ref0 = st.m[0];   // -inf only while all of the head's tokens so far are masked
    ref1 = st.m[1];
  } else if constexpr (F16) {
    // unified phase, f16 P: the reference r = phi + 16 k (see above), raised when this stage
    // pair's largest logit passes r + 15
    float m0 = fmaxf(valid[0] ? x[0] : -INFINITY, valid[2] ? x[2] : -INFINITY);
    float m1 = fmaxf(valid[1] ? x[1] : -INFINITY, valid[3] ? x[3] : -INFINITY);
#pragma unroll
    for (int o = 4; o <= 16; o <<= 1) {
      m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
      m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
    }
    const bool up0 = m0 > -INFINITY && !(m0 <= st.m[0] + 15.f);   // also when r is still -inf
    const bool up1 = m1 > -INFINITY && !(m1 <= st.m[1] + 15.f);
    if (__any_sync(0xffffffffu, up0 || up1)) {
      const float r0 = up0 ? p.phi2 + 16.f * ceilf((m0 - p.phi2 - 15.f) * 0.0625f) : st.m[0];
      const float r1 = up1 ? p.phi2 + 16.f * ceilf((m1 - p.phi2 - 15.f) * 0.0625f) : st.m[1];
      const float al0 = up0 && st.m[0] > -INFINITY ? fast_exp2(st.m[0] - r0) : 1.f;
      const float al1 = up1 && st.m[1] > -INFINITY ? fast_exp2(st.m[1] - r1) : 1.f;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        st.o[mt][0] *= al0;
        st.o[mt][1] *= al1;
        st.o[mt][2] *= al0;
        st.o[mt][3] *= al1;
      }
      st.den[0] *= al0;
      st.den[1] *= al1;
      st.m[0] = r0;
      st.m[1] = r1;
    }
    ref0 = st.m[0];   // -inf only while all of the head's tokens so far are masked
    ref1 = st.m[1];
  }
  float pr[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    pr[c] = valid[c] ? fast_exp2(x[c] - ((c & 1) ? ref1 : ref0)) : 0.f;
    if (UNIFIED && valid[c] && (x[c] < p.lo2 || x[c] > p.hi2)) fmask |= 1u << (hp + (c & 1));
  }
  st.den[0] += pr[0] + pr[2];
  st.den[1] += pr[1] + pr[3];

  // P as hi + lo (lower half = head hp), transposed into B fragments of P^T:
  // b0 = stage-0 tokens 2 (lane % 4), +1 of head lane / 4, b1 = the same of stage 1
  uint32_t h0, h1, l0, l1;
  if constexpr (F16) {
    h0 = f16x2_rn(pr[0], pr[1]);
    h1 = f16x2_rn(pr[2], pr[3]);
    l0 = f16x2_rn(pr[0] - f16_lo(h0), pr[1] - f16_hi(h0));
    l1 = f16x2_rn(pr[2] - f16_lo(h1), pr[3] - f16_hi(h1));
  } else {
    h0 = bf16x2_rn(pr[0], pr[1]);
    h1 = bf16x2_rn(pr[2], pr[3]);
    l0 = bf16x2_rn(pr[0] - __uint_as_float(h0 << 16), pr[1] - __uint_as_float(h0 & 0xffff0000u));
    l1 = bf16x2_rn(pr[2] - __uint_as_float(h1 << 16), pr[3] - __uint_as_float(h1 & 0xffff0000u));
  }
  bh0 = movm_t(h0);
  bh1 = movm_t(h1);
  bl0 = movm_t(l0);
  bl1 = movm_t(l1);

}

// Masks that zero the V fragments' halves of tokens past a stage's end (0 * NaN would poison
// the MMA): vm0 for stage 0, vm1 for stage 1; all ones for a warp whose rows are all valid.
__device__ __forceinline__ void v_masks(const int (&n)[2], int row0, int lane, uint32_t& vm0,
                                        uint32_t& vm1) {
  vm0 = 0xffffffffu;
  vm1 = 0xffffffffu;
  if (!(row0 + kTokensPerWarp <= n[0] && row0 + kTokensPerWarp <= n[1])) {
    const int tk = row0 + 2 * (lane & 3);
    vm0 = (tk < n[0] ? 0x0000ffffu : 0u) | (tk + 1 < n[0] ? 0xffff0000u : 0u);
    vm1 = (tk < n[1] ? 0x0000ffffu : 0u) | (tk + 1 < n[1] ? 0xffff0000u : 0u);
  }
}

// Consume the warp's 8 rows of two consecutive stages (16 tokens = one MMA k-extent of P . V).
// kt / vt: shared-memory addresses of the K and V tiles of stages 0 and 1 (with n[1] == 0 there
// is no second stage: the caller passes stage 0's tiles again and every stage-1 token is
// masked, so no stale shared memory enters the MMA).
// S^T = K q^T over the warp's 8 rows of two stages of bf16 tiles (kt as in mma_consume), as
// two accumulator chains (even and odd k-steps, which halves the dependent latency): the
// logits are sa + sb in the C-fragment layout (token lane/4 of stage 0 in [0], [1], of stage
// 1 in [2], [3]; heads 2 (lane % 4) and that + 1).
template <int D, int G>
__device__ __forceinline__ void mma_logits(const MmaState<D, G>& st, const MmaLane<D>& ml,
                                           const uint32_t (&kt)[2], float (&sa)[4],
                                           float (&sb)[4]) {
  constexpr int KS = MmaState<D, G>::KS;
  const uint32_t kbase = ml.kst ? kt[1] : kt[0];
#pragma unroll
  for (int i = 0; i < 4; ++i) sa[i] = sb[i] = 0.f;
#pragma unroll
  for (int kk = 0; kk < KS; ++kk) {
    uint32_t a0, a1, a2, a3;
    ldsm_x4(kbase + ml.koff[kk], a0, a1, a2, a3);
    if (kk & 1)
      mma_bf16(sb, a0, a1, a2, a3, st.qb[kk][0], st.qb[kk][1]);
    else
      mma_bf16(sa, a0, a1, a2, a3, st.qb[kk][0], st.qb[kk][1]);
  }
}

template <int D, int G, bool UNIFIED, bool LOCAL>
__device__ __forceinline__ void mma_consume(const Params& p, MmaState<D, G>& st,
                                            const MmaLane<D>& ml, const uint32_t (&kt)[2],
                                            const uint32_t (&vt)[2], const int (&n)[2], int row0,
                                            int lane, uint32_t& fmask) {
  constexpr int KS = MmaState<D, G>::KS;
  const uint32_t vbase = ml.vst ? vt[1] : vt[0];

  float sa[4], sb[4];
  mma_logits<D, G>(st, ml, kt, sa, sb);
  uint32_t bh0, bh1, bl0, bl1, vm0, vm1;
  mma_softmax<D, G, UNIFIED, LOCAL, false>(p, st, sa, sb, n, row0, lane, fmask, bh0, bh1, bl0,
                                           bl1);
  v_masks(n, row0, lane, vm0, vm1);

  // O^T += V^T P^T: per m-tile of 16 d, A fragments (d 0-7 | 8-15) x (stage-0 | stage-1 tokens)
#pragma unroll
  for (int mt = 0; mt < KS; ++mt) {
    uint32_t a0, a1, a2, a3;
    ldsm_x4_t(vbase + ml.voff[mt], a0, a1, a2, a3);
    a0 &= vm0;
    a1 &= vm0;
    a2 &= vm1;
    a3 &= vm1;
    mma_bf16(st.o[mt], a0, a1, a2, a3, bh0, bh1);
    mma_bf16(st.o[mt], a0, a1, a2, a3, bl0, bl1);
  }
}

// ---- FP8 caches ------------------------------------------------------------------------
// The same two contractions over E4M3 tiles, on f16 MMAs: every E4M3 code is a binary16
// number, converted exactly by one cvt per pair of codes. ldmatrix cannot transpose byte
// tiles, so each lane reads its operand bytes with plain shared-memory loads, and both
// contractions use an order of their index sets that makes a lane's bytes contiguous:
//   S^T = K q^T sums over d, in any order as long as K and q^T agree: k-step kk takes, in the
//   fragment slots of lane (g, c) = (lane / 4, lane % 4), d = c * D/4 + 4 kk + {0, 1} (slots
//   2c, 2c + 1) and + {2, 3} (slots 2c + 8, 2c + 9). The lane's K bytes for all k-steps are
//   then D/4 consecutive bytes of its row, and q^T is loaded in the same order. q (bf16) is
//   scaled by a power of two 2^s into f16's range, exactly for every element above 2^-29
//   of the group's largest (f16 has 11 significant bits to bf16's 8), and the logits are
//   scaled back by 2^-s.
//   O^T += V^T P^T keeps the token order (P^T's B fragment comes out of the S^T layout) and
//   permutes the output rows instead: row r of m-tile mt is d = (D/8) * (r mod 8) + 2 mt +
//   r / 8, so lane (g, c) holds d = (D/8) g + 2 mt + {0, 1} of tokens 2c, 2c + 1 of each
//   stage, D/8 consecutive bytes of each of four rows for all m-tiles; prmt pairs the two
//   tokens' bytes of one d. publish_mma undoes the row order. P enters as f16 hi + lo (see
//   mma_softmax for its range).

// q^T fragments in the FP8 order (see above) from the stage's q area (G x D bf16), as f16
// scaled by 2^s with s such that the group's largest |q| lands in [2^14, 2^15); st.qmul
// becomes qscale * 2^-s.
template <int D, int G>
__device__ __forceinline__ void mma_load_q_fp8(const Params& p, MmaState<D, G>& st,
                                               const uint8_t* qsm, int lane) {
  constexpr int KS = MmaState<D, G>::KS;
  const int head = lane >> 2, c = lane & 3;
  const bool hv = head < G;
  uint32_t raw[KS][2];
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < KS; ++k) {
    const __nv_bfloat16* qr =
        reinterpret_cast<const __nv_bfloat16*>(qsm) + head * D + c * (D / 4) + 4 * k;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      raw[k][i] = hv ? *reinterpret_cast<const uint32_t*>(qr + 2 * i) : 0u;
      amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(raw[k][i] << 16)),
                               fabsf(__uint_as_float(raw[k][i] & 0xffff0000u))));
    }
  }
#pragma unroll
  for (int o = 1; o <= 16; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  // amax = 0.f1 * 2^e with e = biased exponent - 126; s = 15 - e, kept where 2^s and 2^-s
  // are normal floats
  const int e = (int)((__float_as_uint(amax) >> 23) & 0xffu) - 126;
  const int sh = amax > 0.f ? min(126, max(-126, 15 - e)) : 0;
  const float up = __uint_as_float((uint32_t)(127 + sh) << 23);
  const float down = __uint_as_float((uint32_t)(127 - sh) << 23);
#pragma unroll
  for (int k = 0; k < KS; ++k)
#pragma unroll
    for (int i = 0; i < 2; ++i)
      st.qb[k][i] = f16x2_rn(__uint_as_float(raw[k][i] << 16) * up,
                             __uint_as_float(raw[k][i] & 0xffff0000u) * up);
  st.qmul = p.qscale * down;
}

// S^T = K q^T over FP8 tiles (kt, row0 as in mma_consume; HP KV heads per token row, as in
// mma_consume_fp8 below), into two accumulator chains shared by the KV heads: the logits are
// sa + sb, laid out as mma_logits leaves them.
template <int D, int G, int HP>
__device__ __forceinline__ void mma_logits_fp8(const MmaState<D, G>& st, const uint32_t (&kt)[2],
                                               int row0, int lane, float (&sa)[4],
                                               float (&sb)[4]) {
  static_assert(G % HP == 0, "every KV head has the same number of query heads");
  constexpr int KS = MmaState<D, G>::KS;
  constexpr int KW = D / 16;   // 4-byte words of a lane's K bytes (one per k-step)
  const int g = lane >> 2, c = lane & 3;
  const int bh = g / (G / HP);   // KV head of this lane's B column (query head g)
  // A rows 0-7 = token row0 + g of stage 0, rows 8-15 = the same of stage 1
#pragma unroll
  for (int i = 0; i < 4; ++i) sa[i] = sb[i] = 0.f;
#pragma unroll
  for (int h = 0; h < HP; ++h) {
    uint32_t k0[KW], k1[KW];
    const int r = (row0 + g) * HP + h;
#pragma unroll
    for (int x = 0; x < D / 64; ++x) {   // 16-byte chunks c * D/64 + x of the row
      const uint4 w0 = lds128(kt[0] + fp8_off<D>(r, c * (D / 64) + x));
      const uint4 w1 = lds128(kt[1] + fp8_off<D>(r, c * (D / 64) + x));
      k0[4 * x] = w0.x; k0[4 * x + 1] = w0.y; k0[4 * x + 2] = w0.z; k0[4 * x + 3] = w0.w;
      k1[4 * x] = w1.x; k1[4 * x + 1] = w1.y; k1[4 * x + 2] = w1.z; k1[4 * x + 3] = w1.w;
    }
    const bool on = HP == 1 || bh == h;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      uint32_t a0, a1, a2, a3;
      e4m3x4_to_f16x2(k0[kk], a0, a2);
      e4m3x4_to_f16x2(k1[kk], a1, a3);
      mma_f16((kk & 1) ? sb : sa, a0, a1, a2, a3, on ? st.qb[kk][0] : 0u,
              on ? st.qb[kk][1] : 0u);
    }
  }
}

// mma_consume over FP8 tiles (kt / vt, n, row0 as there). HP > 1: the tiles hold HP KV heads'
// rows of every token (row t * HP + h) and the group's G columns are HP blocks of G / HP query
// heads, one block per KV head. Each contraction then runs once per KV head with the other
// heads' columns of its B operand zeroed, so that all of them add into the same accumulators:
// S^T = sum_h K_h [q^T, head h's columns], O^T += sum_h V_h^T [P^T, head h's columns]. The
// MMA's 8 columns are then all in use, where an unpacked group of 4 heads leaves half of them
// (and of the softmax work) idle.
template <int D, int G, int HP, bool UNIFIED, bool LOCAL>
__device__ __forceinline__ void mma_consume_fp8(const Params& p, MmaState<D, G>& st,
                                                const uint32_t (&kt)[2], const uint32_t (&vt)[2],
                                                const int (&n)[2], int row0, int lane,
                                                uint32_t& fmask) {
  constexpr int KS = MmaState<D, G>::KS;
  const int g = lane >> 2, c = lane & 3;
  const int bh = g / (G / HP);   // KV head of this lane's B column (query head g)
  float sa[4], sb[4];
  mma_logits_fp8<D, G, HP>(st, kt, row0, lane, sa, sb);
  uint32_t bh0, bh1, bl0, bl1, vm0, vm1;
  mma_softmax<D, G, UNIFIED, LOCAL, true>(p, st, sa, sb, n, row0, lane, fmask, bh0, bh1, bl0,
                                          bl1);
  v_masks(n, row0, lane, vm0, vm1);
  const bool tail = (vm0 & vm1) != 0xffffffffu;

  // O^T += V^T P^T: the lane's D/8 bytes (d = (D/8) g + 0 .. D/8 - 1) of tokens row0 + 2c and
  // row0 + 2c + 1 of both stages, for every KV head; word w of a row covers m-tiles 2w and
  // 2w + 1
  constexpr int VW = D / 32;   // 4-byte words per row and lane
  uint32_t va[HP][VW], vb[HP][VW], vc[HP][VW], vd[HP][VW];
#pragma unroll
  for (int h = 0; h < HP; ++h) {
    const int t = row0 + 2 * c;
    const int r0 = t * HP + h, r1 = (t + 1) * HP + h;
    if constexpr (D == 128) {
      const uint4 x = lds128(vt[0] + fp8_off<D>(r0, g)), y = lds128(vt[0] + fp8_off<D>(r1, g));
      const uint4 z = lds128(vt[1] + fp8_off<D>(r0, g)), u = lds128(vt[1] + fp8_off<D>(r1, g));
      va[h][0] = x.x; va[h][1] = x.y; va[h][2] = x.z; va[h][3] = x.w;
      vb[h][0] = y.x; vb[h][1] = y.y; vb[h][2] = y.z; vb[h][3] = y.w;
      vc[h][0] = z.x; vc[h][1] = z.y; vc[h][2] = z.z; vc[h][3] = z.w;
      vd[h][0] = u.x; vd[h][1] = u.y; vd[h][2] = u.z; vd[h][3] = u.w;
    } else {
      const uint32_t o = (uint32_t)(8 * g);
      const uint2 x = lds64(vt[0] + r0 * D + o), y = lds64(vt[0] + r1 * D + o);
      const uint2 z = lds64(vt[1] + r0 * D + o), u = lds64(vt[1] + r1 * D + o);
      va[h][0] = x.x; va[h][1] = x.y;
      vb[h][0] = y.x; vb[h][1] = y.y;
      vc[h][0] = z.x; vc[h][1] = z.y;
      vd[h][0] = u.x; vd[h][1] = u.y;
    }
  }
#pragma unroll
  for (int mt = 0; mt < KS; ++mt) {
    // bytes [token 2c, token 2c + 1] of d (the lower half) and of d + 1 (the upper half)
    const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
#pragma unroll
    for (int h = 0; h < HP; ++h) {
      const uint32_t x0 = prmt(va[h][mt >> 1], vb[h][mt >> 1], sel);
      const uint32_t x1 = prmt(vc[h][mt >> 1], vd[h][mt >> 1], sel);
      uint32_t a0, a1, a2, a3;
      e4m3x4_to_f16x2(x0, a0, a1);
      e4m3x4_to_f16x2(x1, a2, a3);
      if (tail) {
        a0 &= vm0;
        a1 &= vm0;
        a2 &= vm1;
        a3 &= vm1;
      }
      const uint32_t pm = HP == 1 || bh == h ? 0xffffffffu : 0u;   // this head's columns
      mma_f16(st.o[mt], a0, a1, a2, a3, bh0 & pm, bh1 & pm);
      mma_f16(st.o[mt], a0, a1, a2, a3, bl0 & pm, bl1 & pm);
    }
  }
}

}  // namespace da
