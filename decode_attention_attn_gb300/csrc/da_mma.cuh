// da_mma.cuh -- tensor-core consumer for packed GQA groups of G >= 4 query heads over bf16
// caches, in both softmax modes.
//
// Per KV tile the group's work is two dense contractions (the logits of G heads against the
// tile's tokens, and P . V). On CUDA cores they made the split kernel issue-bound on GB300
// (the consumers alone, with no HBM traffic, took about as long as the whole kernel), so for
// these groups they run on the tensor cores with warp-level m16n8k16 bf16 MMAs, in transposed
// form so that the 16 rows of the MMA are never wasted on a small group:
//   S^T = K q^T: A = the warp's 16 K rows (8 of each of two stages) read with ldmatrix from
//   the 128-byte-swizzled TMA tile, B = q^T (k = d, n = heads; unscaled bf16 so the operand is
//   exact, the scale applied to the FP32 logits), 8 MMAs for d = 128;
//   O^T += V^T P^T: A = V^T read with ldmatrix.trans (rows = d), B = P^T, which movmatrix
//   transposes out of the S^T accumulator layout in registers; 8 m-tiles for d = 128.
// O accumulates in the MMA registers across the whole piece. With one constant phi
// (FlashDecoding++ Eq. 3 / Eq. 4) the accumulators are never rescaled. In the synchronised
// mode each warp keeps a running maximum per head (the online-softmax recurrence of
// "FlashAttention: tiling plus online softmax"); when one of them grows the warp rescales its
// accumulators and denominators by 2^(m_old - m_new), which after the first tiles is rare.
// P enters the MMA as a bf16 pair p_hi + p_lo (p_lo = bf16 of the rounding residual), which
// keeps P exact to ~2^-17; the softmax denominators are summed from the FP32 p.
#pragma once

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

// Transpose of an 8x8 matrix of 16-bit values held in the warp's fragment layout.
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

// Two FP32 values -> bf16x2 (round to nearest even); `hi_elem` lands in the upper half.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo_elem, float hi_elem) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi_elem), "f"(lo_elem));
  return r;
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

template <int D, int G>
struct MmaState {
  static constexpr int KS = D / 16;     // k-steps of the logits / m-tiles of the output
  uint32_t qb[KS][2];                   // B fragments of q^T (k = d, n = head); heads >= G zero
  float o[KS][4];                       // O^T: [0] (d, head hp), [1] (d, hp + 1), [2] (d + 8, hp),
                                        // [3] (d + 8, hp + 1) with d = 16 mt + lane / 4
  float den[2];                         // this lane's share of heads hp, hp + 1 denominators
  float m[2];                           // synchronised recurrence: their running maxima
  float mt[2];                          // split-local fallback, before the switch: the lane's
                                        // maximum logit of each head so far
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

// Consume the warp's 8 rows of two consecutive stages (16 tokens = one MMA k-extent of P . V).
// kt / vt: shared-memory addresses of the K and V tiles of stages 0 and 1 (with n[1] == 0 there
// is no second stage: the caller passes stage 0's tiles again and every stage-1 token is
// masked, so no stale shared memory enters the MMA).
template <int D, int G, bool UNIFIED, bool LOCAL>
__device__ __forceinline__ void mma_consume(const Params& p, MmaState<D, G>& st,
                                            const MmaLane<D>& ml, const uint32_t (&kt)[2],
                                            const uint32_t (&vt)[2], const int (&n)[2], int row0,
                                            int lane, uint32_t& fmask) {
  constexpr int KS = MmaState<D, G>::KS;
  const uint32_t kbase = ml.kst ? kt[1] : kt[0], vbase = ml.vst ? vt[1] : vt[0];

  // S^T = K q^T: two accumulator chains (even and odd k-steps) halve the dependent latency
  float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int kk = 0; kk < KS; ++kk) {
    uint32_t a0, a1, a2, a3;
    ldsm_x4(kbase + ml.koff[kk], a0, a1, a2, a3);
    if (kk & 1)
      mma_bf16(sb, a0, a1, a2, a3, st.qb[kk][0], st.qb[kk][1]);
    else
      mma_bf16(sa, a0, a1, a2, a3, st.qb[kk][0], st.qb[kk][1]);
  }

  // The lane's logits: [0], [1] = token lane/4 of stage 0 for heads hp, hp + 1; [2], [3] = the
  // same row of stage 1. A head's 16 logits sit in the 8 lanes that share lane % 4.
  const int hp = 2 * (lane & 3), tr = row0 + (lane >> 2);
  float x[4];
  bool valid[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    x[c] = (sa[c] + sb[c]) * p.qscale;
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
      for (int c = 0; c < 4; ++c) {
        if (valid[c]) {
          out = out || x[c] < p.lo2 || x[c] > p.hi2;
          st.mt[c & 1] = fmaxf(st.mt[c & 1], x[c]);
        }
      }
      if (__any_sync(0xffffffffu, out)) {
        float m0 = st.mt[0], m1 = st.mt[1];
#pragma unroll
        for (int o = 4; o <= 16; o <<= 1) {
          m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
          m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
        }
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
  }
  float pr[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    pr[c] = valid[c] ? fast_exp2(x[c] - ((c & 1) ? ref1 : ref0)) : 0.f;
    if (UNIFIED && valid[c] && (x[c] < p.lo2 || x[c] > p.hi2)) fmask |= 1u << (hp + (c & 1));
  }
  st.den[0] += pr[0] + pr[2];
  st.den[1] += pr[1] + pr[3];

  // P as bf16 hi + lo (lower half = head hp), transposed into B fragments of P^T:
  // b0 = stage-0 tokens 2 (lane % 4), +1 of head lane / 4, b1 = the same of stage 1
  const uint32_t h0 = bf16x2_rn(pr[0], pr[1]), h1 = bf16x2_rn(pr[2], pr[3]);
  const uint32_t l0 = bf16x2_rn(pr[0] - __uint_as_float(h0 << 16),
                                pr[1] - __uint_as_float(h0 & 0xffff0000u));
  const uint32_t l1 = bf16x2_rn(pr[2] - __uint_as_float(h1 << 16),
                                pr[3] - __uint_as_float(h1 & 0xffff0000u));
  const uint32_t bh0 = movm_t(h0), bh1 = movm_t(h1), bl0 = movm_t(l0), bl1 = movm_t(l1);

  // V rows of masked tokens are zeroed in the fragments (0 * NaN would poison the MMA); only
  // a warp whose rows run past a stage's end needs it
  uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
  if (!(row0 + kTokensPerWarp <= n[0] && row0 + kTokensPerWarp <= n[1])) {
    const int tk = row0 + 2 * (lane & 3);
    vm0 = (tk < n[0] ? 0x0000ffffu : 0u) | (tk + 1 < n[0] ? 0xffff0000u : 0u);
    vm1 = (tk < n[1] ? 0x0000ffffu : 0u) | (tk + 1 < n[1] ? 0xffff0000u : 0u);
  }

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

}  // namespace da
