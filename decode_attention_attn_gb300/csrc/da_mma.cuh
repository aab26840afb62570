// da_mma.cuh -- tensor-core consumer for packed GQA groups of G >= 4 query heads over bf16
// caches, in both softmax modes.
//
// Per KV tile the group's work is two dense contractions ([G x d] . [d x T] for the logits,
// [G x T] . [T x d] for P . V). On CUDA cores they made the split kernel ALU-bound on GB300
// (the consumers alone, with no HBM traffic, took as long as the whole kernel), so for these
// groups they run on the tensor cores with warp-level m16n8k16 bf16 MMAs:
//   S^T-free form S = Q K^T: A = the group's q (rows = heads, padded to 16, unscaled bf16 so
//   the operand is exact; the scale is applied to the FP32 logits), B = K rows read from the
//   128-byte-swizzled TMA tile with ldmatrix;
//   O += P V: A = P taken straight from the S accumulators (rows = heads, k = tokens), B = V
//   rows read transposed with ldmatrix.trans.
// O accumulates in the MMA registers across the whole piece. With one constant phi
// (FlashDecoding++ Eq. 3 / Eq. 4) the accumulators are never rescaled. In the synchronised
// mode each warp keeps a running maximum per head (the online-softmax recurrence of
// "FlashAttention: tiling plus online softmax"); when one of them grows the warp rescales its
// accumulators and denominators by 2^(m_old - m_new), which after the first tiles is rare.
// P enters the MMA as a bf16 pair p_hi + p_lo (p_lo = bf16 of the rounding residual), which
// keeps P exact to ~2^-17; the softmax denominators are summed from the FP32 p.
//
// Each consumer warp takes 8 rows of two consecutive stages (16 tokens = one MMA k-extent).
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

// D += A (16x16, rows 8..15 zero) * B (16x8), bf16 inputs, FP32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0,
                                         uint32_t b1) {
  const uint32_t z = 0u;
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(z), "r"(a2), "r"(z), "r"(b0), "r"(b1));
}

// Two FP32 values -> bf16x2 (round to nearest even); `hi_elem` lands in the upper half.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo_elem, float hi_elem) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi_elem), "f"(lo_elem));
  return r;
}

// Shared-memory address of element e (a multiple of 8) of row t in a tile written by a TMA box
// of 64-element (128-byte) rows with the 128-byte swizzle: 128-byte row r = t * (D / 64) +
// e / 64 stores its 16-byte chunk c at chunk c ^ (r mod 8). The tile base is 1024-aligned.
template <int D>
__device__ __forceinline__ uint32_t swz(uint32_t base, int t, int e) {
  const int r = t * (D / 64) + e / 64;
  const int c = (e >> 3) & 7;
  return base + (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

template <int D, int G>
struct MmaState {
  static constexpr int KS = D / 16;     // MMA k-steps of the logits
  static constexpr int NT = D / 8;      // 8-wide n-tiles of the output
  uint32_t qa[KS][2];                   // A fragments of q (a0, a2); rows 8..15 are zero
  float o[NT][4];                       // O accumulators (rows = heads; rows >= G unused)
  float den;                            // this lane's share of its head's denominator
  float m;                              // synchronised mode: its head's running maximum
};

// Load the group's q fragments from the stage's q area (G x D bf16, row-major, unscaled).
template <int D, int G>
__device__ __forceinline__ void mma_load_q(MmaState<D, G>& st, const uint8_t* qsm, int lane) {
  const int head = lane >> 2, kq = 2 * (lane & 3);
  const bool hv = head < G;
#pragma unroll
  for (int k = 0; k < MmaState<D, G>::KS; ++k) {
    const __nv_bfloat16* qr = reinterpret_cast<const __nv_bfloat16*>(qsm) + head * D + k * 16 + kq;
    st.qa[k][0] = hv ? *reinterpret_cast<const uint32_t*>(qr) : 0u;
    st.qa[k][1] = hv ? *reinterpret_cast<const uint32_t*>(qr + 8) : 0u;
  }
}

// Consume the warp's 8 rows of two consecutive stages (n[1] == 0: no second stage; its rows are
// masked and read stage 0's tile instead, so no stale shared memory enters the MMA).
template <int D, int G, bool UNIFIED>
__device__ __forceinline__ void mma_consume(const Params& p, MmaState<D, G>& st,
                                            const uint8_t* const (&ks)[2],
                                            const uint8_t* const (&vs)[2], const int (&n)[2],
                                            int row0, int lane, uint32_t& fmask) {
  constexpr int KS = MmaState<D, G>::KS;
  const uint32_t kb[2] = {smem_u32(ks[0]), smem_u32(n[1] > 0 ? ks[1] : ks[0])};
  const uint32_t vb[2] = {smem_u32(vs[0]), smem_u32(n[1] > 0 ? vs[1] : vs[0])};

  // logits S = Q K^T for the 8 rows of each stage (one 16x8 accumulator per stage)
  float s[2][4];
#pragma unroll
  for (int b = 0; b < 2; ++b)
#pragma unroll
    for (int i = 0; i < 4; ++i) s[b][i] = 0.f;
  const int lrow = lane & 7, lmat = lane >> 3;
#pragma unroll
  for (int k2 = 0; k2 < KS / 2; ++k2) {
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      uint32_t r0, r1, r2, r3;
      ldsm_x4(swz<D>(kb[b], row0 + lrow, k2 * 32 + lmat * 8), r0, r1, r2, r3);
      mma_bf16(s[b], st.qa[2 * k2][0], st.qa[2 * k2][1], r0, r1);
      mma_bf16(s[b], st.qa[2 * k2 + 1][0], st.qa[2 * k2 + 1][1], r2, r3);
    }
  }

  // softmax on the accumulator elements this lane holds: head lane/4, tokens
  // 2 (lane % 4) + {0, 1} of each stage; the quad of lanes 4h..4h+3 holds head h's 16 logits
  const int head = lane >> 2, tk = 2 * (lane & 3);
  const bool hv = head < G;
  float x[2][2];
  bool valid[2][2];
#pragma unroll
  for (int b = 0; b < 2; ++b)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      x[b][e] = s[b][e] * p.qscale;
      valid[b][e] = hv && row0 + tk + e < n[b];
    }
  float ref = p.phi2;
  if constexpr (!UNIFIED) {
    float mx = -INFINITY;
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
      for (int e = 0; e < 2; ++e)
        if (valid[b][e]) mx = fmaxf(mx, x[b][e]);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(st.m, mx);
    if (__any_sync(0xffffffffu, m_new > st.m)) {
      const float alpha = m_new > st.m ? fast_exp2(st.m - m_new) : 1.f;   // 0 from -inf
#pragma unroll
      for (int j = 0; j < MmaState<D, G>::NT; ++j) {
        st.o[j][0] *= alpha;   // rows 8..15 ([2], [3]) stay zero
        st.o[j][1] *= alpha;
      }
      st.den *= alpha;
      st.m = m_new;
    }
    ref = st.m;   // -inf only while all of the head's tokens so far are masked
  }
  float pr[2][2];
#pragma unroll
  for (int b = 0; b < 2; ++b)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      pr[b][e] = valid[b][e] ? fast_exp2(x[b][e] - ref) : 0.f;
      if (UNIFIED && valid[b][e] && (x[b][e] < p.lo2 || x[b][e] > p.hi2)) fmask |= 1u << head;
      st.den += pr[b][e];
    }
  // P as A fragments (k = token: stage 0 rows in k 0..7, stage 1 rows in k 8..15), hi + lo
  uint32_t ahi[2], alo[2];
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    ahi[b] = bf16x2_rn(pr[b][0], pr[b][1]);
    const float h0 = __uint_as_float(ahi[b] << 16), h1 = __uint_as_float(ahi[b] & 0xffff0000u);
    alo[b] = bf16x2_rn(pr[b][0] - h0, pr[b][1] - h1);
  }
  // V rows of masked tokens are zeroed in the fragments (0 * NaN would poison the MMA)
  uint32_t vm[2];
#pragma unroll
  for (int b = 0; b < 2; ++b)
    vm[b] = (row0 + tk < n[b] ? 0x0000ffffu : 0u) | (row0 + tk + 1 < n[b] ? 0xffff0000u : 0u);

  // O += P V, 16 output columns per ldmatrix.x4.trans: matrices (stage 0, cols +0..7),
  // (stage 1, +0..7), (stage 0, +8..15), (stage 1, +8..15)
  const int vst = lmat & 1, vcol = (lmat >> 1) * 8;
#pragma unroll
  for (int j2 = 0; j2 < D / 16; ++j2) {
    uint32_t v0, v1, v2, v3;
    ldsm_x4_t(swz<D>(vb[vst], row0 + lrow, j2 * 16 + vcol), v0, v1, v2, v3);
    v0 &= vm[0];
    v1 &= vm[1];
    v2 &= vm[0];
    v3 &= vm[1];
    mma_bf16(st.o[2 * j2], ahi[0], ahi[1], v0, v1);
    mma_bf16(st.o[2 * j2], alo[0], alo[1], v0, v1);
    mma_bf16(st.o[2 * j2 + 1], ahi[0], ahi[1], v2, v3);
    mma_bf16(st.o[2 * j2 + 1], alo[0], alo[1], v2, v3);
  }
}

}  // namespace da
