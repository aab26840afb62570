// da_merge.cu -- the split-KV reduction kernel: exact log-sum-exp merge of the partials of
// every group that the split kernel cut into more than one piece ("Flash-Decoding:
// Mathematical Foundations, ...", "The Rescaling and Online Softmax Reduction Algorithm":
// L = log sum_s exp(L_s), O = sum_s exp(L_s - L) O_s), plus each row's overflow flag, the OR
// of its pieces' range checks (FlashDecoding++, "The Overflow Fallback: Recomputation").
//
// It is launched right behind the split kernel as a programmatic dependent with no shared
// memory, so its CTAs become resident beside the split kernel's and start merging as soon as
// the split kernel's writes are visible. One warp owns one (group, row, 32-wide d chunk) and
// takes the group's pieces 32 at a time: lane s loads piece s's L and flags while every lane
// loads its d element of all 32 partial outputs (coalesced 128-byte rows), all before any is
// used, so a block costs one L2 round trip; blocks combine with a running max rescale.
#include "da_device.cuh"

namespace da {

__global__ void __launch_bounds__(128) merge_kernel(const __grid_constant__ MergeParams mp) {
  pdl_wait();
  pdl_launch_dependents();
  constexpr float kLn2 = 0.6931471805599453f;
  constexpr int kBlk = 32;   // pieces whose loads are all in flight at once
  const int lane = threadIdx.x & 31;
  const int R = mp.rows_per_group, D = mp.head_dim, DC = D / 32;
  const long long items = (long long)mp.n_groups * R * DC;
  const long long nwarps = (long long)gridDim.x * (blockDim.x / 32);
  for (long long it = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; it < items;
       it += nwarps) {
    const int g = (int)(it / (R * DC));
    const int r = (int)((it / DC) % R);
    const int c = (int)(it % DC);
    const int2 ds = mp.desc[g];
    const int S = ds.y;
    if (S <= 1) continue;   // written directly by the split kernel (or an empty sequence)
    const long long base = ds.x;
    const float* pl = mp.part_l + base * R + r;                         // stride R per piece
    const float* po = mp.part_o + (base * R + r) * D + c * 32 + lane;   // stride R * D
    const long long so = (long long)R * D;
    // running (max, sum of weights, weighted sum) over blocks of 32 pieces
    float m_run = -INFINITY, sum = 0.f, num = 0.f;
    uint32_t f = 0;
    for (int s0 = 0; s0 < S; s0 += kBlk) {
      const int cnt = min(kBlk, S - s0);
      // every load of the block is issued before any is used
      const float L = lane < cnt ? __ldcg(pl + (long long)(s0 + lane) * R) : -INFINITY;
      if (c == 0 && lane < cnt) f |= __ldcg(mp.part_flags + base + s0 + lane);
      float o[kBlk];
#pragma unroll
      for (int k = 0; k < kBlk; ++k) o[k] = k < cnt ? __ldcg(po + (long long)(s0 + k) * so) : 0.f;
      float M = L;
#pragma unroll
      for (int x = 16; x >= 1; x >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, x));
      const float m_new = fmaxf(m_run, M);
      if (m_new == -INFINITY) continue;   // every piece so far is empty
      const float scale = m_run == -INFINITY ? 0.f : fast_exp2(m_run - m_new);
      const float w = L > -INFINITY ? fast_exp2(L - m_new) : 0.f;
      float bsum = w;
#pragma unroll
      for (int x = 16; x >= 1; x >>= 1) bsum += __shfl_xor_sync(0xffffffffu, bsum, x);
      float bnum = 0.f;
#pragma unroll
      for (int k = 0; k < kBlk; ++k) bnum += __shfl_sync(0xffffffffu, w, k) * o[k];
      sum = sum * scale + bsum;
      num = num * scale + bnum;
      m_run = m_new;
    }
    const long long row = (long long)g * R + r;
    store_out(mp.out, row * D + c * 32 + lane, mp.out_dtype, sum > 0.f ? num / sum : 0.f);
    if (c == 0) {
      f = __reduce_or_sync(0xffffffffu, f);
      if (lane == 0) {
        if (mp.out_lse) mp.out_lse[row] = sum > 0.f ? (m_run + fast_log2(sum)) * kLn2 : -INFINITY;
        if (mp.row_flags && mp.write_flags) mp.row_flags[row] = (uint8_t)((f >> r) & 1u);
        if (r == 0 && mp.write_flags && f) {
          atomicAdd(mp.stats + 0, (unsigned long long)__popc(f));
          const int at = atomicAdd(mp.list_state, 1);
          if (at < mp.n_groups) mp.flag_list[at] = g;
        }
      }
    }
  }
}

const void* merge_kernel_ptr() { return reinterpret_cast<const void*>(&merge_kernel); }

}  // namespace da
