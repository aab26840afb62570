// da_kernels_fp8.cu -- instantiations of the split-KV kernel for FP8 (E4M3) K / V caches with
// bf16 q (tensor-core consumers), and of its packed form for pairs of KV heads with groups of 4
// query heads each (8 query heads per split-kernel group).
#include "da_kernel.cuh"

namespace da {

const void* kernel_fp8(int head_dim, int group, int mode, int kv_heads) {
  if (kv_heads == 2) {
    if (group != 8) return nullptr;
    if (head_dim == 64) return pick_mode<fp8e4m3_heads<2>, 64, 8>(mode);
    if (head_dim == 128) return pick_mode<fp8e4m3_heads<2>, 128, 8>(mode);
    return nullptr;
  }
  if (kv_heads != 1) return nullptr;
  if (head_dim == 64) return pick_kernel<fp8e4m3, 64>(group, mode);
  if (head_dim == 128) return pick_kernel<fp8e4m3, 128>(group, mode);
  return nullptr;
}

}  // namespace da
