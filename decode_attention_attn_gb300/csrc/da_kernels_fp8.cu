// da_kernels_fp8.cu -- instantiations of the split-KV kernel for FP8 (E4M3) K / V caches with
// bf16 q (tensor-core consumers).
#include "da_kernel.cuh"

namespace da {

const void* kernel_fp8(int head_dim, int group, int mode) {
  if (head_dim == 64) return pick_kernel<fp8e4m3, 64>(group, mode);
  if (head_dim == 128) return pick_kernel<fp8e4m3, 128>(group, mode);
  return nullptr;
}

}  // namespace da
