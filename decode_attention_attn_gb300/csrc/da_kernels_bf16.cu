// da_kernels_bf16.cu -- instantiations of the split-KV kernel for __nv_bfloat16 storage.
#include "da_kernel.cuh"

namespace da {

const void* kernel_bf16(int head_dim, int group, int mode) {
  if (head_dim == 64) return pick_kernel<__nv_bfloat16, 64>(group, mode);
  if (head_dim == 128) return pick_kernel<__nv_bfloat16, 128>(group, mode);
  return nullptr;
}

}  // namespace da
