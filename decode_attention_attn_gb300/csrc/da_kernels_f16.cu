// da_kernels_f16.cu -- instantiations of the split-KV kernel for __half storage.
#include "da_kernel.cuh"

namespace da {

const void* kernel_f16(int head_dim, int group, int mode) {
  if (head_dim == 64) return pick_kernel<__half, 64>(group, mode);
  if (head_dim == 128) return pick_kernel<__half, 128>(group, mode);
  return nullptr;
}

}  // namespace da
