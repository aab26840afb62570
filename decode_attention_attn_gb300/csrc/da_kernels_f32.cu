// da_kernels_f32.cu -- instantiations of the split-KV kernel for float storage.
#include "da_kernel.cuh"

namespace da {

const void* kernel_f32(int head_dim, int group, int mode) {
  if (head_dim == 64) return pick_kernel<float, 64>(group, mode);
  if (head_dim == 128) return pick_kernel<float, 128>(group, mode);
  return nullptr;
}

}  // namespace da
