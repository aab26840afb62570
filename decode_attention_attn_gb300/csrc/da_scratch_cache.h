// da_scratch_cache.h -- host-side cache of a device symbol's address, one entry per CUDA
// context (host code only; no CUDA types).
//
// A __device__ variable has one address per context that loaded the module holding it: a
// device reset gives the device a new primary context, and a caller may run its own driver
// context on the same device. The key is the context's unique ID (cuCtxGetId), which no later
// context reuses, so a cached address is never applied to a context it does not belong to.
#pragma once

#include <mutex>

namespace da {

template <int N>
class SymbolAddressCache {
 public:
  // The address for context `ctx_id`: cached, or resolve(&addr) (returning 0 on success),
  // which is then cached. When all N entries are taken the oldest is replaced.
  template <class Resolve>
  int get(unsigned long long ctx_id, Resolve&& resolve, void** out) {
    std::lock_guard<std::mutex> lock(mu_);
    for (int i = 0; i < used_; ++i) {
      if (ids_[i] == ctx_id) {
        *out = addr_[i];
        return 0;
      }
    }
    void* a = nullptr;
    const int rc = resolve(&a);
    if (rc != 0) return rc;
    const int slot = used_ < N ? used_++ : next_;
    if (used_ == N) next_ = (slot + 1) % N;
    ids_[slot] = ctx_id;
    addr_[slot] = a;
    *out = a;
    return 0;
  }

 private:
  std::mutex mu_;
  unsigned long long ids_[N] = {};
  void* addr_[N] = {};
  int used_ = 0, next_ = 0;
};

}  // namespace da
