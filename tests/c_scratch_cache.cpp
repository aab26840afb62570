// Host-side check of the per-context address cache behind decode_attn_run_static (plain C++,
// no CUDA): a context is resolved once, a new context ID (a device reset, a caller's own driver
// context) is resolved again, a failed lookup is not cached, and a full cache replaces its
// oldest entry.
#include <cstdio>

#include "da_scratch_cache.h"

static int fails = 0;
#define CHECK(c) do { if (!(c)) { std::printf("FAIL line %d: %s\n", __LINE__, #c); ++fails; } } while (0)

int main() {
  da::SymbolAddressCache<2> cache;
  int calls = 0;
  char a, b, c;
  void* next = &a;
  int next_rc = 0;
  auto resolve = [&](void** out) { ++calls; *out = next; return next_rc; };
  void* got = nullptr;
  CHECK(cache.get(7, resolve, &got) == 0 && got == &a && calls == 1);
  next = &b;
  CHECK(cache.get(7, resolve, &got) == 0 && got == &a && calls == 1);   // cached
  CHECK(cache.get(8, resolve, &got) == 0 && got == &b && calls == 2);   // new context
  next_rc = -5;
  CHECK(cache.get(9, resolve, &got) == -5 && calls == 3);                // error returned
  next_rc = 0;
  next = &c;
  CHECK(cache.get(9, resolve, &got) == 0 && got == &c && calls == 4);   // not cached on error
  CHECK(cache.get(8, resolve, &got) == 0 && got == &b && calls == 4);   // still held
  CHECK(cache.get(7, resolve, &got) == 0 && calls == 5);                 // the oldest was replaced
  if (fails == 0) std::printf("ok\n");
  return fails ? 1 : 0;
}
