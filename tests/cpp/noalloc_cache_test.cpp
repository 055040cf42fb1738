// Host-only check of the no-alloc scratch address cache (gated_deltanet_cpr_gb300/csrc/
// noalloc_cache.h) with fake context identities and fake symbol lookups: no GPU, no CUDA.
// Prints "ok" and returns 0 when every case holds; otherwise names the failed case.
#include <stdint.h>
#include <stdio.h>

#include "../../gated_deltanet_cpr_gb300/csrc/noalloc_cache.h"

namespace {
int failures = 0;
void expect(bool c, const char* what) {
  if (!c) {
    printf("FAILED: %s\n", what);
    ++failures;
  }
}

struct Fake {
  bool ctx_ok = true;   // whether the current context's identity can be read
  uint64_t ctx = 7;     // the current context's identity
  bool lookup_ok = true;
  uintptr_t addr = 0x1000;
  int lookups = 0;
};
}  // namespace

int main() {
  using Cache = gdn::ScratchAddressCache<4>;
  Fake f;
  auto ctx_id = [&f](uint64_t* id) {
    if (!f.ctx_ok) return false;
    *id = f.ctx;
    return true;
  };
  auto lookup = [&f](void** p) {
    ++f.lookups;
    if (!f.lookup_ok) return false;
    *p = reinterpret_cast<void*>(f.addr);
    return true;
  };
  Cache c;
  void* p = nullptr;

  expect(c.get(0, ctx_id, lookup, &p) == Cache::kOk && p == (void*)0x1000 && f.lookups == 1,
         "first call looks the address up");
  expect(c.get(0, ctx_id, lookup, &p) == Cache::kOk && p == (void*)0x1000 && f.lookups == 1,
         "same context: cached, no second lookup");

  // the context is destroyed and made again (device reset): new identity, new address
  f.ctx = 8;
  f.addr = 0x2000;
  expect(c.get(0, ctx_id, lookup, &p) == Cache::kOk && p == (void*)0x2000 && f.lookups == 2,
         "new context: looked up again, new address returned");
  expect(c.get(0, ctx_id, lookup, &p) == Cache::kOk && p == (void*)0x2000 && f.lookups == 2,
         "new context: cached afterwards");

  // another device has its own entry
  f.addr = 0x3000;
  expect(c.get(1, ctx_id, lookup, &p) == Cache::kOk && p == (void*)0x3000 && f.lookups == 3,
         "second device: its own lookup");
  f.addr = 0x2000;
  expect(c.get(0, ctx_id, lookup, &p) == Cache::kOk && p == (void*)0x2000 && f.lookups == 3,
         "first device still cached");

  // a failed lookup is reported and not cached
  f.ctx = 9;
  f.lookup_ok = false;
  p = nullptr;
  expect(c.get(0, ctx_id, lookup, &p) == Cache::kLookupFailed && p == nullptr && f.lookups == 4,
         "failed lookup reported");
  f.lookup_ok = true;
  f.addr = 0x4000;
  expect(c.get(0, ctx_id, lookup, &p) == Cache::kOk && p == (void*)0x4000 && f.lookups == 5,
         "after a failed lookup the next call looks up again");

  // identity unreadable: the address is returned but never kept
  f.ctx_ok = false;
  f.addr = 0x5000;
  expect(c.get(2, ctx_id, lookup, &p) == Cache::kOk && p == (void*)0x5000 && f.lookups == 6,
         "unknown identity: looked up");
  expect(c.get(2, ctx_id, lookup, &p) == Cache::kOk && p == (void*)0x5000 && f.lookups == 7,
         "unknown identity: looked up on every call");
  expect(c.get(0, ctx_id, lookup, &p) == Cache::kOk && f.lookups == 8,
         "unknown identity: a cached entry is not trusted");

  // device index outside the table
  f.ctx_ok = true;
  expect(c.get(-1, ctx_id, lookup, &p) == Cache::kBadDevice, "negative device rejected");
  expect(c.get(4, ctx_id, lookup, &p) == Cache::kBadDevice, "device beyond the table rejected");
  expect(f.lookups == 8, "rejected devices do no lookup");

  if (failures == 0) printf("ok\n");
  return failures == 0 ? 0 : 1;
}
