// noalloc_cache.h -- per-device cache of the built-in scratch array's device address, for
// gdn_cpr_decode_step_noalloc.  Host code only; no CUDA types, so the logic can be compiled
// and tested on its own with fake lookups.
//
// The address of a __device__ array is only valid in the context it was looked up in.  If a
// device's primary context is destroyed (cudaDeviceReset) and made again, the module is
// loaded again and the array may sit elsewhere, so an address cached by device index alone
// could point at unmapped memory.  Each entry therefore records the identity of the context
// it was looked up in (a driver context ID, unique for the process's lifetime) and is looked
// up again whenever the current context's identity differs.  When the identity cannot be
// read, nothing is cached and every call looks the address up.
#pragma once

#include <stdint.h>

#include <mutex>

namespace gdn {

template <int kMaxDevices>
class ScratchAddressCache {
 public:
  enum Result { kOk = 0, kBadDevice = 1, kLookupFailed = 2 };

  // dev: the current device index.  ctx_id(uint64_t* id) -> bool: the current context's
  // identity (false if none is current or it cannot be read).  lookup(void** p) -> bool: the
  // array's address in the current context (making the device's primary context current if
  // none was).  On kOk, *out is an address valid in the current context.
  template <class CtxId, class Lookup>
  Result get(int dev, CtxId ctx_id, Lookup lookup, void** out) {
    if (dev < 0 || dev >= kMaxDevices) return kBadDevice;
    std::lock_guard<std::mutex> lock(mu_);
    Entry& e = entry_[dev];
    uint64_t id = 0;
    if (e.addr != nullptr && ctx_id(&id) && id == e.ctx) {
      *out = e.addr;
      return kOk;
    }
    void* p = nullptr;
    if (!lookup(&p) || p == nullptr) return kLookupFailed;
    if (ctx_id(&id)) {
      e.ctx = id;
      e.addr = p;
    } else {
      e.addr = nullptr;  // identity unknown: do not keep an address that could go stale
    }
    *out = p;
    return kOk;
  }

 private:
  struct Entry {
    uint64_t ctx = 0;
    void* addr = nullptr;
  };
  std::mutex mu_;
  Entry entry_[kMaxDevices];
};

}  // namespace gdn
