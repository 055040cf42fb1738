// noalloc.cu -- a decode step for callers that cannot allocate device memory.
//
// gdn_cpr_decode_step needs a workspace for the resynchronisation every C tokens.  Some
// callers cannot provide one: a serving loop whose device memory is reserved up front by
// another allocator, code that must not call cudaMalloc while other work is being
// captured or replayed, or plain C hosts with no device allocator of their own.  For them
// gdn_cpr_decode_step_noalloc runs the very same decode step with its workspace placed in
// the fixed-size device array below, which the CUDA runtime reserves on each device when
// this library's module is loaded there and releases only at process exit.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "../../include/gdn_cpr.h"
#include "noalloc_cache.h"

namespace {

constexpr size_t kScratchBytes = GDN_CPR_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

// Host code cannot use &g_decode_scratch as a device address (it names a host-side
// stand-in), so each device's address is looked up with that device current and cached
// together with the identity of the context it belongs to (see noalloc_cache.h).
gdn::ScratchAddressCache<64> g_scratch;

// Driver entry points for the current context's identity, resolved through the runtime
// (no link against the driver library).  Either may stay NULL on an old driver; then the
// address is looked up on every call.
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_entry_once;

void resolve_entry_points() {
  std::call_once(g_entry_once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
    cudaGetLastError();
  });
}

bool current_context_id(uint64_t* id) {
  if (!g_ctx_current || !g_ctx_id) return false;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  unsigned long long v = 0;
  if (g_ctx_id(ctx, &v) != CUDA_SUCCESS) return false;
  *id = (uint64_t)v;
  return true;
}

gdn_status scratch_of_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
  resolve_entry_points();
  auto lookup = [](void** p) {
    if (cudaGetSymbolAddress(p, g_decode_scratch) != cudaSuccess) {
      cudaGetLastError();  // do not leave the failure pending for the caller's next call
      return false;
    }
    return true;
  };
  return g_scratch.get(dev, current_context_id, lookup, out) == decltype(g_scratch)::kOk ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

extern "C" gdn_status gdn_cpr_decode_step_noalloc(const gdn_cpr_shape* shape, const void* q,
                                                  const void* k, const void* v, const float* g,
                                                  const float* beta, const int32_t* slot,
                                                  const gdn_cpr_cache* cache, void* o,
                                                  gdn_stream_t stream) {
  size_t need = 0;
  gdn_status rc = gdn_cpr_workspace_size(shape, GDN_MODE_DECODE, nullptr, &need);
  if (rc != GDN_OK) return rc;
  if (need > kScratchBytes) return GDN_ERR_WORKSPACE;
  void* ws = nullptr;
  rc = scratch_of_current_device(&ws);
  if (rc != GDN_OK) return rc;
  return gdn_cpr_decode_step(shape, q, k, v, g, beta, slot, cache, o, ws, kScratchBytes, stream);
}

extern "C" gdn_status gdn_cpr_noalloc_device_error(gdn_stream_t stream, int32_t* code) {
  if (!code) return GDN_ERR_INVALID_ARG;
  void* ws = nullptr;
  const gdn_status rc = scratch_of_current_device(&ws);
  if (rc != GDN_OK) return rc;
  return gdn_cpr_get_device_error(ws, stream, code);
}
