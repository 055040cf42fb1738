// noalloc.cu -- a decode step for callers that cannot allocate device memory.
//
// gdn_cpr_decode_step needs a workspace for the resynchronisation every C tokens.  Some
// callers cannot provide one: a serving loop whose device memory is reserved up front by
// another allocator, code that must not call cudaMalloc while other work is being
// captured or replayed, or plain C hosts with no device allocator of their own.  For them
// gdn_cpr_decode_step_noalloc runs the very same decode step with its workspace placed in
// the fixed-size device array below, which the CUDA runtime reserves on each device when
// this library's module is loaded there and releases only at process exit.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/gdn_cpr.h"

namespace {

constexpr size_t kScratchBytes = GDN_CPR_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

// Host code cannot use &g_decode_scratch as a device address (it names a host-side
// stand-in), so each device's address is fetched once, with that device current.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

gdn_status scratch_of_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // do not leave the failure pending for the caller's next call
      return GDN_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return GDN_OK;
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
