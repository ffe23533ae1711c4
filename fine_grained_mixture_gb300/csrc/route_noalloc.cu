// route_noalloc.cu - moe_route_noalloc: the routing call for callers that cannot allocate device memory.
//
// Some callers of this library never get to call cudaMalloc: a plugin inside a host program whose
// allocator owns every device byte and forbids raw allocations, or a request path under a fixed memory
// budget where an allocation (and the device synchronisation cudaMalloc may imply) is not allowed.  They
// still own the routing outputs and pass them in; only the routing scratch moves into a fixed-size
// array that is part of the library image on every GPU that loads it.
//
// The array is a file-scope __device__ symbol.  Host code cannot pass the symbol itself to a kernel (on
// the host it names a host-side shadow, not device memory), so the device address is looked up with
// cudaGetSymbolAddress, once per device, on the first call made with that device current.
#include <mutex>

#include "internal.h"

namespace moe {
namespace {

static __device__ __align__(256) unsigned char g_route_scratch[MOE_ROUTE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxScratchDevices] = {nullptr};

// Device address of g_route_scratch on the current device (looked up on first use per device).
int scratch_address(void **out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return record_cuda_error(err);
  if (dev < 0 || dev >= kMaxScratchDevices) return MOE_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    err = cudaGetSymbolAddress(&p, g_route_scratch);
    if (err != cudaSuccess) {
      cudaGetLastError();  // do not leave the failure pending for a later, unrelated error check
      return record_cuda_error(err);
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" int moe_route_noalloc(const float *logits, int T, int E, int K, int mode, const moe_routing *r,
                                 int32_t *P_host, void *stream) {
  // stochastic rounding needs per-expert uniforms, which only moe_route_ex takes
  if (mode == MOE_ROUTE_TR_STOCHASTIC) return MOE_ERR_INVALID_ARG;
  size_t need = 0;
  int rc = moe_route_workspace_size(T, E, K, mode, &need);
  if (rc != MOE_OK) return rc;
  // token rounding's expert-major key copy (4*T*E bytes) is a speed-up, not a necessity: drop it when it
  // would not fit, and the selection reads the logits in place
  bool em_keys = true;
  if (need > MOE_ROUTE_NOALLOC_SCRATCH_BYTES) {
    em_keys = false;
    need = moe::route_workspace_bytes(T, E, K, mode, false);
  }
  if (need > MOE_ROUTE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;
  // the device check comes first, so a wrong GPU reads MOE_ERR_DEVICE (as from moe_route) rather than a
  // failed symbol lookup
  rc = moe::check_device();
  if (rc != MOE_OK) return rc;
  void *scratch = nullptr;
  rc = moe::scratch_address(&scratch);
  if (rc != MOE_OK) return rc;
  // Same kernels and validation as moe_route; the scratch is the library's own array instead of the
  // caller's workspace.  Every per-call scratch word is rewritten before it is read.
  return moe::route_call(logits, nullptr, T, E, K, mode, r, scratch, need, P_host, stream, em_keys);
}
