// compkv_decode_static: the decode step with the library's own scratch.
//
// Some callers cannot allocate device memory when they call us: an engine
// that reserved the whole GPU for its KV-cache pool at start-up and gives
// plug-ins no allocator, code running under a memory budget where a new
// cudaMalloc would fail or force a device-wide synchronisation, or a host
// application that owns the CUDA context and forbids its plug-ins to allocate.
// For them this entry point runs the same fused decode kernel as
// compkv_decode, but its scratch is the file-scope device array below instead
// of a caller buffer.  The array has a fixed size and every GPU that loads
// the library keeps it until the process exits.
//
// In host code `g_compkv_static_scratch` is only a host-side handle for the
// device symbol, not a device address: the address is fetched once per
// device with cudaGetSymbolAddress, with that device current, and passed to
// the kernel.
#include <mutex>

#include "../../include/compkv.h"

static __device__ __align__(256) unsigned char g_compkv_static_scratch[COMPKV_STATIC_SCRATCH_BYTES];

compkv_status compkv_internal_decode_in(const compkv_config* cfg, const compkv_buffers* bufs, void* scratch,
                                        size_t scratch_bytes, int layer, const float* q, const void* k_new,
                                        const void* v_new, float* out, int* sel, void* stream);
compkv_status compkv_internal_fail(compkv_status st, const char* what, const char* detail);

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the static scratch on the current device (looked up on
// the first call made with that device current).
cudaError_t static_scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_compkv_static_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}
}  // namespace

extern "C" compkv_status compkv_decode_static(const compkv_config* cfg, const compkv_buffers* bufs, int layer,
                                              const float* q, const void* k_new, const void* v_new, float* out,
                                              int* sel, void* stream) {
  void* scratch = nullptr;
  const cudaError_t e = static_scratch_address(&scratch);
  if (e != cudaSuccess) return compkv_internal_fail(COMPKV_ERR_CUDA, "static scratch address", cudaGetErrorString(e));
  return compkv_internal_decode_in(cfg, bufs, scratch, COMPKV_STATIC_SCRATCH_BYTES, layer, q, k_new, v_new, out, sel,
                                   stream);
}
