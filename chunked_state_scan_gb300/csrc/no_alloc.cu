// no_alloc.cu -- a backward entry point whose scratch memory lives inside the
// library, for callers that cannot allocate device memory.
//
// zeco_gla_bwd needs a caller-provided workspace.  Some callers have no way to
// provide one: code running where cudaMalloc is forbidden or unavailable (for
// example inside a host callback or a custom allocator hook that must not
// recurse into the allocator), plugins whose host framework owns all device
// memory and hands out only input/output buffers, or real-time code that may
// not allocate after start-up.  zeco_gla_bwd_noalloc serves them: its
// scratch is a fixed-size array in the library's own device memory, so the
// caller passes only inputs and outputs and nothing is allocated per call.
//
// Costs and limits, stated in include/zeco_gla.h as well:
//   - every GPU that loads this library holds ZECO_NOALLOC_MAX_WS_BYTES of
//     device memory for the array until the process exits;
//   - shapes whose backward workspace (zeco_gla_workspace_bytes(shape, 1))
//     exceeds that size are refused with ZECO_ERR_WORKSPACE;
//   - all calls on one GPU share the array, so calls whose GPU work overlaps
//     (different streams, or threads without ordering) race on it; callers
//     must order them;
//   - the first call on each device looks up the array's device address, with
//     that device current, and caches it for the life of the process; make that
//     first call before any stream capture on that device.  A cudaDeviceReset
//     frees the array with the rest of the device's memory and leaves the cached
//     address stale, so a process must not call this entry point on a device
//     after resetting it.
#include <mutex>

#include "common.cuh"

namespace {

// The scratch itself.  In host code `g_noalloc_ws` names a host-side stand-in,
// not device memory: host code must use the address cudaGetSymbolAddress
// returns for the current device, never the symbol.
static __device__ __align__(256) unsigned char g_noalloc_ws[ZECO_NOALLOC_MAX_WS_BYTES];

constexpr int kMaxDevices = 128;
std::mutex g_mu;
void* g_ws_ptr[kMaxDevices] = {};

// Device address of the array on the current device (looked up by the first
// call on each device, with that device current).
int noalloc_workspace(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ZECO_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_ws_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_ws) != cudaSuccess || !p) return ZECO_ERR_CUDA;
    g_ws_ptr[dev] = p;
  }
  *out = g_ws_ptr[dev];
  return ZECO_OK;
}

}  // namespace

extern "C" int zeco_gla_bwd_noalloc(const zeco_shape* shape, const void* q, const void* k,
                                    const void* v, const void* log_alpha, const void* saved,
                                    const void* d_o, const float* dS_final, void* dq, void* dk,
                                    void* dv, void* dlog_alpha, float* dS0,
                                    zeco_stream_t stream) {
  // invalid or unsupported shapes: the same code as zeco_gla_bwd, before any CUDA call
  const int path = zeco_gla_resolve_path(shape);
  if (path < 0) return path;
  void* ws = nullptr;
  const int rc = noalloc_workspace(&ws);
  if (rc != ZECO_OK) return rc;
  // zeco_gla_bwd checks the pointers and then the scratch size against the
  // array's: oversized shapes get ZECO_ERR_WORKSPACE from it.  Every byte of the
  // workspace that the backward reads it has written earlier in the same call,
  // so the previous call's leftovers need no clearing.
  return zeco_gla_bwd(shape, q, k, v, log_alpha, saved, d_o, dS_final, dq, dk, dv, dlog_alpha,
                      dS0, ws, (size_t)ZECO_NOALLOC_MAX_WS_BYTES, stream);
}
