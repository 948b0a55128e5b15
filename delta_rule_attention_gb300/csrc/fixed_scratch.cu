// falcon1_fwd_chunked_fixed_scratch: the Falcon-1 chunked forward for callers
// that cannot allocate device memory.
//
// The regular entry point needs a caller-provided workspace (the per-chunk
// affine maps written by the first launch and read by the second).  Some
// callers have no way to provide one: a C host program or plugin that is
// handed only its input and output buffers, a framework whose allocator is
// not reachable from the call site, or a serving loop that forbids any
// allocation after start-up.  This entry point serves them with scratch that
// lives in the library itself: a file-scope __device__ array of fixed size,
// FALCON_FIXED_SCRATCH_BYTES, which every GPU that loads the library holds
// until the process exits.
//
// Set-up: the first call on each device (with that device current) asks the
// runtime for the array's device address with cudaGetSymbolAddress and keeps
// it for later calls.  In host code the array's name is only a host-side
// stand-in, never a device address, so kernels get the resolved pointer.
// Make that first call before any stream capture begins on the device.
//
// All calls on a device share the one array and it keeps the previous call's
// contents.  Nothing needs clearing: the first launch writes every scratch
// element the second launch reads.  Calls whose GPU work overlaps (different
// streams, or host threads racing on one device) race on the array; order
// them on one stream.
#include <mutex>

#include "common.cuh"

namespace falcon {
// Defined with the C ABI: the Falcon-1 chunked forward over a workspace of
// workspace_bytes whose device address `resolve` gives once the argument and
// device checks have passed.
int fwd_chunked_resolved(const falcon_shape* s, const void* q, const void* k, const void* v,
                         const float* beta, const float* lambda, const float* S0,
                         const float* x_prev, void* o, float* S_out, float* x_last,
                         int (*resolve)(void**), size_t workspace_bytes, cudaStream_t stream);
}  // namespace falcon

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_fixed_scratch[FALCON_FIXED_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_fixed_scratch on the current device (resolved once).
int fixed_scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FALCON_ERR_CUDA;
  // A device ordinal beyond the library's per-device table: a runtime
  // configuration the library cannot serve, reported like a failed query.
  if (dev < 0 || dev >= kMaxDevices) return FALCON_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fixed_scratch) != cudaSuccess || !p) return FALCON_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FALCON_OK;
}

}  // namespace

extern "C" int falcon1_fwd_chunked_fixed_scratch(const falcon_shape* shape, const void* q,
                                                 const void* k, const void* v, const float* beta,
                                                 const float* lambda, const float* S0,
                                                 const float* x_prev, void* o, float* S_out,
                                                 float* x_last, cudaStream_t stream) {
  // falcon_workspace_bytes is 0 for a NULL or invalid shape, which the
  // forward's own checks then reject; the array's address is resolved only
  // after every argument check has passed.
  if (falcon_workspace_bytes(shape) > (size_t)FALCON_FIXED_SCRATCH_BYTES)
    return FALCON_ERR_SCRATCH_LIMIT;
  return falcon::fwd_chunked_resolved(shape, q, k, v, beta, lambda, S0, x_prev, o, S_out, x_last,
                                      fixed_scratch_address, (size_t)FALCON_FIXED_SCRATCH_BYTES,
                                      stream);
}
