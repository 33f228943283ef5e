// Selective-scan entry point for callers that must not allocate device memory.
//
// The regular entry point takes its chunk-carry workspace from a stream-ordered
// memory pool.  Some callers cannot let a library allocate: an application that hands
// all device memory to its own arena at start-up, a serving loop that forbids any
// allocation after warm-up so that latency and memory use stay fixed, or code whose
// allocator must not be entered from this thread.  For them this file keeps the
// workspace in a fixed, file-scope device array instead.
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "scan_internal.h"
#include "ssm_scan.h"

namespace {

// The workspace of every no-allocation call on a device: SSM_NOALLOC_SCRATCH_BYTES,
// loaded with the library on every GPU that uses it and held until the process ends.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SSM_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
std::vector<void*> g_addr;  // device address of g_noalloc_scratch, per device ordinal

// The scratch's device address on the current device.  The host-side symbol is only a
// stand-in; the address must be asked of the runtime once per device, with that device
// current.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SSM_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if ((int)g_addr.size() <= dev) g_addr.resize(dev + 1, nullptr);
  if (!g_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return SSM_ERR_CUDA;
    g_addr[dev] = ptr;
  }
  *out = g_addr[dev];
  return SSM_OK;
}

}  // namespace

extern "C" int ssm_selective_scan_fwd_noalloc(const void* x, const void* delta, const float* A,
                                              const void* B, const void* C, const float* D,
                                              const void* z, const float* delta_bias, void* out,
                                              float* final_state, const ssm_dims* dims,
                                              cudaStream_t stream) {
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != SSM_OK) return rc;
  // The call clears the scratch's chunk-carry flags itself (in stream order) before its
  // kernel; everything else a kernel reads from the scratch was written earlier in the
  // same call.
  return ssm_internal::scan_forward(x, delta, A, B, C, D, z, delta_bias, out, final_state, dims, stream,
                                    scratch, SSM_NOALLOC_SCRATCH_BYTES, nullptr);
}
