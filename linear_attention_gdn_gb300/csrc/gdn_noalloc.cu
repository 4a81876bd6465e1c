// gdn_noalloc.cu -- a forward entry point for callers that cannot allocate
// device memory.
//
// Some hosts hand a library only its input and output buffers: plugin-style
// runtimes that have no workspace query in their interface, or latency-bound
// callers that may not call cudaMalloc on their path (it synchronises the
// device).  gdn_fwd_noalloc() serves them by running the ordinary forward with
// its workspace placed in a fixed array that lives in device memory for as
// long as the library is loaded, instead of in a caller-owned buffer.
//
// The array is a file-scope __device__ variable.  Host code cannot use its
// name as a device address (the host-side symbol is only a stand-in), so the
// entry point looks the address up with cudaGetSymbolAddress once per device,
// on the first call made with that device current, and passes that pointer
// down.  That first call therefore does set-up work and should be made before
// any stream capture.  No cudaMalloc, cudaFree or allocating library routine
// is called here or in the forward it delegates to.
#include <cuda_runtime.h>

#include <mutex>

#include "gdn.h"

namespace {

static __device__ __align__(256) unsigned char g_fwd_scratch[GDN_FWD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;

// device address of g_fwd_scratch on the current device (looked up once per device)
gdn_status scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fwd_scratch) != cudaSuccess || !p) return GDN_ERR_CUDA;
    addr[dev] = p;
  }
  *out = addr[dev];
  return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_fwd_noalloc(const gdn_problem* prob, const void* q, const void* k, const void* v,
                                      const float* g, const float* beta, const int32_t* cu_seqlens_dev,
                                      const int32_t* cu_seqlens_host, void* o, struct CUstream_st* stream) {
  if (!o) return GDN_ERR_INVALID_ARG;
  void* scratch = nullptr;
  gdn_status st = scratch_address(&scratch);
  if (st != GDN_OK) return st;
  // gdn_fwd refuses (GDN_ERR_WORKSPACE_TOO_SMALL) a problem whose workspace
  // would not fit in the fixed array; it clears the error word it keeps there
  return gdn_fwd(prob, q, k, v, g, beta, cu_seqlens_dev, cu_seqlens_host, o, nullptr, scratch,
                 (size_t)GDN_FWD_NOALLOC_SCRATCH_BYTES, stream);
}
