// gdn_prefill_noalloc: the prefill for callers that cannot allocate device
// memory.
//
// Some callers cannot call cudaMalloc: an inference engine that reserves all
// of HBM for its own memory planner at start-up, a runtime that forbids
// allocation once its serving loop has warmed up (an allocation there can
// stall on the driver or fail under memory pressure), or code that runs from
// inside another allocator's callback, where allocating would re-enter that
// allocator.  gdn_prefill needs a small device workspace; this entry point
// takes it from a fixed array in the library's own device memory instead of
// from the caller or from cudaMallocAsync.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds it (kNoAllocScratchBytes) until the process exits.  Host code
// cannot use the array's name as a device address: it names a host-side
// stand-in.  The device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, on the first call made on
// it; that first call should therefore come before any stream capture.  The
// address is kept for the life of the process: after a cudaDeviceReset() of a
// device the kept address is stale, so a process that resets a device must not
// call this entry point on that device again.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/gdn.h"

namespace {

constexpr size_t kNoAllocScratchBytes = GDN_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, or nullptr.
void *scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_addr[dev] = ptr;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" {

int gdn_prefill_noalloc(const gdn_dims *dims, const void *q, const void *k, const void *v,
                        const void *a, const void *b, const void *z, const float *conv_w,
                        const float *A_log, const float *dt_bias, const float *norm_w,
                        const int32_t *cu_seqlens, const float *init_state, void *out,
                        float *final_state, void *stream) {
  if (gdn_prefill_workspace_bytes(dims) > kNoAllocScratchBytes) return GDN_ERR_WORKSPACE;
  void *scratch = scratch_on_current_device();
  if (!scratch) return GDN_ERR_CUDA;
  // With a workspace given, gdn_prefill allocates nothing; it clears the
  // status word at the start of the scratch on `stream` before its kernels.
  return gdn_prefill(dims, q, k, v, a, b, z, conv_w, A_log, dt_bias, norm_w, cu_seqlens, init_state,
                     out, final_state, scratch, kNoAllocScratchBytes, stream);
}

}  // extern "C"
