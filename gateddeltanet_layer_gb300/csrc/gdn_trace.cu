// Kernel timing trace: CUDA events around each launch, on the launching stream;
// and an NVTX range (host side) around every launch, for profilers.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <mutex>

#include "../../include/gdn_trace.h"
#include "gdn_internal.h"

namespace {

struct Record {
  int kind;
  cudaEvent_t begin, end;
};

struct Trace {
  std::mutex mu;
  bool on = false;
  int device = -1;
  cudaEvent_t pool[2 * GDN_TRACE_MAX_LAUNCHES];
  int pool_size = 0;
  Record rec[GDN_TRACE_MAX_LAUNCHES];
  int n = 0;
  int open = -1;  // index of a launch whose begin event is recorded and end is not
};

Trace &trace() {
  static Trace t;
  return t;
}

}  // namespace

namespace gdn {

void trace_begin(cudaStream_t s, int kind) {
  nvtxRangePushA(gdn_trace_kernel_name(kind));  // host-side range around the launch (no-op without a tool)
  Trace &t = trace();
  std::lock_guard<std::mutex> lock(t.mu);
  if (!t.on || t.open >= 0 || t.n >= GDN_TRACE_MAX_LAUNCHES) return;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != t.device) return;
  Record &r = t.rec[t.n];
  r.kind = kind;
  r.begin = t.pool[2 * t.n];
  r.end = t.pool[2 * t.n + 1];
  if (cudaEventRecord(r.begin, s) != cudaSuccess) return;
  t.open = t.n;
}

void trace_end(cudaStream_t s) {
  nvtxRangePop();
  Trace &t = trace();
  std::lock_guard<std::mutex> lock(t.mu);
  if (t.open < 0) return;
  if (cudaEventRecord(t.rec[t.open].end, s) == cudaSuccess) ++t.n;
  t.open = -1;
}

}  // namespace gdn

extern "C" {

int gdn_trace_enable(int on) {
  Trace &t = trace();
  std::lock_guard<std::mutex> lock(t.mu);
  if (!on) {
    t.on = false;
    return GDN_OK;
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
  if (t.pool_size > 0 && dev != t.device) {  // pool of another device: drop it
    for (int i = 0; i < t.pool_size; ++i) cudaEventDestroy(t.pool[i]);
    t.pool_size = 0;
    t.n = 0;
  }
  while (t.pool_size < 2 * GDN_TRACE_MAX_LAUNCHES) {
    if (cudaEventCreate(&t.pool[t.pool_size]) != cudaSuccess) return GDN_ERR_CUDA;
    ++t.pool_size;
  }
  t.device = dev;
  t.on = true;
  return GDN_OK;
}

int gdn_trace_read(int cap, int *launches, double *total_ms) {
  if (cap < 1 || !launches || !total_ms) return GDN_ERR_INVALID_ARG;
  Trace &t = trace();
  std::lock_guard<std::mutex> lock(t.mu);
  for (int k = 0; k < cap; ++k) {
    launches[k] = 0;
    total_ms[k] = 0.0;
  }
  int status = GDN_OK;
  for (int i = 0; i < t.n; ++i) {
    const Record &r = t.rec[i];
    float ms = 0.0f;
    if (cudaEventSynchronize(r.end) != cudaSuccess || cudaEventElapsedTime(&ms, r.begin, r.end) != cudaSuccess) {
      status = GDN_ERR_CUDA;
      continue;
    }
    if (r.kind >= 0 && r.kind < cap) {
      ++launches[r.kind];
      total_ms[r.kind] += ms;
    }
  }
  t.n = 0;
  t.open = -1;
  return status;
}

const char *gdn_trace_kernel_name(int kind) {
  switch (kind) {
    case GDN_K_CHUNK_TABLE: return "chunk_table_kernel";
    case GDN_K_CHUNK_PREP: return "chunk_prep_kernel";
    case GDN_K_STATE: return "state_kernel";
    case GDN_K_PREFILL_SIMT: return "prefill_simt_kernel";
    case GDN_K_DECODE: return "decode_kernel";
    case GDN_K_BWD_CHAIN: return "bwd_state_kernels";
    case GDN_K_BWD_PROLOGUE: return "bwd_prologue_kernel";
    case GDN_K_SEG_SCAN: return "seg_scan_kernels";
    default: return "";
  }
}

}  // extern "C"
