// Internal launch interface between the C ABI (gdn_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

struct PrefillParams {
  int T, N, h_qk, h_v, d_k, d_v;
  const void *q, *k, *v, *a, *b, *z;
  const float *conv_w, *A_log, *dt_bias, *norm_w;
  const int32_t *cu_seqlens;
  const float *init_state;
  const void *init_conv;  // [N, Cc, 3] io dtype: raw inputs before each sequence start, oldest first; may be null
  void *out;
  float *final_state;
  int *status;       // device status word (workspace), may be null
  uint8_t *ws;       // workspace base (256-byte aligned)
  size_t ws_bytes;
};

struct DecodeParams {
  int B, h_qk, h_v, d_k, d_v;
  const void *q, *k, *v, *a, *b, *z;
  const float *conv_w, *A_log, *dt_bias, *norm_w;
  void *conv_state;
  float *state;
  void *out;
  const int32_t *slots;  // [B] pool entry of each sequence, or null (entry b)
  int num_slots;         // entries in the conv_state / state pools when slots is set
  int *status;           // device status word for out-of-range slots, may be null
};

struct ConvCacheParams {
  int T, N, h_qk, h_v, d_k, d_v;
  const void *q, *k, *v;
  const int32_t *cu_seqlens;
  const void *init_conv; // [N, Cc, 3] history before each sequence start, or null (zeros); may equal conv_cache
  void *conv_cache;      // [N, Cc, 3]
};

// Backward pass of a prefill: the gradient of sum(dy * y) (+ sum(dfinal * final_state)).
struct BwdParams {
  int T, N, h_qk, h_v, d_k, d_v;
  const void *q, *k, *v, *a, *b, *z;
  const void *dy;              // [T, h_v, d_v] io dtype
  const float *conv_w, *A_log, *dt_bias, *norm_w;
  const int32_t *cu_seqlens;
  const float *init_state;     // may be null
  const float *dfinal_state;   // may be null
  float *dq, *dk, *dv, *da, *db, *dz;               // stream gradients (fp32, the streams' layouts)
  float *dconv_w, *dA_log, *ddt_bias, *dnorm_w;     // parameter gradients (fp32)
  float *dinit_state;          // may be null
  int *status;
  uint8_t *ws;
  size_t ws_bytes;
};
cudaError_t launch_prefill_backward(const BwdParams &p, bool bf16, cudaStream_t s);
size_t prefill_backward_workspace_bytes(int T, int N, int h_qk, int h_v, int d_k, int d_v);

// Token-sequential fp32 prefill (any supported shape, bf16 or fp32 streams).
cudaError_t launch_prefill_simt(const PrefillParams &p, bool bf16, cudaStream_t s);
// Its workspace (after the status block): the per-token inputs (fp32), computed once.
size_t prefill_simt_workspace_bytes(int T, int h_qk, int h_v, int d_k, int d_v);
// Chunked tensor-core prefill (bf16 streams, d_k = d_v = 128).  Its chunk
// preparation takes up to kTcMaxRep value heads of a q/k head per CTA (more
// value heads per q/k head: several CTAs, each redoing the q/k part).
constexpr int kTcMaxRep = 8;
cudaError_t launch_prefill_tc(const PrefillParams &p, cudaStream_t s);
size_t prefill_tc_workspace_bytes(int T, int N, int h_qk, int h_v);
// Segment-parallel chunked prefill (the same shapes): every sequence cut into
// segments of `seg` chunks, run in parallel and joined by an affine scan.
cudaError_t launch_prefill_segmented(const PrefillParams &p, int seg, cudaStream_t s);
size_t prefill_segmented_workspace_bytes(int T, int N, int h_qk, int h_v, int seg);
// Decode step.
cudaError_t launch_decode(const DecodeParams &p, bool bf16, cudaStream_t s);
// Conv cache of each sequence after a prefill (its last three raw inputs).
cudaError_t launch_conv_cache(const ConvCacheParams &p, bool bf16, cudaStream_t s);

// Kernel timing trace (gdn_trace.cu): events around one launch on its stream;
// no-ops while tracing is off.  `kind` is a gdn_kernel_kind.
void trace_begin(cudaStream_t s, int kind);
void trace_end(cudaStream_t s);

}  // namespace gdn
