// C ABI of the GatedDeltaNet layer library: argument validation and dispatch.
// Everything here runs on the host and only enqueues work; the layer itself
// is computed by the kernels in this directory.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdn.h"
#include "gdn_internal.h"

namespace {

constexpr size_t kStatusBytes = 256;  // status word, padded to keep what follows aligned

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool head_dim_ok(int d) { return d >= 16 && d <= 128 && d % 16 == 0; }

// Checks shared by prefill and decode.  Returns GDN_OK or a status.
int check_dims(const gdn_dims *d) {
  if (!d) return GDN_ERR_INVALID_ARG;
  if (d->num_tokens < 0 || d->h_qk <= 0 || d->h_v <= 0 || d->d_k <= 0 || d->d_v <= 0)
    return GDN_ERR_INVALID_ARG;
  if (d->h_v % d->h_qk != 0) return GDN_ERR_INVALID_ARG;
  if (d->io_dtype != GDN_BF16 && d->io_dtype != GDN_FP32) return GDN_ERR_INVALID_ARG;
  if (!head_dim_ok(d->d_k) || !head_dim_ok(d->d_v)) return GDN_ERR_UNSUPPORTED;
  return GDN_OK;
}

bool use_tensor_core_prefill(const gdn_dims *d) {
  return d->io_dtype == GDN_BF16 && d->d_k == 128 && d->d_v == 128;
}

}  // namespace

extern "C" {

size_t gdn_prefill_workspace_bytes(const gdn_dims *d) {
  if (check_dims(d) != GDN_OK || d->num_seqs <= 0) return 0;
  size_t bytes = kStatusBytes;
  if (use_tensor_core_prefill(d))
    bytes += gdn::prefill_tc_workspace_bytes(d->num_tokens, d->num_seqs, d->h_qk, d->h_v);
  else
    bytes += gdn::prefill_simt_workspace_bytes(d->num_tokens, d->h_qk, d->h_v, d->d_k, d->d_v);
  return bytes;
}

size_t gdn_prefill_segmented_workspace_bytes(const gdn_dims *d, int seg_chunks) {
  if (check_dims(d) != GDN_OK || d->num_seqs <= 0 || seg_chunks < 1 || !use_tensor_core_prefill(d)) return 0;
  return kStatusBytes +
         gdn::prefill_segmented_workspace_bytes(d->num_tokens, d->num_seqs, d->h_qk, d->h_v, seg_chunks);
}

}  // extern "C"

namespace {

// gdn_prefill, gdn_prefill_carry and gdn_prefill_segmented (seg > 0):
// validation, workspace, the kernels, and (when final_conv is given) the conv
// cache the call leaves.
int prefill_impl(const gdn_dims *d, const void *q, const void *k, const void *v, const void *a, const void *b,
                 const void *z, const float *conv_w, const float *A_log, const float *dt_bias,
                 const float *norm_w, const int32_t *cu_seqlens, const float *init_state, const void *init_conv,
                 void *out, float *final_state, void *final_conv, void *workspace, size_t ws_bytes,
                 void *stream, int seg = 0) {
  int st = check_dims(d);
  if (st != GDN_OK) return st;
  if (d->num_seqs <= 0 || seg < 0) return GDN_ERR_INVALID_ARG;
  if (seg > 0 && !use_tensor_core_prefill(d)) return GDN_ERR_UNSUPPORTED;
  if (!conv_w || !A_log || !dt_bias || !norm_w || !cu_seqlens) return GDN_ERR_INVALID_ARG;
  if (d->num_tokens > 0 && (!q || !k || !v || !a || !b || !z || !out)) return GDN_ERR_INVALID_ARG;
  const void *streams[] = {q, k, v, a, b, z, out, init_state, final_state, conv_w};
  for (const void *p : streams)
    if (p && !aligned16(p)) return GDN_ERR_INVALID_ARG;
  const size_t need = seg > 0 ? gdn_prefill_segmented_workspace_bytes(d, seg) : gdn_prefill_workspace_bytes(d);
  if (workspace && (ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
    return GDN_ERR_WORKSPACE;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void *ws = workspace;
  bool owned = false;
  if (!ws) {
    if (cudaMallocAsync(&ws, need, s) != cudaSuccess) return GDN_ERR_CUDA;
    owned = true;
  }
  if (cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) {
    if (owned) cudaFreeAsync(ws, s);
    return GDN_ERR_CUDA;
  }

  gdn::PrefillParams p{};
  p.T = d->num_tokens; p.N = d->num_seqs; p.h_qk = d->h_qk; p.h_v = d->h_v;
  p.d_k = d->d_k; p.d_v = d->d_v;
  p.q = q; p.k = k; p.v = v; p.a = a; p.b = b; p.z = z;
  p.conv_w = conv_w; p.A_log = A_log; p.dt_bias = dt_bias; p.norm_w = norm_w;
  p.cu_seqlens = cu_seqlens; p.init_state = init_state; p.init_conv = init_conv;
  p.out = out; p.final_state = final_state;
  p.status = static_cast<int *>(ws);
  p.ws = static_cast<uint8_t *>(ws) + kStatusBytes;
  p.ws_bytes = need - kStatusBytes;

  cudaError_t e;
  if (seg > 0)
    e = gdn::launch_prefill_segmented(p, seg, s);
  else if (use_tensor_core_prefill(d))
    e = gdn::launch_prefill_tc(p, s);
  else
    e = gdn::launch_prefill_simt(p, d->io_dtype == GDN_BF16, s);
  if (e == cudaSuccess && final_conv) {  // after every kernel that reads init_conv (stream order)
    gdn::ConvCacheParams c{};
    c.T = d->num_tokens; c.N = d->num_seqs; c.h_qk = d->h_qk; c.h_v = d->h_v; c.d_k = d->d_k; c.d_v = d->d_v;
    c.q = q; c.k = k; c.v = v; c.cu_seqlens = cu_seqlens; c.init_conv = init_conv; c.conv_cache = final_conv;
    e = gdn::launch_conv_cache(c, d->io_dtype == GDN_BF16, s);
  }
  if (owned) cudaFreeAsync(ws, s);
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

extern "C" {

int gdn_prefill(const gdn_dims *d, const void *q, const void *k, const void *v, const void *a,
                const void *b, const void *z, const float *conv_w, const float *A_log,
                const float *dt_bias, const float *norm_w, const int32_t *cu_seqlens,
                const float *init_state, void *out, float *final_state, void *workspace,
                size_t ws_bytes, void *stream) {
  return prefill_impl(d, q, k, v, a, b, z, conv_w, A_log, dt_bias, norm_w, cu_seqlens, init_state, nullptr, out,
                      final_state, nullptr, workspace, ws_bytes, stream);
}

int gdn_prefill_carry(const gdn_dims *d, const void *q, const void *k, const void *v, const void *a,
                      const void *b, const void *z, const float *conv_w, const float *A_log,
                      const float *dt_bias, const float *norm_w, const int32_t *cu_seqlens,
                      const float *init_state, const void *init_conv, void *out, float *final_state,
                      void *final_conv, void *workspace, size_t ws_bytes, void *stream) {
  return prefill_impl(d, q, k, v, a, b, z, conv_w, A_log, dt_bias, norm_w, cu_seqlens, init_state, init_conv, out,
                      final_state, final_conv, workspace, ws_bytes, stream);
}

int gdn_prefill_segmented(const gdn_dims *d, const void *q, const void *k, const void *v, const void *a,
                          const void *b, const void *z, const float *conv_w, const float *A_log,
                          const float *dt_bias, const float *norm_w, const int32_t *cu_seqlens,
                          const float *init_state, void *out, float *final_state, int seg_chunks, void *workspace,
                          size_t ws_bytes, void *stream) {
  if (seg_chunks < 1) return GDN_ERR_INVALID_ARG;
  return prefill_impl(d, q, k, v, a, b, z, conv_w, A_log, dt_bias, norm_w, cu_seqlens, init_state, nullptr, out,
                      final_state, nullptr, workspace, ws_bytes, stream, seg_chunks);
}

size_t gdn_prefill_backward_workspace_bytes(const gdn_dims *d) {
  if (check_dims(d) != GDN_OK || d->num_seqs <= 0) return 0;
  return kStatusBytes +
         gdn::prefill_backward_workspace_bytes(d->num_tokens, d->num_seqs, d->h_qk, d->h_v, d->d_k, d->d_v);
}

int gdn_prefill_backward(const gdn_dims *d, const void *q, const void *k, const void *v, const void *a,
                         const void *b, const void *z, const float *conv_w, const float *A_log,
                         const float *dt_bias, const float *norm_w, const int32_t *cu_seqlens,
                         const float *init_state, const void *dy, const float *dfinal_state, float *dq, float *dk,
                         float *dv, float *da, float *db, float *dz, float *dconv_w, float *dA_log,
                         float *ddt_bias, float *dnorm_w, float *dinit_state, void *workspace, size_t ws_bytes,
                         void *stream) {
  int st = check_dims(d);
  if (st != GDN_OK) return st;
  if (d->num_seqs <= 0) return GDN_ERR_INVALID_ARG;
  if (!conv_w || !A_log || !dt_bias || !norm_w || !cu_seqlens || !dconv_w || !dA_log || !ddt_bias || !dnorm_w)
    return GDN_ERR_INVALID_ARG;
  if (d->num_tokens > 0 &&
      (!q || !k || !v || !a || !b || !z || !dy || !dq || !dk || !dv || !da || !db || !dz))
    return GDN_ERR_INVALID_ARG;
  const void *ptrs[] = {q, k, v, a, b, z, dy, init_state, dfinal_state, dq, dk, dv, dz, dinit_state, conv_w};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return GDN_ERR_INVALID_ARG;
  const size_t need = gdn_prefill_backward_workspace_bytes(d);
  if (workspace && (ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
    return GDN_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void *ws = workspace;
  bool owned = false;
  if (!ws) {
    if (cudaMallocAsync(&ws, need, s) != cudaSuccess) return GDN_ERR_CUDA;
    owned = true;
  }
  if (cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) {
    if (owned) cudaFreeAsync(ws, s);
    return GDN_ERR_CUDA;
  }
  gdn::BwdParams p{};
  p.T = d->num_tokens; p.N = d->num_seqs; p.h_qk = d->h_qk; p.h_v = d->h_v; p.d_k = d->d_k; p.d_v = d->d_v;
  p.q = q; p.k = k; p.v = v; p.a = a; p.b = b; p.z = z; p.dy = dy;
  p.conv_w = conv_w; p.A_log = A_log; p.dt_bias = dt_bias; p.norm_w = norm_w;
  p.cu_seqlens = cu_seqlens; p.init_state = init_state; p.dfinal_state = dfinal_state;
  p.dq = dq; p.dk = dk; p.dv = dv; p.da = da; p.db = db; p.dz = dz;
  p.dconv_w = dconv_w; p.dA_log = dA_log; p.ddt_bias = ddt_bias; p.dnorm_w = dnorm_w; p.dinit_state = dinit_state;
  p.status = static_cast<int *>(ws);
  p.ws = static_cast<uint8_t *>(ws) + kStatusBytes;
  p.ws_bytes = need - kStatusBytes;
  cudaError_t e = gdn::launch_prefill_backward(p, d->io_dtype == GDN_BF16, s);
  if (owned) cudaFreeAsync(ws, s);
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int gdn_decode_step(const gdn_dims *d, const void *q, const void *k, const void *v, const void *a,
                    const void *b, const void *z, const float *conv_w, const float *A_log,
                    const float *dt_bias, const float *norm_w, void *conv_state, float *state,
                    void *out, void *stream) {
  return gdn_decode_step_slots(d, q, k, v, a, b, z, conv_w, A_log, dt_bias, norm_w, conv_state, state, nullptr, 0,
                               out, nullptr, stream);
}

int gdn_decode_step_slots(const gdn_dims *d, const void *q, const void *k, const void *v, const void *a,
                          const void *b, const void *z, const float *conv_w, const float *A_log,
                          const float *dt_bias, const float *norm_w, void *conv_state, float *state,
                          const int32_t *slots, int num_slots, void *out, int *device_status, void *stream) {
  if (slots && num_slots <= 0) return GDN_ERR_INVALID_ARG;
  int st = check_dims(d);
  if (st != GDN_OK) return st;
  if (!conv_w || !A_log || !dt_bias || !norm_w) return GDN_ERR_INVALID_ARG;
  if (d->num_tokens > 0 && (!q || !k || !v || !a || !b || !z || !out || !conv_state || !state))
    return GDN_ERR_INVALID_ARG;
  const void *ptrs[] = {q, k, v, a, b, z, out, state, conv_w};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return GDN_ERR_INVALID_ARG;
  gdn::DecodeParams p{};
  p.B = d->num_tokens; p.h_qk = d->h_qk; p.h_v = d->h_v; p.d_k = d->d_k; p.d_v = d->d_v;
  p.q = q; p.k = k; p.v = v; p.a = a; p.b = b; p.z = z;
  p.conv_w = conv_w; p.A_log = A_log; p.dt_bias = dt_bias; p.norm_w = norm_w;
  p.conv_state = conv_state; p.state = state; p.out = out;
  p.slots = slots; p.num_slots = num_slots; p.status = device_status;
  cudaError_t e = gdn::launch_decode(p, d->io_dtype == GDN_BF16, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int gdn_conv_cache_from_prefill(const gdn_dims *d, const void *q, const void *k, const void *v,
                                const int32_t *cu_seqlens, void *conv_cache, void *stream) {
  int st = check_dims(d);
  if (st != GDN_OK) return st;
  if (d->num_seqs <= 0 || !cu_seqlens || !conv_cache) return GDN_ERR_INVALID_ARG;
  if (d->num_tokens > 0 && (!q || !k || !v)) return GDN_ERR_INVALID_ARG;
  gdn::ConvCacheParams p{};
  p.T = d->num_tokens; p.N = d->num_seqs; p.h_qk = d->h_qk; p.h_v = d->h_v; p.d_k = d->d_k; p.d_v = d->d_v;
  p.q = q; p.k = k; p.v = v; p.cu_seqlens = cu_seqlens; p.conv_cache = conv_cache;
  cudaError_t e = gdn::launch_conv_cache(p, d->io_dtype == GDN_BF16, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int gdn_workspace_status(void *workspace, void *stream, int *device_status) {
  if (!workspace || !device_status) return GDN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int host = 0;
  if (cudaMemcpyAsync(&host, workspace, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return GDN_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof(int), s) != cudaSuccess) return GDN_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_CUDA;
  *device_status = host;
  return GDN_OK;
}

const char *gdn_status_string(int status) {
  switch (status) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG: invalid argument";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: unsupported shape or dtype";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE: workspace too small or misaligned";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA: CUDA runtime or launch failure";
    case GDN_ERR_DEVICE_CHECK: return "GDN_ERR_DEVICE_CHECK: device-side validation failed (cu_seqlens)";
    case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT: a bounded device wait ran out";
    default: return "GDN_ERR_UNKNOWN";
  }
}

}  // extern "C"
