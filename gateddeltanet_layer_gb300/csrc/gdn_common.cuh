// Shared device helpers of the GatedDeltaNet kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

// ----------------------------------------------------------------- I/O types
template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// ----------------------------------------------------------------- scalar math
// Gates and activations of the layer, in fp32 with CUDA's libm functions.
__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + expf(-x)); }
__device__ __forceinline__ float silu_f(float x) { return x * sigmoid_f(x); }
// softplus(x) = log(1 + e^x); above 20 it equals x to within e^-20 relative.
__device__ __forceinline__ float softplus_f(float x) { return x > 20.0f ? x : log1pf(expf(x)); }
// g = -exp(A_log) * softplus(a + dt_bias)
__device__ __forceinline__ float gate_g(float a, float A_log_exp, float dt_bias) {
  return -A_log_exp * softplus_f(a + dt_bias);
}

constexpr float kEpsL2 = 1e-6f;
constexpr float kEpsRms = 1e-6f;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum over the 32 lanes of the warp of each of the NV values v[i] (NV a power
// of two <= 32): lane l returns the sum for i = l >> (5 - log2 NV).
template <int NV>
__device__ __forceinline__ float reduce_scatter(float (&v)[NV], int lane) {
#pragma unroll
  for (int st = 0; st < 5; ++st) {
    const int off = 16 >> st;
    const int half = (NV >> st) >> 1;  // values kept after this stage (0: plain butterfly)
    if (half > 0) {
      const bool upper = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < half; ++i) {
        const float send = upper ? v[i] : v[i + half];
        const float keep = upper ? v[i + half] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
      }
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
    }
  }
  return v[0];
}

// ----------------------------------------------------------------- device status
// First error wins; 0 = OK.  Codes are the public gdn_status values.
enum : int { kDevOk = 0, kDevBadSeqlens = 5, kDevTimeout = 6 };
__device__ __forceinline__ void set_status(int *st, int code) {
  if (st) atomicCAS(st, 0, code);
}

}  // namespace gdn
