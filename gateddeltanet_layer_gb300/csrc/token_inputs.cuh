// The recurrence's per-token inputs, computed once per token for every kernel
// that runs the rule token by token on the CUDA cores (the fp32 prefill and
// the backward): q^ and k^ (depthwise conv(4) over the sequence's own tokens,
// or the carried conv history before its first token, SiLU, L2 norm),
// silu(conv(v)), alpha = e^g and beta, in fp32.
#pragma once

#include "gdn_common.cuh"

namespace gdn {

// Sequence n of token t and its range [s0, s1) (binary search over cu_seqlens;
// an empty sequence never holds a token).
struct SeqOf {
  int n, s0, s1;
};
__device__ __forceinline__ SeqOf seq_of(const int32_t *cu, int N, int t) {
  int lo = 0, hi = N - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return SeqOf{lo, cu[lo], cu[lo + 1]};
}

struct TokenInputs {
  const void *q, *k, *v, *a, *b;  // the streams (IO)
  const float *conv_w, *A_log, *dt_bias;
  const int32_t *cu_seqlens;
  const void *init_conv;  // [N][Cc][3] IO, raw inputs of the three tokens before each sequence; or null
  int T, N, h_qk, h_v, d_k, d_v;
  float *xq, *xk;         // [T][h_qk][d_k]
  float *xv;              // [T][h_v][d_v]
  float *xal, *xbe;       // [T][h_v]
};

// One warp per (token, row): row y < h_qk is q head y, then the k heads, then
// the value heads (which also write alpha and beta); lane l takes channels
// l, l + 32, ... (head dims up to 128).  256 threads: 8 rows per CTA.
constexpr int kTokenRowsPerCta = 8;
template <typename IO>
__global__ void __launch_bounds__(32 * kTokenRowsPerCta) token_inputs_kernel(const TokenInputs p) {
  const int h_v = p.h_v, h_qk = p.h_qk, dk = p.d_k, dv = p.d_v, rows = 2 * h_qk + h_v;
  const int Cc = 2 * h_qk * dk + h_v * dv;
  const size_t row = (size_t)blockIdx.x * kTokenRowsPerCta + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= (size_t)p.T * rows) return;
  const int t = (int)(row / rows), y = (int)(row % rows);
  const SeqOf sq = seq_of(p.cu_seqlens, p.N, t);
  const IO *hist = static_cast<const IO *>(p.init_conv);
  const IO *src;
  size_t stride;
  int cb, D;
  float *dst;
  if (y < 2 * h_qk) {
    const int hq = y < h_qk ? y : y - h_qk;
    src = static_cast<const IO *>(y < h_qk ? p.q : p.k) + hq * dk;
    stride = (size_t)h_qk * dk;
    cb = y * dk;  // conv channels: [q heads | k heads | v heads]
    D = dk;
    dst = (y < h_qk ? p.xq : p.xk) + ((size_t)t * h_qk + hq) * dk;
  } else {
    const int hv = y - 2 * h_qk;
    src = static_cast<const IO *>(p.v) + hv * dv;
    stride = (size_t)h_v * dv;
    cb = 2 * h_qk * dk + hv * dv;
    D = dv;
    dst = p.xv + ((size_t)t * h_v + hv) * dv;
    if (lane == 0) {
      const size_t gi = (size_t)t * h_v + hv;
      p.xal[gi] = expf(gate_g(to_f(static_cast<const IO *>(p.a)[gi]), expf(p.A_log[hv]), p.dt_bias[hv]));
      p.xbe[gi] = sigmoid_f(to_f(static_cast<const IO *>(p.b)[gi]));
    }
  }
  float x[4];
  float ss = 0.0f;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int c = lane + 32 * r;
    float pre = 0.0f;
    if (c < D) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int tau = t - 3 + j;
        const float w = p.conv_w[(size_t)(cb + c) * 4 + j];
        if (tau >= sq.s0)
          pre = fmaf(w, to_f(src[(size_t)tau * stride + c]), pre);
        else if (hist)  // the carried input of token tau = s0 - 3 + m sits at m (oldest first)
          pre = fmaf(w, to_f(hist[((size_t)sq.n * Cc + cb + c) * 3 + (tau - sq.s0 + 3)]), pre);
      }
    }
    x[r] = c < D ? silu_f(pre) : 0.0f;
    ss = fmaf(x[r], x[r], ss);
  }
  const float inv = y < 2 * h_qk ? rsqrtf(warp_sum(ss) + kEpsL2) : 1.0f;
#pragma unroll
  for (int r = 0; r < 4; ++r)
    if (lane + 32 * r < D) dst[lane + 32 * r] = x[r] * inv;
}

// Bytes of the arrays token_inputs_kernel writes (each array 256-byte aligned).
inline size_t token_inputs_bytes(int T, int h_qk, int h_v, int d_k, int d_v) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  return 2 * up((size_t)T * h_qk * d_k * 4) + up((size_t)T * h_v * d_v * 4) + 2 * up((size_t)T * h_v * 4);
}
// Carve the arrays out of `base` (256-byte aligned).
inline void token_inputs_carve(TokenInputs &ti, uint8_t *base) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  ti.xq = reinterpret_cast<float *>(base);
  base += up((size_t)ti.T * ti.h_qk * ti.d_k * 4);
  ti.xk = reinterpret_cast<float *>(base);
  base += up((size_t)ti.T * ti.h_qk * ti.d_k * 4);
  ti.xv = reinterpret_cast<float *>(base);
  base += up((size_t)ti.T * ti.h_v * ti.d_v * 4);
  ti.xal = reinterpret_cast<float *>(base);
  base += up((size_t)ti.T * ti.h_v * 4);
  ti.xbe = reinterpret_cast<float *>(base);
}

}  // namespace gdn
