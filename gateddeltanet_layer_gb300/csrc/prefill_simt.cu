// Token-sequential prefill in fp32 on the CUDA cores.
//
// Serves fp32 streams (where a bf16 tensor-core operand would not meet a 1e-4
// tolerance) and every supported shape other than the d = 128 bf16 case.
// Three launches: the per-token inputs once (token_inputs.cuh); then one CTA
// per (sequence, value head, slice of 32 state columns) with the state
// H = S^T (d_k x d_v) in registers: warp w owns columns [2w, 2w+2) of the
// slice, lane l rows l, l+32, l+64, l+96.  Columns of H evolve independently
// under the rule (p_j = H[:,j] . k, u_j = beta (v_j - alpha p_j),
// H[:,j] <- alpha H[:,j] + k u_j), so each warp advances its columns through
// the whole sequence without waiting for the others, writing o of every
// token; the RMSNormGated, which needs whole rows, runs after, one warp per
// (token, value head).
#include "gdn_common.cuh"
#include "../../include/gdn_trace.h"
#include "gdn_internal.h"
#include "token_inputs.cuh"

namespace gdn {
namespace {

constexpr int kTB = 32;      // tokens per batch of copied inputs
constexpr int kCW = 2;       // state columns per warp
constexpr int kColLanes = 32 / kCW;  // a reduce-scatter over the warp leaves column c in lane c kColLanes
constexpr int kRows = 4;     // rows per lane (d_k <= 128)
constexpr int kSliceCols = 32, kSliceWarps = kSliceCols / kCW, kSliceThreads = 32 * kSliceWarps;

// One CTA per (chain, slice of kSliceCols state columns): the rule token by
// token on the slice's columns, o (scaled) of every token to `wo`.  DK: the
// head dim d_k when it is fixed at compile time (128), else 0 (read from p).
template <typename IO, int DK>
__global__ void __launch_bounds__(kSliceThreads, 1) prefill_simt_kernel(PrefillParams p, const TokenInputs ti,
                                                                     float *wo) {
  const int h_v = p.h_v, h_qk = p.h_qk, dk = DK ? DK : p.d_k, dv = p.d_v;
  const int slices = (dv + kSliceCols - 1) / kSliceCols;
  const int sl = blockIdx.x % slices, chain = blockIdx.x / slices;
  const int n = chain / h_v, h = chain % h_v, hq = h / (h_v / h_qk), jsl = kSliceCols * sl;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int s0 = p.cu_seqlens[n], s1 = p.cu_seqlens[n + 1];
  if (s0 < 0 || s1 < s0 || s1 > p.T) {
    if (threadIdx.x == 0) set_status(p.status, kDevBadSeqlens);
    return;
  }

  extern __shared__ __align__(16) float smem[];
  float *sq = smem;                    // [kTB][dk]
  float *sk = sq + kTB * dk;           // [kTB][dk]
  float *sv = sk + kTB * dk;           // [kTB][kSliceCols]
  float *salpha = sv + kTB * kSliceCols;  // [kTB]
  float *sbeta = salpha + kTB;         // [kTB]

  const size_t state_off = ((size_t)n * h_v + h) * dk * dv;
  const int j0 = jsl + warp * kCW;     // this warp's first column
  float H[kRows][kCW];
#pragma unroll
  for (int r = 0; r < kRows; ++r)
#pragma unroll
    for (int c = 0; c < kCW; ++c) {
      const int i = lane + 32 * r, j = j0 + c;
      H[r][c] = (p.init_state && i < dk && j < dv) ? p.init_state[state_off + (size_t)i * dv + j] : 0.0f;
    }
  const float scale = rsqrtf((float)dk);

  for (int t0 = s0; t0 < s1; t0 += kTB) {
    const int nt = min(kTB, s1 - t0);
    __syncthreads();  // the previous batch's buffers are consumed
    // the batch's inputs (q^, k^, the slice's columns of silu(conv(v)), alpha, beta) from the token-inputs
    // pass: float4 copies (head dims and slices are multiples of 16 floats), kU in flight per thread
    {
      const int nq = dk / 4, nv = kSliceCols / 4, per_tok = 2 * nq + nv, total = nt * per_tok;
      const float4 *gq = reinterpret_cast<const float4 *>(ti.xq), *gk = reinterpret_cast<const float4 *>(ti.xk);
      float4 *sq4 = reinterpret_cast<float4 *>(sq), *sk4 = reinterpret_cast<float4 *>(sk);
      float4 *sv4 = reinterpret_cast<float4 *>(sv);
      constexpr int kU = 4;
      for (int base = threadIdx.x; base < total; base += kU * blockDim.x) {
        float4 val[kU];
        float4 *dst[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int idx = base + u * blockDim.x;
          dst[u] = nullptr;
          if (idx < total) {
            const int tt = idx / per_tok, c = idx % per_tok;
            const size_t t = (size_t)(t0 + tt);
            if (c < nq) {
              val[u] = gq[(t * h_qk + hq) * nq + c];
              dst[u] = sq4 + tt * nq + c;
            } else if (c < 2 * nq) {
              val[u] = gk[(t * h_qk + hq) * nq + c - nq];
              dst[u] = sk4 + tt * nq + c - nq;
            } else {
              const int j = jsl + 4 * (c - 2 * nq);
              val[u] = j < dv ? *reinterpret_cast<const float4 *>(ti.xv + (t * h_v + h) * dv + j)
                              : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
              dst[u] = sv4 + tt * nv + c - 2 * nq;
            }
          }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u)
          if (dst[u]) *dst[u] = val[u];
      }
      for (int tt = threadIdx.x; tt < nt; tt += blockDim.x) {
        salpha[tt] = ti.xal[(size_t)(t0 + tt) * h_v + h];
        sbeta[tt] = ti.xbe[(size_t)(t0 + tt) * h_v + h];
      }
    }
    __syncthreads();
    // the rule, token by token, on this warp's columns
    if (j0 < dv) {
      for (int tt = 0; tt < nt; ++tt) {
        float kr[kRows], qr[kRows];
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          const int i = lane + 32 * r;
          kr[r] = i < dk ? sk[tt * dk + i] : 0.0f;
          qr[r] = i < dk ? sq[tt * dk + i] : 0.0f;
        }
        const float al = salpha[tt], be = sbeta[tt];
        float pc[kCW];
#pragma unroll
        for (int c = 0; c < kCW; ++c) {
          float s_ = 0.0f;
#pragma unroll
          for (int r = 0; r < kRows; ++r) s_ = fmaf(H[r][c], kr[r], s_);
          pc[c] = s_;
        }
        {  // the warp's column sums together: reduce-scatter (lane l: column l / kColLanes), then broadcast
          const float ps = reduce_scatter<kCW>(pc, lane);
#pragma unroll
          for (int c = 0; c < kCW; ++c) pc[c] = __shfl_sync(0xffffffffu, ps, kColLanes * c);
        }
        float oc[kCW];
#pragma unroll
        for (int c = 0; c < kCW; ++c) {
          const int jj = warp * kCW + c;  // column within the slice
          const float u = be * (sv[tt * kSliceCols + jj] - al * pc[c]);
          float s_ = 0.0f;
#pragma unroll
          for (int r = 0; r < kRows; ++r) {
            H[r][c] = fmaf(kr[r], u, al * H[r][c]);
            s_ = fmaf(H[r][c], qr[r], s_);
          }
          oc[c] = s_;
        }
        const float os = reduce_scatter<kCW>(oc, lane);  // lane l: column l / kColLanes
        if (lane % kColLanes == 0 && j0 + lane / kColLanes < dv)
          wo[((size_t)(t0 + tt) * h_v + h) * dv + j0 + lane / kColLanes] = os * scale;
      }
    }
  }

  if (p.final_state) {
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
      for (int c = 0; c < kCW; ++c) {
        const int i = lane + 32 * r, j = j0 + c;
        if (i < dk && j < dv) p.final_state[state_off + (size_t)i * dv + j] = H[r][c];
      }
  }
}

// RMSNormGated, one warp per (token, value head) row, from o of every token.
template <typename IO>
__global__ void __launch_bounds__(256) simt_norm_kernel(const PrefillParams p, const float *wo) {
  const size_t row = (size_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31, dv = p.d_v;
  if (row >= (size_t)p.T * p.h_v) return;
  const float *o = wo + row * dv;
  const IO *xz = static_cast<const IO *>(p.z) + row * dv;
  IO *out = static_cast<IO *>(p.out) + row * dv;
  float ss = 0.0f;
  for (int j = lane; j < dv; j += 32) ss = fmaf(o[j], o[j], ss);
  const float inv = rsqrtf(warp_sum(ss) / (float)dv + kEpsRms);
  for (int j = lane; j < dv; j += 32) out[j] = from_f<IO>(o[j] * inv * p.norm_w[j] * silu_f(to_f(xz[j])));
}

}  // namespace

size_t prefill_simt_workspace_bytes(int T, int h_qk, int h_v, int d_k, int d_v) {
  return token_inputs_bytes(T, h_qk, h_v, d_k, d_v) + (size_t)T * h_v * d_v * sizeof(float);
}

cudaError_t launch_prefill_simt(const PrefillParams &p, bool bf16, cudaStream_t s) {
  const int slices = (p.d_v + kSliceCols - 1) / kSliceCols;
  const size_t smem = sizeof(float) * (size_t)(kTB * (2 * p.d_k + kSliceCols) + 2 * kTB);
  const unsigned grid = (unsigned)p.N * (unsigned)p.h_v * (unsigned)slices;
  if (grid == 0) return cudaSuccess;
  if (p.ws_bytes < prefill_simt_workspace_bytes(p.T, p.h_qk, p.h_v, p.d_k, p.d_v)) return cudaErrorInvalidValue;
  TokenInputs ti{};
  ti.q = p.q; ti.k = p.k; ti.v = p.v; ti.a = p.a; ti.b = p.b;
  ti.conv_w = p.conv_w; ti.A_log = p.A_log; ti.dt_bias = p.dt_bias; ti.cu_seqlens = p.cu_seqlens;
  ti.init_conv = p.init_conv;
  ti.T = p.T; ti.N = p.N; ti.h_qk = p.h_qk; ti.h_v = p.h_v; ti.d_k = p.d_k; ti.d_v = p.d_v;
  token_inputs_carve(ti, p.ws);
  float *wo = reinterpret_cast<float *>(p.ws + token_inputs_bytes(p.T, p.h_qk, p.h_v, p.d_k, p.d_v));
  const unsigned irows =
      (unsigned)(((size_t)p.T * (2 * p.h_qk + p.h_v) + kTokenRowsPerCta - 1) / kTokenRowsPerCta);
  const unsigned nrows = (unsigned)(((size_t)p.T * p.h_v + 7) / 8);
  auto run = [&](auto in_k, auto kern128, auto kern, auto norm_k) -> cudaError_t {
    if (p.d_k == 128) kern = kern128;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    trace_begin(s, GDN_K_PREFILL_SIMT);
    if (p.T > 0) in_k<<<irows, 32 * kTokenRowsPerCta, 0, s>>>(ti);
    kern<<<grid, kSliceThreads, smem, s>>>(p, ti, wo);
    if (p.T > 0) norm_k<<<nrows, 256, 0, s>>>(p, wo);
    trace_end(s);
    return cudaGetLastError();
  };
  if (bf16)
    return run(token_inputs_kernel<__nv_bfloat16>, prefill_simt_kernel<__nv_bfloat16, 128>,
               prefill_simt_kernel<__nv_bfloat16, 0>, simt_norm_kernel<__nv_bfloat16>);
  return run(token_inputs_kernel<float>, prefill_simt_kernel<float, 128>, prefill_simt_kernel<float, 0>,
             simt_norm_kernel<float>);
}

}  // namespace gdn
