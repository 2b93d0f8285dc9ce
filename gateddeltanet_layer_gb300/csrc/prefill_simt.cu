// Token-sequential prefill in fp32 on the CUDA cores.
//
// Serves fp32 streams (where a bf16 tensor-core operand would not meet a 1e-4
// tolerance) and every supported shape other than the d = 128 bf16 case.
// One CTA per (sequence, value head) chain.  The state H = S^T (d_k x d_v)
// lives in registers: warp w owns columns [4w, 4w+4) of H, lane l owns rows
// l, l+32, l+64, l+96.  Columns of H evolve independently under the rule
// (p_j = H[:,j] . k, u_j = beta (v_j - alpha p_j), H[:,j] <- alpha H[:,j] + k u_j),
// so each warp advances its columns through the whole sequence without
// waiting for the others; only the RMSNormGated epilogue needs every column,
// and it runs once per batch of kTB tokens.
#include "gdn_common.cuh"
#include "../../include/gdn_trace.h"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kTB = 32;      // tokens per prologue/epilogue batch
constexpr int kCW = 4;       // state columns per warp (d_v / 4 warps: up to 1024 threads)
constexpr int kColLanes = 32 / kCW;  // a reduce-scatter over the warp leaves column c in lane c kColLanes
constexpr int kRows = 4;     // rows per lane (d_k <= 128)

template <typename IO>
__global__ void __launch_bounds__(32 * 128 / kCW) prefill_simt_kernel(PrefillParams p) {
  const int h_v = p.h_v, h_qk = p.h_qk, dk = p.d_k, dv = p.d_v;
  const int n = blockIdx.x / h_v;
  const int h = blockIdx.x % h_v;
  const int hq = h / (h_v / h_qk);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;

  const int s0 = p.cu_seqlens[n], s1 = p.cu_seqlens[n + 1];
  if (s0 < 0 || s1 < s0 || s1 > p.T) {
    if (threadIdx.x == 0) set_status(p.status, kDevBadSeqlens);
    return;
  }

  const IO *__restrict__ xq = static_cast<const IO *>(p.q);
  const IO *__restrict__ xk = static_cast<const IO *>(p.k);
  const IO *__restrict__ xv = static_cast<const IO *>(p.v);
  const IO *__restrict__ xa = static_cast<const IO *>(p.a);
  const IO *__restrict__ xb = static_cast<const IO *>(p.b);
  const IO *__restrict__ xz = static_cast<const IO *>(p.z);
  IO *__restrict__ out = static_cast<IO *>(p.out);

  extern __shared__ float smem[];
  float *sq = smem;               // [kTB][dk]
  float *sk = sq + kTB * dk;      // [kTB][dk]
  float *sv = sk + kTB * dk;      // [kTB][dv]
  float *so = sv + kTB * dv;      // [kTB][dv]
  float *salpha = so + kTB * dv;  // [kTB]
  float *sbeta = salpha + kTB;    // [kTB]

  const size_t state_off = ((size_t)n * h_v + h) * dk * dv;
  const int j0 = warp * kCW;
  float H[kRows][kCW];
#pragma unroll
  for (int r = 0; r < kRows; ++r)
#pragma unroll
    for (int c = 0; c < kCW; ++c) {
      const int i = lane + 32 * r, j = j0 + c;
      H[r][c] = (p.init_state && i < dk && j < dv) ? p.init_state[state_off + (size_t)i * dv + j] : 0.0f;
    }

  const float A_exp = expf(p.A_log[h]);
  const float dtb = p.dt_bias[h];
  const float scale = rsqrtf((float)dk);
  const int nch = 2 * dk + dv;
  const int Cc = 2 * h_qk * dk + h_v * dv;
  const IO *__restrict__ hist = static_cast<const IO *>(p.init_conv);  // conv history, or null (zeros)

  for (int t0 = s0; t0 < s1; t0 += kTB) {
    const int nt = min(kTB, s1 - t0);
    __syncthreads();  // the previous batch's buffers are consumed
    // conv (width 4; before s0 the carried history, or zeros) + SiLU: kU elements per thread at a time,
    // their 4 kU input loads issued before any is used
    constexpr int kU = 2;
    for (int base = threadIdx.x; base < nt * nch; base += kU * blockDim.x) {
      float xin[kU][4], w[kU][4];
      float *dst[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int idx = base + u * blockDim.x;
        dst[u] = nullptr;
#pragma unroll
        for (int j = 0; j < 4; ++j) xin[u][j] = w[u][j] = 0.0f;
        if (idx < nt * nch) {
          const int tt = idx / nch, c = idx % nch;
          const int t = t0 + tt;
          const IO *src;
          size_t stride;
          int ch;
          if (c < dk) {
            src = xq + hq * dk + c; stride = (size_t)h_qk * dk; ch = hq * dk + c; dst[u] = sq + tt * dk + c;
          } else if (c < 2 * dk) {
            const int cc = c - dk;
            src = xk + hq * dk + cc; stride = (size_t)h_qk * dk; ch = h_qk * dk + hq * dk + cc;
            dst[u] = sk + tt * dk + cc;
          } else {
            const int cc = c - 2 * dk;
            src = xv + h * dv + cc; stride = (size_t)h_v * dv; ch = 2 * h_qk * dk + h * dv + cc;
            dst[u] = sv + tt * dv + cc;
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int tau = t - 3 + j;
            w[u][j] = p.conv_w[ch * 4 + j];
            if (tau >= s0)
              xin[u][j] = to_f(src[(size_t)tau * stride]);
            else if (hist)  // the carried input of token tau = s0 - 3 + m sits at m (oldest first)
              xin[u][j] = to_f(hist[((size_t)n * Cc + ch) * 3 + (tau - s0 + 3)]);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (dst[u]) {
          float pre = 0.0f;  // a tap with no input (before s0, no history) adds w * 0
#pragma unroll
          for (int j = 0; j < 4; ++j) pre = fmaf(w[u][j], xin[u][j], pre);
          *dst[u] = silu_f(pre);
        }
    }
    for (int tt = threadIdx.x; tt < nt; tt += blockDim.x) {
      const size_t t = (size_t)(t0 + tt);
      salpha[tt] = expf(gate_g(to_f(xa[t * h_v + h]), A_exp, dtb));
      sbeta[tt] = sigmoid_f(to_f(xb[t * h_v + h]));
    }
    __syncthreads();
    // L2-normalise the q and k rows (one warp per row)
    for (int row = warp; row < 2 * nt; row += nwarps) {
      float *x = row < nt ? sq + row * dk : sk + (row - nt) * dk;
      float ss = 0.0f;
      for (int i = lane; i < dk; i += 32) ss = fmaf(x[i], x[i], ss);
      const float inv = rsqrtf(warp_sum(ss) + kEpsL2);
      for (int i = lane; i < dk; i += 32) x[i] *= inv;
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
          float s = 0.0f;
#pragma unroll
          for (int r = 0; r < kRows; ++r) s = fmaf(H[r][c], kr[r], s);
          pc[c] = s;
        }
        {  // the warp's column sums together: reduce-scatter (lane l: column l / kColLanes), then broadcast
          const float ps = reduce_scatter<kCW>(pc, lane);
#pragma unroll
          for (int c = 0; c < kCW; ++c) pc[c] = __shfl_sync(0xffffffffu, ps, kColLanes * c);
        }
        float oc[kCW];
#pragma unroll
        for (int c = 0; c < kCW; ++c) {
          const int j = j0 + c;
          const float u = be * ((j < dv ? sv[tt * dv + j] : 0.0f) - al * pc[c]);
          float s = 0.0f;
#pragma unroll
          for (int r = 0; r < kRows; ++r) {
            H[r][c] = fmaf(kr[r], u, al * H[r][c]);
            s = fmaf(H[r][c], qr[r], s);
          }
          oc[c] = s;
        }
        const float os = reduce_scatter<kCW>(oc, lane);  // lane l: column l / kColLanes
        if (lane % kColLanes == 0 && j0 + lane / kColLanes < dv) so[tt * dv + j0 + lane / kColLanes] = os * scale;
      }
    }
    __syncthreads();
    // RMSNormGated epilogue (one warp per token)
    for (int tt = warp; tt < nt; tt += nwarps) {
      float ss = 0.0f;
      for (int j = lane; j < dv; j += 32) ss = fmaf(so[tt * dv + j], so[tt * dv + j], ss);
      const float inv = rsqrtf(warp_sum(ss) / (float)dv + kEpsRms);
      const size_t row = ((size_t)(t0 + tt) * h_v + h) * dv;
      for (int j = lane; j < dv; j += 32) {
        const float y = so[tt * dv + j] * inv * p.norm_w[j] * silu_f(to_f(xz[row + j]));
        out[row + j] = from_f<IO>(y);
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

}  // namespace

cudaError_t launch_prefill_simt(const PrefillParams &p, bool bf16, cudaStream_t s) {
  const int warps = (p.d_v + kCW - 1) / kCW;
  const int threads = 32 * warps;
  const size_t smem = sizeof(float) * (size_t)(kTB * (2 * p.d_k + 2 * p.d_v) + 2 * kTB);
  const unsigned grid = (unsigned)p.N * (unsigned)p.h_v;
  if (grid == 0) return cudaSuccess;
  if (bf16) {
    auto kern = prefill_simt_kernel<__nv_bfloat16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    trace_begin(s, GDN_K_PREFILL_SIMT);
    kern<<<grid, threads, smem, s>>>(p);
    trace_end(s);
  } else {
    auto kern = prefill_simt_kernel<float>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    trace_begin(s, GDN_K_PREFILL_SIMT);
    kern<<<grid, threads, smem, s>>>(p);
    trace_end(s);
  }
  return cudaGetLastError();
}

}  // namespace gdn
