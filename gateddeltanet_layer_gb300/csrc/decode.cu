// Decode step: one token per sequence against a carried fp32 state.
//
// The step is a pure stream over the state (4 MiB read + 4 MiB written per
// 32-head sequence at d = 128): per value head it needs p = H^T k and
// s = H^T q from one read pass, then u = beta (v - alpha p),
// o = scale (alpha s + (k . q) u) (equal to (alpha H + k u^T)^T q * scale), and
// writes H <- alpha H + k u^T back in place.
//
// One CTA per (sequence, query/key head): the CTA owns the conv-cache channels
// of that q/k head and of its h_v / h_qk value heads, so no two CTAs touch
// the same cache entry.  Thread layout per value head: warp w owns rows
// [w*R, (w+1)*R) of H (R = d_k / 8), lane l owns columns [4l, 4l+4); each
// thread keeps its R x 4 block in registers between the read and the write.
#include "gdn_common.cuh"
#include "../../include/gdn_trace.h"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxRows = 16;  // d_k / kWarps for d_k <= 128

// D: the head dims when both are fixed at compile time (128), else 0 (read from p).
template <typename IO, int D>
__global__ void __launch_bounds__(kThreads) decode_kernel(DecodeParams p) {
  const int h_qk = p.h_qk, h_v = p.h_v, dk = D ? D : p.d_k, dv = D ? D : p.d_v;
  const int rep = h_v / h_qk;
  const int b = blockIdx.x / h_qk;
  const int hq = blockIdx.x % h_qk;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Cc = 2 * h_qk * dk + h_v * dv;
  // pool entry of this sequence's state and conv cache
  const int sb = p.slots ? p.slots[b] : b;
  if (p.slots && (sb < 0 || sb >= p.num_slots)) {  // no pool access: zero output, report
    IO *o = static_cast<IO *>(p.out);
    for (int j = tid; j < (h_v / h_qk) * dv; j += kThreads)
      o[((size_t)b * h_v + hq * (h_v / h_qk)) * dv + j] = from_f<IO>(0.0f);
    if (tid == 0 && p.status) set_status(p.status, kDevBadSeqlens);
    return;
  }

  const IO *__restrict__ xq = static_cast<const IO *>(p.q);
  const IO *__restrict__ xk = static_cast<const IO *>(p.k);
  const IO *__restrict__ xv = static_cast<const IO *>(p.v);
  const IO *__restrict__ xa = static_cast<const IO *>(p.a);
  const IO *__restrict__ xb = static_cast<const IO *>(p.b);
  const IO *__restrict__ xz = static_cast<const IO *>(p.z);
  IO *__restrict__ cache = static_cast<IO *>(p.conv_state);
  IO *__restrict__ out = static_cast<IO *>(p.out);

  // per value head, two buffers by head parity: a head's buffer is written only after every thread has
  // passed the previous head's second barrier, so every read of it two heads back is done (no barrier
  // at the end of a head)
  __shared__ float sq[128], sk[128];
  __shared__ float sv[2][128], su[2][128];
  __shared__ float red_p[2][kWarps][128], red_s[2][kWarps][128];
  __shared__ float sred[2][kWarps];
  __shared__ float s_kq, s_alpha[2], s_beta[2];

  // conv with the cache + SiLU for the q and k channels of this head
  for (int c = tid; c < 2 * dk; c += kThreads) {
    const bool isq = c < dk;
    const int i = isq ? c : c - dk;
    const int ch = (isq ? 0 : h_qk * dk) + hq * dk + i;
    const float x = to_f((isq ? xq : xk)[((size_t)b * h_qk + hq) * dk + i]);
    IO *cc = cache + ((size_t)sb * Cc + ch) * 3;
    const float c0 = to_f(cc[0]), c1 = to_f(cc[1]), c2 = to_f(cc[2]);
    const float *w = p.conv_w + (size_t)ch * 4;
    const float pre = fmaf(w[0], c0, fmaf(w[1], c1, fmaf(w[2], c2, w[3] * x)));
    cc[0] = cc[1];
    cc[1] = cc[2];
    cc[2] = (isq ? xq : xk)[((size_t)b * h_qk + hq) * dk + i];
    (isq ? sq : sk)[i] = silu_f(pre);
  }
  __syncthreads();
  // L2 norms of q, k and their dot product
  if (warp < 2) {
    float *x = warp == 0 ? sq : sk;
    float ss = 0.0f;
    for (int i = lane; i < dk; i += 32) ss = fmaf(x[i], x[i], ss);
    const float inv = rsqrtf(warp_sum(ss) + kEpsL2);
    for (int i = lane; i < dk; i += 32) x[i] *= inv;
  }
  __syncthreads();
  if (warp == 0) {
    float s = 0.0f;
    for (int i = lane; i < dk; i += 32) s = fmaf(sq[i], sk[i], s);
    s = warp_sum(s);
    if (lane == 0) s_kq = s;
  }

  const int rows = (dk + kWarps - 1) / kWarps;
  const int i0 = warp * rows;
  const int j0 = lane * 4;
  const bool col_ok = j0 < dv;
  const float scale = rsqrtf((float)dk);

  for (int vv = 0; vv < rep; ++vv) {
    const int h = hq * rep + vv, bf = vv & 1;
    float *Hg = p.state + ((size_t)sb * h_v + h) * dk * dv;
    // issue the state loads first: they are the stream this kernel exists for
    float4 Hr[kMaxRows];
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
      const int i = i0 + r;
      Hr[r] = (r < rows && i < dk && col_ok) ? *reinterpret_cast<const float4 *>(Hg + (size_t)i * dv + j0)
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // conv + SiLU of this head's v channels; gates
    for (int j = tid; j < dv; j += kThreads) {
      const int ch = 2 * h_qk * dk + h * dv + j;
      const size_t xi = ((size_t)b * h_v + h) * dv + j;
      const float x = to_f(xv[xi]);
      IO *cc = cache + ((size_t)sb * Cc + ch) * 3;
      const float c0 = to_f(cc[0]), c1 = to_f(cc[1]), c2 = to_f(cc[2]);
      const float *w = p.conv_w + (size_t)ch * 4;
      const float pre = fmaf(w[0], c0, fmaf(w[1], c1, fmaf(w[2], c2, w[3] * x)));
      cc[0] = cc[1];
      cc[1] = cc[2];
      cc[2] = xv[xi];
      sv[bf][j] = silu_f(pre);
    }
    if (tid == 0) {
      const size_t gi = (size_t)b * h_v + h;
      s_alpha[bf] = expf(gate_g(to_f(xa[gi]), expf(p.A_log[h]), p.dt_bias[h]));
      s_beta[bf] = sigmoid_f(to_f(xb[gi]));
    }
    // partial H^T k and H^T q over this warp's rows (sv, alpha and beta are read after the next barrier)
    float pk[4] = {0.f, 0.f, 0.f, 0.f}, pq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
      if (r < rows && i0 + r < dk) {
        const float kv = sk[i0 + r], qv = sq[i0 + r];
        pk[0] = fmaf(Hr[r].x, kv, pk[0]); pk[1] = fmaf(Hr[r].y, kv, pk[1]);
        pk[2] = fmaf(Hr[r].z, kv, pk[2]); pk[3] = fmaf(Hr[r].w, kv, pk[3]);
        pq[0] = fmaf(Hr[r].x, qv, pq[0]); pq[1] = fmaf(Hr[r].y, qv, pq[1]);
        pq[2] = fmaf(Hr[r].z, qv, pq[2]); pq[3] = fmaf(Hr[r].w, qv, pq[3]);
      }
    }
    if (col_ok) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        red_p[bf][warp][j0 + c] = pk[c];
        red_s[bf][warp][j0 + c] = pq[c];
      }
    }
    __syncthreads();
    const float al = s_alpha[bf], be = s_beta[bf];
    float o_j = 0.0f;
    if (tid < dv) {
      float pj = 0.f, sj = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        pj += red_p[bf][w][tid];
        sj += red_s[bf][w][tid];
      }
      const float u = be * (sv[bf][tid] - al * pj);
      su[bf][tid] = u;
      o_j = scale * fmaf(al, sj, s_kq * u);
    }
    // RMSNormGated needs sum_j o_j^2: the warps' sums, then each thread adds them up itself
    float ss = warp_sum(tid < dv ? o_j * o_j : 0.0f);
    if (lane == 0) sred[bf][warp] = ss;
    __syncthreads();
    if (tid < dv) {
      float t = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) t += sred[bf][w];
      const float inv = rsqrtf(t / (float)dv + kEpsRms);
      const size_t oi = ((size_t)b * h_v + h) * dv + tid;
      out[oi] = from_f<IO>(o_j * inv * p.norm_w[tid] * silu_f(to_f(xz[oi])));
    }
    // H <- alpha H + k u^T, written back in place
    if (col_ok) {
      const float u0 = su[bf][j0], u1 = su[bf][j0 + 1], u2 = su[bf][j0 + 2], u3 = su[bf][j0 + 3];
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r) {
        const int i = i0 + r;
        if (r < rows && i < dk) {
          const float kv = sk[i];
          float4 hn;
          hn.x = fmaf(kv, u0, al * Hr[r].x);
          hn.y = fmaf(kv, u1, al * Hr[r].y);
          hn.z = fmaf(kv, u2, al * Hr[r].z);
          hn.w = fmaf(kv, u3, al * Hr[r].w);
          *reinterpret_cast<float4 *>(Hg + (size_t)i * dv + j0) = hn;
        }
      }
    }
  }
}

// Conv cache after a prefill: for sequence n and conv channel c, the raw
// inputs of its last three tokens, oldest first; where the sequence is shorter
// than three tokens, the carried history before its start (init_conv) or
// zeros.  One thread per (sequence, channel), which reads everything it needs
// before it writes (so the cache may overwrite the history in place); an
// invalid cu_seqlens range gives zeros.
template <typename IO>
__global__ void __launch_bounds__(256) conv_cache_kernel(ConvCacheParams p) {
  const int n = blockIdx.y;
  const int ch = blockIdx.x * blockDim.x + threadIdx.x;
  const int cq = p.h_qk * p.d_k, Cc = 2 * cq + p.h_v * p.d_v;
  if (ch >= Cc) return;
  const int s0 = p.cu_seqlens[n], s1 = p.cu_seqlens[n + 1];
  const bool ok = s0 >= 0 && s1 >= s0 && s1 <= p.T;
  const IO *src;
  size_t stride, col;
  if (ch < cq) {
    src = static_cast<const IO *>(p.q); stride = cq; col = ch;
  } else if (ch < 2 * cq) {
    src = static_cast<const IO *>(p.k); stride = cq; col = ch - cq;
  } else {
    src = static_cast<const IO *>(p.v); stride = (size_t)p.h_v * p.d_v; col = ch - 2 * cq;
  }
  const IO *hist = p.init_conv ? static_cast<const IO *>(p.init_conv) + ((size_t)n * Cc + ch) * 3 : nullptr;
  IO val[3];
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const int t = s1 - 3 + j;  // >= s0 - 3: history entry t - s0 + 3 when t < s0
    val[j] = !ok ? from_f<IO>(0.0f) : t >= s0 ? src[(size_t)t * stride + col] : hist ? hist[t - s0 + 3] : from_f<IO>(0.0f);
  }
  IO *dst = static_cast<IO *>(p.conv_cache) + ((size_t)n * Cc + ch) * 3;
#pragma unroll
  for (int j = 0; j < 3; ++j) dst[j] = val[j];
}

}  // namespace

cudaError_t launch_conv_cache(const ConvCacheParams &p, bool bf16, cudaStream_t s) {
  const int Cc = 2 * p.h_qk * p.d_k + p.h_v * p.d_v;
  if (p.N <= 0) return cudaSuccess;
  const dim3 grid((unsigned)((Cc + 255) / 256), (unsigned)p.N);
  if (bf16)
    conv_cache_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(p);
  else
    conv_cache_kernel<float><<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeParams &p, bool bf16, cudaStream_t s) {
  const unsigned grid = (unsigned)p.B * (unsigned)p.h_qk;
  if (grid == 0) return cudaSuccess;
  trace_begin(s, GDN_K_DECODE);
  const bool d128 = p.d_k == 128 && p.d_v == 128;
  if (bf16) {
    if (d128) decode_kernel<__nv_bfloat16, 128><<<grid, kThreads, 0, s>>>(p);
    else decode_kernel<__nv_bfloat16, 0><<<grid, kThreads, 0, s>>>(p);
  } else {
    if (d128) decode_kernel<float, 128><<<grid, kThreads, 0, s>>>(p);
    else decode_kernel<float, 0><<<grid, kThreads, 0, s>>>(p);
  }
  trace_end(s);
  return cudaGetLastError();
}

}  // namespace gdn
