// Backward pass of the layer (reverse mode), fp32 on the CUDA cores.
//
// The gradient of a scalar loss with respect to every input, given the
// gradient dy of the output y (and optionally of the final state).  Three
// launches on the caller's stream:
//
//   bwd_chain_kernel     one CTA per (sequence, value head) chain.  Forward
//                        over the sequence in blocks of kB tokens, writing the
//                        state H = S^T at each block start to the workspace;
//                        then the blocks in reverse: the block's q, k, v, gates
//                        and states recomputed from its checkpoint (every
//                        state kept in the workspace), RMSNormGated in reverse
//                        (dz, dnorm_w, do), and the rule in reverse token by
//                        token with the gradient G of the state in registers:
//                          G += scale q do^T,        dq = scale H_t do
//                          dalpha = <G, H_{t-1}>,    du = G^T k,  dk = G u
//                          dbeta = du.(v - alpha p), dv = beta du
//                          dalpha -= beta du.p,      dp = -alpha beta du
//                          dk += H_{t-1} dp,         G <- alpha G + k dp^T
//                        Writes dz, the gradients of the normalised q, k, of
//                        the conv'd v and of the gates per (token, value head)
//                        to the workspace, and the initial state's gradient.
//   bwd_prologue_kernel  per (token tile, conv head): the q / k gradients of
//                        the value heads of a q/k head summed, L2 norm and
//                        SiLU in reverse (the conv recomputed), then the
//                        conv(4) in reverse: d x and d conv_w.
//   bwd_gate_kernel      per (token, value head): da, db, and the sums into
//                        dA_log and ddt_bias.
//
// The state layout follows the forward fp32 kernel: warp w owns columns
// [8w, 8w+8) of H, lane l rows l, l+32, l+64, l+96.  Sums over tokens or
// heads into one parameter (conv_w, A_log, dt_bias, norm_w) are fp32 atomic
// adds, so their rounding order is not fixed from run to run.
#include "gdn_common.cuh"
#include "../../include/gdn_trace.h"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kB = 32;     // tokens per block (checkpoint interval, prologue batch)
constexpr int kCW = 8;     // state columns per warp
constexpr int kRows = 4;   // rows per lane (d_k <= 128)
constexpr int kSlot = kRows * kCW;  // state values per thread

struct BwdWs {
  float *ckpt;   // [slots][h_v][threads][kSlot]: the state at each block start
  float *hs;     // [N][h_v][kB + 1][threads][kSlot]: the states of the block in reverse
  float *dqn;    // [T][h_v][d_k]: gradient of the normalised q (per value head)
  float *dkn;    // [T][h_v][d_k]
  float *dvs;    // [T][h_v][d_v]: gradient of silu(conv(v))
  float *dg;     // [T][h_v]
  float *dbeta;  // [T][h_v]
  int slots;     // ceil(T / kB) + N
};

struct BwdLayout {
  size_t ckpt, hs, dqn, dkn, dvs, dg, dbeta, total;
  int slots;
  BwdLayout(int T, int N, int h_v, int d_k, int d_v) {
    const size_t threads = 32 * (size_t)((d_v + kCW - 1) / kCW);
    const size_t st = threads * kSlot * sizeof(float);
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    slots = (T + kB - 1) / kB + N;
    ckpt = 0;
    hs = up(ckpt + (size_t)slots * h_v * st);
    dqn = up(hs + (size_t)N * h_v * (kB + 1) * st);
    dkn = up(dqn + (size_t)T * h_v * d_k * sizeof(float));
    dvs = up(dkn + (size_t)T * h_v * d_k * sizeof(float));
    dg = up(dvs + (size_t)T * h_v * d_v * sizeof(float));
    dbeta = up(dg + (size_t)T * h_v * sizeof(float));
    total = up(dbeta + (size_t)T * h_v * sizeof(float));
  }
};

// The block's prologue (as the forward fp32 kernel): conv(4) + SiLU of q, k,
// v, L2 norm of q, k, and the gates, for tokens [t0, t0 + nt) of sequence
// [s0, s1) into shared memory.
template <typename IO>
__device__ void block_prologue(const BwdParams &p, int h, int hq, int s0, int t0, int nt, float *sq, float *sk,
                               float *sv, float *salpha, float *sbeta, float A_exp, float dtb) {
  const int h_v = p.h_v, h_qk = p.h_qk, dk = p.d_k, dv = p.d_v;
  const int nch = 2 * dk + dv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  const IO *xq = static_cast<const IO *>(p.q), *xk = static_cast<const IO *>(p.k), *xv = static_cast<const IO *>(p.v);
  const IO *xa = static_cast<const IO *>(p.a), *xb = static_cast<const IO *>(p.b);
  for (int idx = threadIdx.x; idx < nt * nch; idx += blockDim.x) {
    const int tt = idx / nch, c = idx % nch;
    const int t = t0 + tt;
    const IO *src;
    size_t stride;
    int ch;
    float *dst;
    if (c < dk) {
      src = xq + hq * dk + c; stride = (size_t)h_qk * dk; ch = hq * dk + c; dst = sq + tt * dk + c;
    } else if (c < 2 * dk) {
      const int cc = c - dk;
      src = xk + hq * dk + cc; stride = (size_t)h_qk * dk; ch = h_qk * dk + hq * dk + cc; dst = sk + tt * dk + cc;
    } else {
      const int cc = c - 2 * dk;
      src = xv + h * dv + cc; stride = (size_t)h_v * dv; ch = 2 * h_qk * dk + h * dv + cc; dst = sv + tt * dv + cc;
    }
    float pre = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int tau = t - 3 + j;
      if (tau >= s0) pre = fmaf(p.conv_w[ch * 4 + j], to_f(src[(size_t)tau * stride]), pre);
    }
    *dst = silu_f(pre);
  }
  for (int tt = threadIdx.x; tt < nt; tt += blockDim.x) {
    const size_t t = (size_t)(t0 + tt);
    salpha[tt] = expf(gate_g(to_f(xa[t * h_v + h]), A_exp, dtb));
    sbeta[tt] = sigmoid_f(to_f(xb[t * h_v + h]));
  }
  __syncthreads();
  for (int row = warp; row < 2 * nt; row += nwarps) {
    float *x = row < nt ? sq + row * dk : sk + (row - nt) * dk;
    float ss = 0.0f;
    for (int i = lane; i < dk; i += 32) ss = fmaf(x[i], x[i], ss);
    const float inv = rsqrtf(warp_sum(ss) + kEpsL2);
    for (int i = lane; i < dk; i += 32) x[i] *= inv;
  }
  __syncthreads();
}

template <typename IO>
__global__ void __launch_bounds__(512) bwd_chain_kernel(const BwdParams p, const BwdWs ws) {
  const int h_v = p.h_v, h_qk = p.h_qk, dk = p.d_k, dv = p.d_v;
  const int n = blockIdx.x / h_v, h = blockIdx.x % h_v, hq = h / (h_v / h_qk);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nwarps = blockDim.x >> 5;
  const int s0 = p.cu_seqlens[n], s1 = p.cu_seqlens[n + 1];
  if (s0 < 0 || s1 < s0 || s1 > p.T) {
    if (tid == 0) set_status(p.status, kDevBadSeqlens);
    return;
  }
  const int L = s1 - s0, nblk = (L + kB - 1) / kB;
  const int slot0 = s0 / kB + n;  // the sequence's first checkpoint slot (sequences never overlap)

  extern __shared__ float smem[];
  float *sq = smem;                 // [kB][dk]
  float *sk = sq + kB * dk;         // [kB][dk]
  float *sv = sk + kB * dk;         // [kB][dv]
  float *so = sv + kB * dv;         // [kB][dv]  o of the block's tokens
  float *sdo = so + kB * dv;        // [kB][dv]  their do
  float *red_q = sdo + kB * dv;     // [nwarps][128]
  float *red_k = red_q + nwarps * 128;
  float *red_s = red_k + nwarps * 128;  // [nwarps][4]
  float *snw = red_s + nwarps * 4;      // [dv] partial dnorm_w
  float *salpha = snw + dv;             // [kB]
  float *sbeta = salpha + kB;           // [kB]

  const IO *xz = static_cast<const IO *>(p.z);
  const IO *gy = static_cast<const IO *>(p.dy);
  const int j0 = warp * kCW;
  const float A_exp = expf(p.A_log[h]), dtb = p.dt_bias[h];
  const float scale = rsqrtf((float)dk);
  for (int j = tid; j < dv; j += blockDim.x) snw[j] = 0.0f;

  auto elem_ok = [&](int r, int c) { return lane + 32 * r < dk && j0 + c < dv; };
  auto slot_ptr = [&](float *base, size_t slot) {
    return base + (slot * blockDim.x + tid) * kSlot;  // this thread's kSlot values, contiguous
  };
  auto store_state = [&](float *dst, const float (&H)[kRows][kCW]) {
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
      for (int c = 0; c < kCW; c += 4)
        *reinterpret_cast<float4 *>(dst + r * kCW + c) = make_float4(H[r][c], H[r][c + 1], H[r][c + 2], H[r][c + 3]);
  };
  auto load_state = [&](const float *src, float (&H)[kRows][kCW]) {
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
      for (int c = 0; c < kCW; c += 4) {
        const float4 f = *reinterpret_cast<const float4 *>(src + r * kCW + c);
        H[r][c] = f.x; H[r][c + 1] = f.y; H[r][c + 2] = f.z; H[r][c + 3] = f.w;
      }
  };
  // one forward step of the rule on this warp's columns; o of the token (scaled) to so[tt] if wanted
  auto step = [&](float (&H)[kRows][kCW], int tt, bool want_o) {
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
      pc[c] = warp_sum(s);
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
    if (want_o) {
#pragma unroll
      for (int c = 0; c < kCW; ++c) {
        const float o = warp_sum(oc[c]);
        if (lane == c && j0 + c < dv) so[tt * dv + j0 + c] = o * scale;
      }
    }
  };

  // ---------------- forward: checkpoints at block starts
  const size_t chain_off = ((size_t)n * h_v + h) * dk * dv;
  float H[kRows][kCW];
#pragma unroll
  for (int r = 0; r < kRows; ++r)
#pragma unroll
    for (int c = 0; c < kCW; ++c)
      H[r][c] = (p.init_state && elem_ok(r, c)) ? p.init_state[chain_off + (size_t)(lane + 32 * r) * dv + j0 + c]
                                                : 0.0f;
  for (int b = 0; b < nblk; ++b) {
    const int t0 = s0 + kB * b, nt = min(kB, s1 - t0);
    store_state(slot_ptr(ws.ckpt, (size_t)(slot0 + b) * h_v + h), H);
    if (b + 1 == nblk) break;  // the last block's tokens are only needed in reverse
    __syncthreads();
    block_prologue<IO>(p, h, hq, s0, t0, nt, sq, sk, sv, salpha, sbeta, A_exp, dtb);
    if (j0 < dv)
      for (int tt = 0; tt < nt; ++tt) step(H, tt, false);
  }

  // ---------------- reverse, block by block
  float G[kRows][kCW];
#pragma unroll
  for (int r = 0; r < kRows; ++r)
#pragma unroll
    for (int c = 0; c < kCW; ++c)
      G[r][c] = (p.dfinal_state && elem_ok(r, c))
                    ? p.dfinal_state[chain_off + (size_t)(lane + 32 * r) * dv + j0 + c] : 0.0f;
  float *hs = ws.hs + ((size_t)n * h_v + h) * (kB + 1) * blockDim.x * kSlot;
  for (int b = nblk - 1; b >= 0; --b) {
    const int t0 = s0 + kB * b, nt = min(kB, s1 - t0);
    __syncthreads();
    block_prologue<IO>(p, h, hq, s0, t0, nt, sq, sk, sv, salpha, sbeta, A_exp, dtb);
    load_state(slot_ptr(ws.ckpt, (size_t)(slot0 + b) * h_v + h), H);
    for (int tt = 0; tt < nt; ++tt) {  // the block's states and outputs again
      store_state(slot_ptr(hs, tt), H);
      if (j0 < dv) step(H, tt, true);
    }
    store_state(slot_ptr(hs, nt), H);
    __syncthreads();
    // RMSNormGated in reverse, one warp per token
    for (int tt = warp; tt < nt; tt += nwarps) {
      const size_t row = ((size_t)(t0 + tt) * h_v + h) * dv;
      float ss = 0.0f, dot = 0.0f;
      for (int j = lane; j < dv; j += 32) {
        const float o = so[tt * dv + j], z = to_f(xz[row + j]);
        ss = fmaf(o, o, ss);
        dot = fmaf(to_f(gy[row + j]) * o, p.norm_w[j] * silu_f(z), dot);
      }
      ss = warp_sum(ss);
      dot = warp_sum(dot);
      const float r = rsqrtf(ss / (float)dv + kEpsRms);
      for (int j = lane; j < dv; j += 32) {
        const float o = so[tt * dv + j], z = to_f(xz[row + j]), g = to_f(gy[row + j]);
        const float s = sigmoid_f(z), silu = z * s, w = p.norm_w[j];
        sdo[tt * dv + j] = r * w * silu * g - o * r * r * r * dot / (float)dv;
        p.dz[row + j] = g * o * r * w * s * (1.0f + z * (1.0f - s));
        atomicAdd(&snw[j], g * o * r * silu);
      }
    }
    __syncthreads();
    const float *hs_c = hs;
    for (int tt = nt - 1; tt >= 0; --tt) {
      const size_t tok = (size_t)(t0 + tt) * h_v + h;
      float Hp[kRows][kCW], Ht[kRows][kCW];
      load_state(slot_ptr(const_cast<float *>(hs_c), tt), Hp);
      load_state(slot_ptr(const_cast<float *>(hs_c), tt + 1), Ht);
      float kr[kRows], qr[kRows];
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        const int i = lane + 32 * r;
        kr[r] = i < dk ? sk[tt * dk + i] : 0.0f;
        qr[r] = i < dk ? sq[tt * dk + i] : 0.0f;
      }
      const float al = salpha[tt], be = sbeta[tt];
      float doc[kCW], vc[kCW];
#pragma unroll
      for (int c = 0; c < kCW; ++c) {
        const int j = j0 + c;
        doc[c] = j < dv ? sdo[tt * dv + j] : 0.0f;
        vc[c] = j < dv ? sv[tt * dv + j] : 0.0f;
      }
      float dqp[kRows], dkp[kRows];
      float s_dal = 0.0f;
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        float sq_ = 0.0f;
#pragma unroll
        for (int c = 0; c < kCW; ++c) {
          G[r][c] = fmaf(scale * qr[r], doc[c], G[r][c]);
          sq_ = fmaf(Ht[r][c], doc[c], sq_);
          s_dal = fmaf(G[r][c], Hp[r][c], s_dal);
        }
        dqp[r] = scale * sq_;
      }
      float pc[kCW], du[kCW];
#pragma unroll
      for (int c = 0; c < kCW; ++c) {
        float a = 0.0f, d = 0.0f;
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          a = fmaf(Hp[r][c], kr[r], a);
          d = fmaf(G[r][c], kr[r], d);
        }
        pc[c] = warp_sum(a);
        du[c] = warp_sum(d);
      }
      float s_db = 0.0f, s_dup = 0.0f, dp[kCW];
#pragma unroll
      for (int c = 0; c < kCW; ++c) {
        const float u = be * (vc[c] - al * pc[c]);
        s_db = fmaf(du[c], vc[c] - al * pc[c], s_db);
        s_dup = fmaf(du[c], pc[c], s_dup);
        dp[c] = -al * be * du[c];
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          if (c == 0) dkp[r] = 0.0f;
          dkp[r] = fmaf(G[r][c], u, dkp[r]);
        }
      }
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
#pragma unroll
        for (int c = 0; c < kCW; ++c) {
          dkp[r] = fmaf(Hp[r][c], dp[c], dkp[r]);
          G[r][c] = fmaf(kr[r], dp[c], al * G[r][c]);
        }
      }
      if (j0 < dv) {
#pragma unroll
        for (int c = 0; c < kCW; ++c)
          if (lane == c && j0 + c < dv) ws.dvs[tok * dv + j0 + c] = be * du[c];
      }
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        red_q[warp * 128 + lane + 32 * r] = dqp[r];
        red_k[warp * 128 + lane + 32 * r] = dkp[r];
      }
      s_dal = warp_sum(s_dal);
      if (lane == 0) {
        red_s[warp * 4 + 0] = s_dal;
        red_s[warp * 4 + 1] = s_db;   // the same in every lane (after the column sums)
        red_s[warp * 4 + 2] = s_dup;
      }
      __syncthreads();
      for (int i = tid; i < dk; i += blockDim.x) {
        float a = 0.0f, c2 = 0.0f;
        for (int w = 0; w < nwarps; ++w) {
          a += red_q[w * 128 + i];
          c2 += red_k[w * 128 + i];
        }
        ws.dqn[tok * dk + i] = a;
        ws.dkn[tok * dk + i] = c2;
      }
      if (tid == 32 * (nwarps - 1)) {  // a lane of the last warp: the scalar sums
        float dal = 0.0f, db = 0.0f, dup = 0.0f;
        for (int w = 0; w < nwarps; ++w) {
          dal += red_s[w * 4 + 0];
          db += red_s[w * 4 + 1];
          dup += red_s[w * 4 + 2];
        }
        ws.dg[tok] = al * (dal - be * dup);
        ws.dbeta[tok] = db;
      }
      __syncthreads();
    }
  }
  if (p.dinit_state) {
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
      for (int c = 0; c < kCW; ++c)
        if (elem_ok(r, c)) p.dinit_state[chain_off + (size_t)(lane + 32 * r) * dv + j0 + c] = G[r][c];
  }
  __syncthreads();
  for (int j = tid; j < dv; j += blockDim.x) atomicAdd(&p.dnorm_w[j], snw[j]);
}

// Sequence [s0, s1) of token t (binary search over cu_seqlens).
__device__ __forceinline__ int2 seq_of(const int32_t *cu, int N, int t) {
  int lo = 0, hi = N - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return make_int2(cu[lo], cu[lo + 1]);
}

__device__ __forceinline__ float block_sum128(float v, float *red) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  const float s = red[0] + red[1] + red[2] + red[3];
  __syncthreads();
  return s;
}

constexpr int kTile = 64;

// per (token tile, conv head): conv head y < h_qk is q head y, then the k
// heads, then the value heads; thread c = channel c of the head (d <= 128).
template <typename IO>
__global__ void __launch_bounds__(128) bwd_prologue_kernel(const BwdParams p, const BwdWs ws) {
  const int h_v = p.h_v, h_qk = p.h_qk, dk = p.d_k, dv = p.d_v, rep = h_v / h_qk;
  const int t0 = blockIdx.x * kTile, y = blockIdx.y, c = threadIdx.x;
  __shared__ float sdp[kTile + 3][128];
  __shared__ float red[4];
  const bool is_q = y < h_qk, is_k = !is_q && y < 2 * h_qk;
  const int D = (is_q || is_k) ? dk : dv;
  const int hq = is_q ? y : y - h_qk, hvv = y - 2 * h_qk;
  const IO *src;
  size_t stride;
  int cb;  // conv channel of channel 0 of this head
  float *dx;
  if (is_q) {
    src = static_cast<const IO *>(p.q) + hq * dk; stride = (size_t)h_qk * dk; cb = hq * dk; dx = p.dq + hq * dk;
  } else if (is_k) {
    src = static_cast<const IO *>(p.k) + hq * dk; stride = (size_t)h_qk * dk; cb = h_qk * dk + hq * dk;
    dx = p.dk + hq * dk;
  } else {
    src = static_cast<const IO *>(p.v) + hvv * dv; stride = (size_t)h_v * dv; cb = 2 * h_qk * dk + hvv * dv;
    dx = p.dv + hvv * dv;
  }
  const bool act = c < D;
  float w[4] = {0.f, 0.f, 0.f, 0.f};
  if (act)
#pragma unroll
    for (int j = 0; j < 4; ++j) w[j] = p.conv_w[(size_t)(cb + c) * 4 + j];
  // d pre of tokens [t0, t0 + kTile + 3) (the ones the tile's inputs feed)
  for (int tt = 0; tt < kTile + 3; ++tt) {
    const int t = t0 + tt;
    if (t >= p.T) break;  // uniform over the CTA
    const int2 sq = seq_of(p.cu_seqlens, p.N, t);
    float pre = 0.0f;
    if (act)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int tau = t - 3 + j;
        if (tau >= sq.x) pre = fmaf(w[j], to_f(src[(size_t)tau * stride + c]), pre);
      }
    const float s = sigmoid_f(pre), xh = pre * s, dsilu = s * (1.0f + pre * (1.0f - s));
    float dxh;
    if (is_q || is_k) {
      const float *gsrc = is_q ? ws.dqn : ws.dkn;
      float gsum = 0.0f;
      if (act)
        for (int r = 0; r < rep; ++r) gsum += gsrc[((size_t)t * h_v + hq * rep + r) * dk + c];
      const float nrm = sqrtf(block_sum128(act ? xh * xh : 0.0f, red) + kEpsL2);
      const float yv = xh / nrm;
      const float yg = block_sum128(act ? yv * gsum : 0.0f, red);
      dxh = (gsum - yv * yg) / nrm;
    } else {
      dxh = act ? ws.dvs[((size_t)t * h_v + hvv) * dv + c] : 0.0f;
    }
    sdp[tt][c] = act ? dxh * dsilu : 0.0f;
  }
  __syncthreads();
  if (!act) return;
  float dw[4] = {0.f, 0.f, 0.f, 0.f};
  const int Tc = p.T;
  for (int tt = 0; tt < kTile; ++tt) {
    const int t = t0 + tt;
    if (t >= Tc) break;
    const int2 sq = seq_of(p.cu_seqlens, p.N, t);
    float acc = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int tp = t + 3 - j;  // the output token that reads input t through tap j
      if (tp < sq.y) acc = fmaf(sdp[tt + 3 - j][c], w[j], acc);
      const int tau = t - 3 + j;  // the input tap j of output t reads
      if (tau >= sq.x) dw[j] = fmaf(sdp[tt][c], to_f(src[(size_t)tau * stride + c]), dw[j]);
    }
    dx[(size_t)t * stride + c] = acc;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) atomicAdd(&p.dconv_w[(size_t)(cb + c) * 4 + j], dw[j]);
}

template <typename IO>
__global__ void __launch_bounds__(256) bwd_gate_kernel(const BwdParams p, const BwdWs ws) {
  const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (size_t)p.T * p.h_v) return;
  const int h = (int)(idx % p.h_v);
  const float a = to_f(static_cast<const IO *>(p.a)[idx]), b = to_f(static_cast<const IO *>(p.b)[idx]);
  const float x = a + p.dt_bias[h], A_exp = expf(p.A_log[h]);
  const float dg = ws.dg[idx];
  const float da = dg * (-A_exp) * sigmoid_f(x);
  const float be = sigmoid_f(b);
  p.da[idx] = da;
  p.db[idx] = ws.dbeta[idx] * be * (1.0f - be);
  atomicAdd(&p.ddt_bias[h], da);
  atomicAdd(&p.dA_log[h], dg * gate_g(a, A_exp, p.dt_bias[h]));
}

}  // namespace

size_t prefill_backward_workspace_bytes(int T, int N, int h_qk, int h_v, int d_k, int d_v) {
  (void)h_qk;
  return BwdLayout(T, N, h_v, d_k, d_v).total;
}

cudaError_t launch_prefill_backward(const BwdParams &p, bool bf16, cudaStream_t s) {
  const BwdLayout L(p.T, p.N, p.h_v, p.d_k, p.d_v);
  if (p.ws_bytes < L.total) return cudaErrorInvalidValue;
  BwdWs ws;
  ws.ckpt = reinterpret_cast<float *>(p.ws + L.ckpt);
  ws.hs = reinterpret_cast<float *>(p.ws + L.hs);
  ws.dqn = reinterpret_cast<float *>(p.ws + L.dqn);
  ws.dkn = reinterpret_cast<float *>(p.ws + L.dkn);
  ws.dvs = reinterpret_cast<float *>(p.ws + L.dvs);
  ws.dg = reinterpret_cast<float *>(p.ws + L.dg);
  ws.dbeta = reinterpret_cast<float *>(p.ws + L.dbeta);
  ws.slots = L.slots;
  const int Cc = 2 * p.h_qk * p.d_k + p.h_v * p.d_v;
  cudaError_t e;
  // the parameter gradients are sums (atomic adds) over tokens and heads
  if ((e = cudaMemsetAsync(p.dconv_w, 0, sizeof(float) * (size_t)Cc * 4, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(p.dA_log, 0, sizeof(float) * (size_t)p.h_v, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(p.ddt_bias, 0, sizeof(float) * (size_t)p.h_v, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(p.dnorm_w, 0, sizeof(float) * (size_t)p.d_v, s)) != cudaSuccess) return e;
  const int warps = (p.d_v + kCW - 1) / kCW;
  const int threads = 32 * warps;
  const size_t smem = sizeof(float) * ((size_t)kB * (2 * p.d_k + 3 * p.d_v) + (size_t)warps * (2 * 128 + 4) +
                                       p.d_v + 2 * kB);
  const unsigned chains = (unsigned)p.N * (unsigned)p.h_v;
  const dim3 pgrid((unsigned)((p.T + kTile - 1) / kTile), (unsigned)(2 * p.h_qk + p.h_v));
  const unsigned ggrid = (unsigned)(((size_t)p.T * p.h_v + 255) / 256);
  auto run = [&](auto chain_k, auto pro_k, auto gate_k) -> cudaError_t {
    cudaError_t err = cudaFuncSetAttribute(chain_k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    trace_begin(s, GDN_K_BWD_CHAIN);
    if (chains) chain_k<<<chains, threads, smem, s>>>(p, ws);
    trace_end(s);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if (p.T > 0) {
      trace_begin(s, GDN_K_BWD_PROLOGUE);
      pro_k<<<pgrid, 128, 0, s>>>(p, ws);
      trace_end(s);
      if ((err = cudaGetLastError()) != cudaSuccess) return err;
      gate_k<<<ggrid, 256, 0, s>>>(p, ws);
    }
    return cudaGetLastError();
  };
  if (bf16)
    return run(bwd_chain_kernel<__nv_bfloat16>, bwd_prologue_kernel<__nv_bfloat16>, bwd_gate_kernel<__nv_bfloat16>);
  return run(bwd_chain_kernel<float>, bwd_prologue_kernel<float>, bwd_gate_kernel<float>);
}

}  // namespace gdn
