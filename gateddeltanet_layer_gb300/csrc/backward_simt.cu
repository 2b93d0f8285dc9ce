// Backward pass of the layer (reverse mode), fp32 on the CUDA cores.
//
// The gradient of a scalar loss with respect to every input, given the
// gradient dy of the output y (and optionally of the final state).  The
// columns j of the state H = S^T (d_v) evolve independently under the rule,
// and so do the columns of its gradient G, so every chain (sequence, value
// head) is split over ceil(d_v / 32) CTAs of 32 columns each; what a token
// step sums over columns (the gradients of q, k, alpha, beta) is added up
// across them with atomic adds.  Five launches on the caller's stream:
//
//   bwd_fwd_kernel       per (chain, column slice): forward over the sequence
//                        in blocks of kB tokens, writing the slice of the
//                        state at each block start and o of every token to
//                        the workspace.
//   bwd_norm_kernel      per (token, value head) row: RMSNormGated in reverse
//                        (it needs whole rows): do to the workspace, dz, and
//                        the sums into dnorm_w.
//   bwd_rev_kernel       per (chain, column slice): the blocks in reverse: the
//                        block's q, k, v and gates, and its states from the
//                        checkpoint (every state kept in the workspace), then
//                        the rule in reverse token by token with the slice of
//                        the state's gradient G in registers:
//                          G += scale q do^T,        dq = scale H_t do
//                          dalpha = <G, H_{t-1}>,    du = G^T k,  dk = G u
//                          dbeta = du.(v - alpha p), dv = beta du
//                          dalpha -= beta du.p,      dp = -alpha beta du
//                          dk += H_{t-1} dp,         G <- alpha G + k dp^T
//                        adding the gradients of the normalised q, k and of
//                        the gates per (token, value head) into the workspace,
//                        writing those of silu(conv(v)) and of the initial
//                        state for its columns.
//   bwd_prologue_kernel  per (token tile, conv head): the q / k gradients of
//                        the value heads of a q/k head summed, L2 norm and
//                        SiLU in reverse (the conv recomputed), then the
//                        conv(4) in reverse: d x and d conv_w.
//   bwd_gate_kernel      per (token, value head): da, db, and the sums into
//                        dA_log and ddt_bias.
//
// The slice layout: warp w owns columns [kCW w, kCW w + kCW) of the slice
// (two, so that a token step's chain of dependent work per warp is short:
// 16 warps per slice of 32 columns measured 8.2 ms on the 4096-token
// workload, against 9.4 with 4 columns per warp and 10.9 with 8; 7.2 with the
// head dim fixed at 128 at compile time), lane l rows
// l, l+32, l+64, l+96.  Sums into one
// value from several CTAs are atomic adds, so their rounding order is not
// fixed from run to run: fp32 for the per-token q, k and gate gradients (a
// few terms each), fp64 for the parameter gradients (conv_w, A_log, dt_bias,
// norm_w: sums over every token and head, converted to fp32 at the end).
#include <algorithm>

#include "gdn_common.cuh"
#include "../../include/gdn_trace.h"
#include "gdn_internal.h"
#include "token_inputs.cuh"

namespace gdn {
namespace {

constexpr int kB = 32;        // tokens per block (checkpoint interval, prologue batch)
constexpr int kCW = 2;        // state columns per warp
constexpr int kRows = 4;      // rows per lane (d_k <= 128)
constexpr int kSlot = kRows * kCW;  // state values per thread
constexpr int kSliceWarps = 16, kSliceCols = kCW * kSliceWarps, kSliceThreads = 32 * kSliceWarps;
constexpr int kColLanes = 32 / kCW;  // a reduce-scatter over the warp leaves column c in lanes c kColLanes ..

struct BwdWs {
  float *ckpt;   // [slots][h_v][slices][kSliceThreads][kSlot]: the state slice at each block start
  float *hs;     // [N][h_v][slices][kB + 1][kSliceThreads][kSlot]: the block's states, in reverse
  float *wo;     // [T][h_v][d_v]: o (scaled) of every token
  float *wdo;    // [T][h_v][d_v]: its gradient
  float *xq;     // [T][h_qk][d_k]: q^ = L2-normalised silu(conv(q)), every token (computed once)
  float *xk;     // [T][h_qk][d_k]: k^
  float *xv;     // [T][h_v][d_v]: silu(conv(v))
  float *xal;    // [T][h_v]: alpha = e^g
  float *xbe;    // [T][h_v]: beta
  float *dqn;    // [T][h_v][d_k]: gradient of the normalised q (per value head; summed over slices)
  float *dkn;    // [T][h_v][d_k]
  float *dvs;    // [T][h_v][d_v]: gradient of silu(conv(v))
  float *dg;     // [T][h_v]
  float *dbeta;  // [T][h_v]
  double *acc;   // fp64 sums: conv_w [Cc][4], A_log [h_v], dt_bias [h_v], norm_w [d_v]
  int slices;    // ceil(d_v / kSliceCols)
};

struct BwdLayout {
  size_t ckpt, hs, wo, wdo, xq, xk, xv, xal, xbe, dqn, dkn, dvs, dg, dbeta, acc, total;
  int slots, slices;
  BwdLayout(int T, int N, int h_qk, int h_v, int d_k, int d_v) {
    slices = (d_v + kSliceCols - 1) / kSliceCols;
    const size_t st = (size_t)kSliceThreads * kSlot * sizeof(float);  // one state slice
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    slots = (T + kB - 1) / kB + N;
    ckpt = 0;
    hs = up(ckpt + (size_t)slots * h_v * slices * st);
    wo = up(hs + (size_t)N * h_v * slices * (kB + 1) * st);
    wdo = up(wo + (size_t)T * h_v * d_v * sizeof(float));
    xq = up(wdo + (size_t)T * h_v * d_v * sizeof(float));
    xk = up(xq + (size_t)T * h_qk * d_k * sizeof(float));
    xv = up(xk + (size_t)T * h_qk * d_k * sizeof(float));
    xal = up(xv + (size_t)T * h_v * d_v * sizeof(float));
    xbe = up(xal + (size_t)T * h_v * sizeof(float));
    dqn = up(xbe + (size_t)T * h_v * sizeof(float));
    dkn = up(dqn + (size_t)T * h_v * d_k * sizeof(float));
    dvs = up(dkn + (size_t)T * h_v * d_k * sizeof(float));
    dg = up(dvs + (size_t)T * h_v * d_v * sizeof(float));
    dbeta = up(dg + (size_t)T * h_v * sizeof(float));
    acc = up(dbeta + (size_t)T * h_v * sizeof(float));
    total = up(acc + sizeof(double) * ((size_t)(2 * h_qk * d_k + h_v * d_v) * 4 + 2 * h_v + d_v));
  }
};

// The block's inputs into shared memory: q^, k^ and the slice's columns
// [j0, j0 + kSliceCols) of silu(conv(v)) (zeros past d_v), alpha and beta, for
// tokens [t0, t0 + nt), from the arrays token_inputs_kernel wrote.
__device__ __forceinline__ void block_prologue(const BwdParams &p, const BwdWs &ws, int dk, int h, int hq, int t0,
                                               int nt, int j0,
                               float *sq, float *sk, float *sv, float *salpha, float *sbeta) {
  const int h_v = p.h_v, h_qk = p.h_qk, dv = p.d_v;
  // float4 copies (d_k, d_v and the row offsets are multiples of 16 floats), kU in flight per thread
  const int nq = dk / 4, nv = kSliceCols / 4, per_tok = 2 * nq + nv, total = nt * per_tok;
  const float4 *gq = reinterpret_cast<const float4 *>(ws.xq), *gk = reinterpret_cast<const float4 *>(ws.xk);
  const float4 *gv = reinterpret_cast<const float4 *>(ws.xv);
  float4 *sq4 = reinterpret_cast<float4 *>(sq), *sk4 = reinterpret_cast<float4 *>(sk);
  float4 *sv4 = reinterpret_cast<float4 *>(sv);
  constexpr int kU = 6;
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
          const int jj = j0 + 4 * (c - 2 * nq);
          val[u] = jj < dv ? gv[((t * h_v + h) * dv + jj) / 4] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
          dst[u] = sv4 + tt * nv + c - 2 * nq;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (dst[u]) *dst[u] = val[u];
  }
  for (int tt = threadIdx.x; tt < nt; tt += blockDim.x) {
    salpha[tt] = ws.xal[(size_t)(t0 + tt) * h_v + h];
    sbeta[tt] = ws.xbe[(size_t)(t0 + tt) * h_v + h];
  }
  __syncthreads();
}

// What a (chain, column slice) CTA works with: its chain, sequence and slice.
struct SliceCtx {
  int n, h, hq, sl, j0, s0, s1, nblk, slot0;
  bool ok;
};
__device__ __forceinline__ SliceCtx slice_ctx(const BwdParams &p, int slices) {
  SliceCtx c;
  const int chain = blockIdx.x / slices;
  c.sl = blockIdx.x % slices;
  c.n = chain / p.h_v;
  c.h = chain % p.h_v;
  c.hq = c.h / (p.h_v / p.h_qk);
  c.j0 = kSliceCols * c.sl;
  c.s0 = p.cu_seqlens[c.n];
  c.s1 = p.cu_seqlens[c.n + 1];
  c.ok = c.s0 >= 0 && c.s1 >= c.s0 && c.s1 <= p.T;
  c.nblk = c.ok ? (c.s1 - c.s0 + kB - 1) / kB : 0;
  c.slot0 = c.s0 / kB + c.n;  // the sequence's first checkpoint slot (sequences never overlap)
  return c;
}

// This thread's kSlot state values of slice `slot` in a [..][kSliceThreads][kSlot] array, contiguous.
__device__ __forceinline__ float *slice_ptr(float *base, size_t slot) {
  return base + (slot * kSliceThreads + threadIdx.x) * kSlot;
}
// (the thread's kSlot values row by row, as float4: kSlot is a multiple of 4)
static_assert(kSlot % 4 == 0, "state slots in float4");
__device__ __forceinline__ void store_state(float *dst, const float (&H)[kRows][kCW]) {
#pragma unroll
  for (int e = 0; e < kSlot; e += 4)
    *reinterpret_cast<float4 *>(dst + e) = make_float4(H[e / kCW][e % kCW], H[(e + 1) / kCW][(e + 1) % kCW],
                                                       H[(e + 2) / kCW][(e + 2) % kCW], H[(e + 3) / kCW][(e + 3) % kCW]);
}
__device__ __forceinline__ void load_state(const float *src, float (&H)[kRows][kCW]) {
#pragma unroll
  for (int e = 0; e < kSlot; e += 4) {
    const float4 f = *reinterpret_cast<const float4 *>(src + e);
    H[e / kCW][e % kCW] = f.x;
    H[(e + 1) / kCW][(e + 1) % kCW] = f.y;
    H[(e + 2) / kCW][(e + 2) % kCW] = f.z;
    H[(e + 3) / kCW][(e + 3) % kCW] = f.w;
  }
}
// One forward step of the rule on this warp's columns (jw = its first column in the slice); o of the
// token (scaled) to wo_row (the token's row of o, at the slice's first column) if given.
__device__ __forceinline__ void fwd_step(float (&H)[kRows][kCW], int tt, int dk, int jw, int jmax, const float *sq,
                                         const float *sk, const float *sv, const float *salpha, const float *sbeta,
                                         float scale, float *wo_row) {
  const int lane = threadIdx.x & 31;
  float kr[kRows], qr[kRows];
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    const int i = lane + 32 * r;
    kr[r] = i < dk ? sk[tt * dk + i] : 0.0f;
    qr[r] = i < dk ? sq[tt * dk + i] : 0.0f;
  }
  const float al = salpha[tt], be = sbeta[tt];
  // p = H^T k over the warp's columns: the column sums together (a reduce-scatter leaves column
  // l / kColLanes in lane l, then each is broadcast), not one butterfly per column
  float s[kCW];
#pragma unroll
  for (int c = 0; c < kCW; ++c) {
    s[c] = 0.0f;
#pragma unroll
    for (int r = 0; r < kRows; ++r) s[c] = fmaf(H[r][c], kr[r], s[c]);
  }
  const float ps = reduce_scatter<kCW>(s, lane);
  float o[kCW];
#pragma unroll
  for (int c = 0; c < kCW; ++c) {
    const float pc = __shfl_sync(0xffffffffu, ps, kColLanes * c);
    const float u = be * (sv[tt * kSliceCols + jw + c] - al * pc);
    o[c] = 0.0f;
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      H[r][c] = fmaf(kr[r], u, al * H[r][c]);
      o[c] = fmaf(H[r][c], qr[r], o[c]);
    }
  }
  if (wo_row) {
    const float os = reduce_scatter<kCW>(o, lane);  // lane l: column l / kColLanes
    if (lane % kColLanes == 0 && jw + lane / kColLanes < jmax) wo_row[jw + lane / kColLanes] = os * scale;
  }
}

constexpr int kRedFloats = kSliceWarps * (2 * 128 + 4);  // one buffer of the reverse step's column sums
constexpr size_t slice_smem_floats(int dk) {
  return (size_t)kB * (2 * dk + 2 * kSliceCols) + 2 * (size_t)kRedFloats + 2 * kB;
}

// Forward with checkpoints: the slice of the state at each block start, and o of every token.
template <typename IO, int DK>
__global__ void __launch_bounds__(kSliceThreads) bwd_fwd_kernel(const BwdParams p, const BwdWs ws) {
  const int h_v = p.h_v, dk = DK ? DK : p.d_k, dv = p.d_v;
  const SliceCtx cx = slice_ctx(p, ws.slices);
  if (!cx.ok) {
    if (threadIdx.x == 0) set_status(p.status, kDevBadSeqlens);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, jw = kCW * warp;
  extern __shared__ __align__(16) float smem[];
  float *sq = smem, *sk = sq + kB * dk, *sv = sk + kB * dk, *salpha = sv + 2 * kB * kSliceCols;
  float *sbeta = salpha + kB;
  const float scale = rsqrtf((float)dk);
  const size_t chain_off = ((size_t)cx.n * h_v + cx.h) * dk * dv;
  float H[kRows][kCW];
#pragma unroll
  for (int r = 0; r < kRows; ++r)
#pragma unroll
    for (int c = 0; c < kCW; ++c) {
      const int i = lane + 32 * r, j = cx.j0 + jw + c;
      H[r][c] = (p.init_state && i < dk && j < dv) ? p.init_state[chain_off + (size_t)i * dv + j] : 0.0f;
    }
  for (int b = 0; b < cx.nblk; ++b) {
    const int t0 = cx.s0 + kB * b, nt = min(kB, cx.s1 - t0);
    store_state(slice_ptr(ws.ckpt, ((size_t)(cx.slot0 + b) * h_v + cx.h) * ws.slices + cx.sl), H);
    __syncthreads();  // the previous block's shared memory is consumed
    block_prologue(p, ws, dk, cx.h, cx.hq, t0, nt, cx.j0, sq, sk, sv, salpha, sbeta);
    for (int tt = 0; tt < nt; ++tt)
      fwd_step(H, tt, dk, jw, dv - cx.j0, sq, sk, sv, salpha, sbeta, scale,
               ws.wo + ((size_t)(t0 + tt) * h_v + cx.h) * dv + cx.j0);
  }
}

// RMSNormGated in reverse, one warp per (token, value head) row; dnorm_w summed per CTA, then atomically.
template <typename IO>
__global__ void __launch_bounds__(256) bwd_norm_kernel(const BwdParams p, const BwdWs ws) {
  const int dv = p.d_v, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ double snw[8][128];
  double acc[4] = {0.0, 0.0, 0.0, 0.0};  // this lane's dnorm_w terms, columns lane + 32 m (d_v <= 128)
  const size_t rows = (size_t)p.T * p.h_v;
  // a grid of a few waves: each warp takes rows rw, rw + 8 gridDim.x, ... and keeps its dnorm_w sums in
  // registers, so each CTA adds to the global sums once
  for (size_t rw = (size_t)blockIdx.x * 8 + warp; rw < rows; rw += (size_t)gridDim.x * 8) {
    const IO *xz = static_cast<const IO *>(p.z) + rw * dv;
    const IO *gy = static_cast<const IO *>(p.dy) + rw * dv;
    const float *o = ws.wo + rw * dv;
    float ss = 0.0f, dot = 0.0f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int j = lane + 32 * m;
      if (j < dv) {
        const float z = to_f(xz[j]);
        ss = fmaf(o[j], o[j], ss);
        dot = fmaf(to_f(gy[j]) * o[j], p.norm_w[j] * silu_f(z), dot);
      }
    }
    ss = warp_sum(ss);
    dot = warp_sum(dot);
    const float r = rsqrtf(ss / (float)dv + kEpsRms);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int j = lane + 32 * m;
      if (j < dv) {
        const float z = to_f(xz[j]), g = to_f(gy[j]);
        const float s = sigmoid_f(z), silu = z * s, w = p.norm_w[j];
        ws.wdo[rw * dv + j] = r * w * silu * g - o[j] * r * r * r * dot / (float)dv;
        p.dz[rw * dv + j] = g * o[j] * r * w * s * (1.0f + z * (1.0f - s));
        acc[m] += (double)(g * o[j] * r * silu);
      }
    }
  }
#pragma unroll
  for (int m = 0; m < 4; ++m)
    if (lane + 32 * m < dv) snw[warp][lane + 32 * m] = acc[m];
  __syncthreads();
  double *acc_nw = ws.acc + (size_t)(2 * p.h_qk * p.d_k + p.h_v * dv) * 4 + 2 * p.h_v;
  for (int j = threadIdx.x; j < dv; j += blockDim.x) {
    double t = 0.0;
#pragma unroll
    for (int w = 0; w < 8; ++w) t += snw[w][j];
    atomicAdd(&acc_nw[j], t);
  }
}

// The rule in reverse, per (chain, column slice).
template <typename IO, int DK>
__global__ void __launch_bounds__(kSliceThreads) bwd_rev_kernel(const BwdParams p, const BwdWs ws) {
  const int h_v = p.h_v, dk = DK ? DK : p.d_k, dv = p.d_v;
  const SliceCtx cx = slice_ctx(p, ws.slices);
  if (!cx.ok) return;  // reported by the forward kernel
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, jw = kCW * warp;
  extern __shared__ __align__(16) float smem[];
  float *sq = smem, *sk = sq + kB * dk, *sv = sk + kB * dk, *sdo = sv + kB * kSliceCols;
  // two buffers (by token parity) of [kSliceWarps][128] q and k sums and [kSliceWarps][4] scalars: a
  // token's sums are written, then read after one barrier; the buffer is written again two tokens later
  float *red = sdo + kB * kSliceCols;
  float *salpha = red + 2 * kRedFloats, *sbeta = salpha + kB;
  const float scale = rsqrtf((float)dk);
  const size_t chain_off = ((size_t)cx.n * h_v + cx.h) * dk * dv;
  auto elem_ok = [&](int r, int c) { return lane + 32 * r < dk && cx.j0 + jw + c < dv; };
  float G[kRows][kCW], H[kRows][kCW];
#pragma unroll
  for (int r = 0; r < kRows; ++r)
#pragma unroll
    for (int c = 0; c < kCW; ++c)
      G[r][c] = (p.dfinal_state && elem_ok(r, c))
                    ? p.dfinal_state[chain_off + (size_t)(lane + 32 * r) * dv + cx.j0 + jw + c] : 0.0f;
  float *hs = ws.hs + (((size_t)cx.n * h_v + cx.h) * ws.slices + cx.sl) * (kB + 1) * kSliceThreads * kSlot;
  for (int b = cx.nblk - 1; b >= 0; --b) {
    const int t0 = cx.s0 + kB * b, nt = min(kB, cx.s1 - t0);
    __syncthreads();
    block_prologue(p, ws, dk, cx.h, cx.hq, t0, nt, cx.j0, sq, sk, sv, salpha, sbeta);
    {  // do of the slice's columns, float4 copies (all of them in flight)
      constexpr int kQuads = kB * kSliceCols / 4, kPer = (kQuads + kSliceThreads - 1) / kSliceThreads;
      float4 dv4[kPer];
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int e = tid + kSliceThreads * u, tt = e / (kSliceCols / 4), jj = cx.j0 + 4 * (e % (kSliceCols / 4));
        dv4[u] = (e < kQuads && tt < nt && jj < dv)
                     ? *reinterpret_cast<const float4 *>(ws.wdo + ((size_t)(t0 + tt) * h_v + cx.h) * dv + jj)
                     : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
#pragma unroll
      for (int u = 0; u < kPer; ++u)
        if (tid + kSliceThreads * u < kQuads) reinterpret_cast<float4 *>(sdo)[tid + kSliceThreads * u] = dv4[u];
    }
    load_state(slice_ptr(ws.ckpt, ((size_t)(cx.slot0 + b) * h_v + cx.h) * ws.slices + cx.sl), H);
    for (int tt = 0; tt < nt; ++tt) {  // the block's states again (before each token)
      store_state(slice_ptr(hs, tt), H);
      fwd_step(H, tt, dk, jw, dv - cx.j0, sq, sk, sv, salpha, sbeta, scale, nullptr);
    }
    __syncthreads();
    // H holds the state after the block; the state before token tt is loaded one token ahead (each
    // thread reads back only values it wrote itself)
    float Ht[kRows][kCW], Hp[kRows][kCW];
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
      for (int c = 0; c < kCW; ++c) Ht[r][c] = H[r][c];
    load_state(slice_ptr(hs, nt - 1), Hp);
    for (int tt = nt - 1; tt >= 0; --tt) {
      const size_t tok = (size_t)(t0 + tt) * h_v + cx.h;
      float *red_q = red + (tt & 1) * kRedFloats, *red_k = red_q + kSliceWarps * 128;
      float *red_s = red_k + kSliceWarps * 128;
      float Hn[kRows][kCW];  // the state before token tt - 1, in flight over this step
      load_state(slice_ptr(hs, tt > 0 ? tt - 1 : 0), Hn);
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
        doc[c] = sdo[tt * kSliceCols + jw + c];
        vc[c] = sv[tt * kSliceCols + jw + c];
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
        dkp[r] = 0.0f;
      }
      float pc[kCW], du[kCW];
      {  // the column sums, all of the warp's at once (reduce-scatter, then broadcast)
        float a[kCW], d[kCW];
#pragma unroll
        for (int c = 0; c < kCW; ++c) {
          a[c] = 0.0f;
          d[c] = 0.0f;
#pragma unroll
          for (int r = 0; r < kRows; ++r) {
            a[c] = fmaf(Hp[r][c], kr[r], a[c]);
            d[c] = fmaf(G[r][c], kr[r], d[c]);
          }
        }
        const float as = reduce_scatter<kCW>(a, lane), ds = reduce_scatter<kCW>(d, lane);
#pragma unroll
        for (int c = 0; c < kCW; ++c) {
          pc[c] = __shfl_sync(0xffffffffu, as, kColLanes * c);
          du[c] = __shfl_sync(0xffffffffu, ds, kColLanes * c);
        }
      }
      float s_db = 0.0f, s_dup = 0.0f, dp[kCW];
#pragma unroll
      for (int c = 0; c < kCW; ++c) {
        const float u = be * (vc[c] - al * pc[c]);
        s_db = fmaf(du[c], vc[c] - al * pc[c], s_db);
        s_dup = fmaf(du[c], pc[c], s_dup);
        dp[c] = -al * be * du[c];
#pragma unroll
        for (int r = 0; r < kRows; ++r) dkp[r] = fmaf(G[r][c], u, dkp[r]);
      }
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
#pragma unroll
        for (int c = 0; c < kCW; ++c) {
          dkp[r] = fmaf(Hp[r][c], dp[c], dkp[r]);
          G[r][c] = fmaf(kr[r], dp[c], al * G[r][c]);
        }
      }
#pragma unroll
      for (int c = 0; c < kCW; ++c)
        if (lane == c && cx.j0 + jw + c < dv) ws.dvs[tok * dv + cx.j0 + jw + c] = be * du[c];
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
      for (int i = tid; i < dk; i += kSliceThreads) {  // this slice's part of the sums over columns
        float a = 0.0f, c2 = 0.0f;
#pragma unroll
        for (int w = 0; w < kSliceWarps; ++w) {
          a += red_q[w * 128 + i];
          c2 += red_k[w * 128 + i];
        }
        atomicAdd(&ws.dqn[tok * dk + i], a);
        atomicAdd(&ws.dkn[tok * dk + i], c2);
      }
      if (tid == kSliceThreads - 32) {  // a lane of the last warp: the scalar sums
        float dal = 0.0f, db = 0.0f, dup = 0.0f;
#pragma unroll
        for (int w = 0; w < kSliceWarps; ++w) {
          dal += red_s[w * 4 + 0];
          db += red_s[w * 4 + 1];
          dup += red_s[w * 4 + 2];
        }
        atomicAdd(&ws.dg[tok], al * (dal - be * dup));  // linear in the slice's parts
        atomicAdd(&ws.dbeta[tok], db);
      }
#pragma unroll
      for (int r = 0; r < kRows; ++r)
#pragma unroll
        for (int c = 0; c < kCW; ++c) {
          Ht[r][c] = Hp[r][c];
          Hp[r][c] = Hn[r][c];
        }
    }
  }
  if (p.dinit_state) {
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
      for (int c = 0; c < kCW; ++c)
        if (elem_ok(r, c)) p.dinit_state[chain_off + (size_t)(lane + 32 * r) * dv + cx.j0 + jw + c] = G[r][c];
  }
}

constexpr int kTile = 64;

// per (token tile, conv head): conv head y < h_qk is q head y, then the k
// heads, then the value heads; thread c = channel c of the head (d <= 128).
template <typename IO>
__global__ void __launch_bounds__(128) bwd_prologue_kernel(const BwdParams p, const BwdWs ws) {
  const int h_v = p.h_v, h_qk = p.h_qk, dk = p.d_k, dv = p.d_v, rep = h_v / h_qk;
  const int t0 = blockIdx.x * kTile, y = blockIdx.y, c = threadIdx.x;
  __shared__ float sdp[kTile + 3][128];
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
  // d pre of tokens [t0, t0 + kTile + 3) (the ones the tile's inputs feed): one warp per token, lane l
  // taking channels l + 32 m, so the L2 norm's two sums over the head are warp sums (no block barrier)
  {
    const int warp = c >> 5, lane = c & 31;
    float wm[4][4];  // conv taps of this lane's channels
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
      for (int j = 0; j < 4; ++j) wm[m][j] = lane + 32 * m < D ? p.conv_w[(size_t)(cb + lane + 32 * m) * 4 + j] : 0.f;
    for (int tt = warp; tt < kTile + 3; tt += 4) {
      const int t = t0 + tt;
      if (t >= p.T) break;  // uniform over the warp
      const SeqOf sq = seq_of(p.cu_seqlens, p.N, t);
      float pre[4], xh[4], dsl[4];
      float ss = 0.0f;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int ch = lane + 32 * m;
        pre[m] = 0.0f;
        if (ch < D)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int tau = t - 3 + j;
            if (tau >= sq.s0) pre[m] = fmaf(wm[m][j], to_f(src[(size_t)tau * stride + ch]), pre[m]);
          }
        const float sg = sigmoid_f(pre[m]);
        xh[m] = ch < D ? pre[m] * sg : 0.0f;
        dsl[m] = sg * (1.0f + pre[m] * (1.0f - sg));
        ss = fmaf(xh[m], xh[m], ss);
      }
      float dxh[4];
      if (is_q || is_k) {
        const float *gsrc = is_q ? ws.dqn : ws.dkn;
        float gsum[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int ch = lane + 32 * m;
          gsum[m] = 0.0f;
          if (ch < D)
            for (int r = 0; r < rep; ++r) gsum[m] += gsrc[((size_t)t * h_v + hq * rep + r) * dk + ch];
        }
        const float nrm = sqrtf(warp_sum(ss) + kEpsL2);
        float yg = 0.0f;
#pragma unroll
        for (int m = 0; m < 4; ++m) yg = fmaf(xh[m] / nrm, gsum[m], yg);
        yg = warp_sum(yg);
#pragma unroll
        for (int m = 0; m < 4; ++m) dxh[m] = (gsum[m] - (xh[m] / nrm) * yg) / nrm;
      } else {
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int ch = lane + 32 * m;
          dxh[m] = ch < D ? ws.dvs[((size_t)t * h_v + hvv) * dv + ch] : 0.0f;
        }
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) sdp[tt][lane + 32 * m] = lane + 32 * m < D ? dxh[m] * dsl[m] : 0.0f;
    }
  }
  __syncthreads();
  if (!act) return;
  float dw[4] = {0.f, 0.f, 0.f, 0.f};
  const int Tc = p.T;
  for (int tt = 0; tt < kTile; ++tt) {
    const int t = t0 + tt;
    if (t >= Tc) break;
    const SeqOf sq = seq_of(p.cu_seqlens, p.N, t);
    float acc = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int tp = t + 3 - j;  // the output token that reads input t through tap j
      if (tp < sq.s1) acc = fmaf(sdp[tt + 3 - j][c], w[j], acc);
      const int tau = t - 3 + j;  // the input tap j of output t reads
      if (tau >= sq.s0) dw[j] = fmaf(sdp[tt][c], to_f(src[(size_t)tau * stride + c]), dw[j]);
    }
    dx[(size_t)t * stride + c] = acc;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) atomicAdd(&ws.acc[(size_t)(cb + c) * 4 + j], (double)dw[j]);
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
  double *acc_g = ws.acc + (size_t)(2 * p.h_qk * p.d_k + p.h_v * p.d_v) * 4;  // A_log [h_v], dt_bias [h_v]
  atomicAdd(&acc_g[h], (double)(dg * gate_g(a, A_exp, p.dt_bias[h])));
  atomicAdd(&acc_g[p.h_v + h], (double)da);
}

// The parameter gradients, from their fp64 sums.
__global__ void __launch_bounds__(256) bwd_param_kernel(const BwdParams p, const BwdWs ws) {
  const int Cc = 2 * p.h_qk * p.d_k + p.h_v * p.d_v;
  const int n = Cc * 4 + 2 * p.h_v + p.d_v;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const float v = (float)ws.acc[i];
    if (i < Cc * 4) p.dconv_w[i] = v;
    else if (i < Cc * 4 + p.h_v) p.dA_log[i - Cc * 4] = v;
    else if (i < Cc * 4 + 2 * p.h_v) p.ddt_bias[i - Cc * 4 - p.h_v] = v;
    else p.dnorm_w[i - Cc * 4 - 2 * p.h_v] = v;
  }
}

}  // namespace

size_t prefill_backward_workspace_bytes(int T, int N, int h_qk, int h_v, int d_k, int d_v) {
  return BwdLayout(T, N, h_qk, h_v, d_k, d_v).total;
}

cudaError_t launch_prefill_backward(const BwdParams &p, bool bf16, cudaStream_t s) {
  const BwdLayout L(p.T, p.N, p.h_qk, p.h_v, p.d_k, p.d_v);
  if (p.ws_bytes < L.total) return cudaErrorInvalidValue;
  BwdWs ws;
  ws.ckpt = reinterpret_cast<float *>(p.ws + L.ckpt);
  ws.hs = reinterpret_cast<float *>(p.ws + L.hs);
  ws.wo = reinterpret_cast<float *>(p.ws + L.wo);
  ws.wdo = reinterpret_cast<float *>(p.ws + L.wdo);
  ws.xq = reinterpret_cast<float *>(p.ws + L.xq);
  ws.xk = reinterpret_cast<float *>(p.ws + L.xk);
  ws.xv = reinterpret_cast<float *>(p.ws + L.xv);
  ws.xal = reinterpret_cast<float *>(p.ws + L.xal);
  ws.xbe = reinterpret_cast<float *>(p.ws + L.xbe);
  ws.dqn = reinterpret_cast<float *>(p.ws + L.dqn);
  ws.dkn = reinterpret_cast<float *>(p.ws + L.dkn);
  ws.dvs = reinterpret_cast<float *>(p.ws + L.dvs);
  ws.dg = reinterpret_cast<float *>(p.ws + L.dg);
  ws.dbeta = reinterpret_cast<float *>(p.ws + L.dbeta);
  ws.acc = reinterpret_cast<double *>(p.ws + L.acc);
  ws.slices = L.slices;
  cudaError_t e;
  // the per-token q, k and gate gradients and the parameter gradients' fp64 sums are atomic adds
  if ((e = cudaMemsetAsync(p.ws + L.dqn, 0, L.total - L.dqn, s)) != cudaSuccess) return e;
  const size_t smem = sizeof(float) * slice_smem_floats(p.d_k);
  const unsigned ctas = (unsigned)p.N * (unsigned)p.h_v * (unsigned)L.slices;
  // the RMSNormGated reverse: 8 rows per CTA at a time, at most 8 CTAs per SM on 152 SMs (each CTA adds
  // its dnorm_w sums once)
  const unsigned rows = (unsigned)std::min<size_t>(((size_t)p.T * p.h_v + 7) / 8, (size_t)152 * 8);
  const dim3 pgrid((unsigned)((p.T + kTile - 1) / kTile), (unsigned)(2 * p.h_qk + p.h_v));
  const unsigned ggrid = (unsigned)(((size_t)p.T * p.h_v + 255) / 256);
  const unsigned irows =
      (unsigned)(((size_t)p.T * (2 * p.h_qk + p.h_v) + kTokenRowsPerCta - 1) / kTokenRowsPerCta);
  TokenInputs ti{};
  ti.q = p.q; ti.k = p.k; ti.v = p.v; ti.a = p.a; ti.b = p.b;
  ti.conv_w = p.conv_w; ti.A_log = p.A_log; ti.dt_bias = p.dt_bias; ti.cu_seqlens = p.cu_seqlens;
  ti.init_conv = nullptr;  // the backward's forward starts every sequence from a zero conv history
  ti.T = p.T; ti.N = p.N; ti.h_qk = p.h_qk; ti.h_v = p.h_v; ti.d_k = p.d_k; ti.d_v = p.d_v;
  ti.xq = ws.xq; ti.xk = ws.xk; ti.xv = ws.xv; ti.xal = ws.xal; ti.xbe = ws.xbe;
  // the token-sequential kernels come in two forms: d_k = 128 fixed at compile time, and any d_k
  auto run = [&](auto in_k, auto fwd_k128, auto fwd_k, auto norm_k, auto rev_k128, auto rev_k, auto pro_k,
                 auto gate_k) -> cudaError_t {
    if (p.d_k == 128) {
      fwd_k = fwd_k128;
      rev_k = rev_k128;
    }
    cudaError_t err = cudaFuncSetAttribute(fwd_k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    if ((err = cudaFuncSetAttribute(rev_k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
      return err;
    if (ctas) {
      trace_begin(s, GDN_K_BWD_CHAIN);
      if (p.T > 0) in_k<<<irows, 32 * kTokenRowsPerCta, 0, s>>>(ti);
      fwd_k<<<ctas, kSliceThreads, smem, s>>>(p, ws);
      if (p.T > 0) norm_k<<<rows, 256, 0, s>>>(p, ws);
      rev_k<<<ctas, kSliceThreads, smem, s>>>(p, ws);
      trace_end(s);
      if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    if (p.T > 0) {
      trace_begin(s, GDN_K_BWD_PROLOGUE);
      pro_k<<<pgrid, 128, 0, s>>>(p, ws);
      trace_end(s);
      if ((err = cudaGetLastError()) != cudaSuccess) return err;
      gate_k<<<ggrid, 256, 0, s>>>(p, ws);
    }
    bwd_param_kernel<<<64, 256, 0, s>>>(p, ws);
    return cudaGetLastError();
  };
  if (bf16)
    return run(token_inputs_kernel<__nv_bfloat16>, bwd_fwd_kernel<__nv_bfloat16, 128>, bwd_fwd_kernel<__nv_bfloat16, 0>,
               bwd_norm_kernel<__nv_bfloat16>, bwd_rev_kernel<__nv_bfloat16, 128>, bwd_rev_kernel<__nv_bfloat16, 0>,
               bwd_prologue_kernel<__nv_bfloat16>, bwd_gate_kernel<__nv_bfloat16>);
  return run(token_inputs_kernel<float>, bwd_fwd_kernel<float, 128>, bwd_fwd_kernel<float, 0>, bwd_norm_kernel<float>,
             bwd_rev_kernel<float, 128>, bwd_rev_kernel<float, 0>, bwd_prologue_kernel<float>,
             bwd_gate_kernel<float>);
}

}  // namespace gdn
