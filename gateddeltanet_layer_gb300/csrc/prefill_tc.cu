// Chunked prefill on the 5th-generation tensor cores (bf16 streams, d_k = d_v = 128).
//
// The chunked WY/UT form of the gated delta rule (Yang et al., "Gated Delta
// Networks", ICLR 2025; "Parallelizing Linear Transformers with the Delta Rule
// over Sequence Length", NeurIPS 2024).  A sequence is cut into chunks of
// C = 64 tokens.  With G_r the running sum of the gates g inside a chunk,
// gamma_r = exp(G_r), H = S^T the state entering the chunk (d_k x d_v):
//
//   A   = strict_lower(beta_r e^(G_r - G_s) k_r.k_s),   T = (I + A)^-1
//   U   = T diag(beta) V - T diag(beta gamma) K H         (row r = the u_r of the rule)
//   O   = d_k^-1/2 (diag(gamma) Q H + (Q K^T o D) U),       D_rs = e^(G_r - G_s), s <= r
//   H  <- gamma_C H + K~^T U,                               K~ = diag(e^(G_C - G)) K
//   y   = RMSNorm(O) w silu(z)
//
// Everything that does not depend on H is computed for all chunks at once, and
// only the H-dependent products run sequentially per chain:
//
//   chunk_table_kernel  cu_seqlens -> chunk list (sequence, first token) and
//                       each sequence's first chunk; validates cu_seqlens.
//   chunk_prep_kernel   one CTA per (chunk, q/k head), all chunks in parallel:
//                       conv(4) + SiLU + L2 norm of q, k (shared by the value
//                       heads of the q/k head) and v, the gates, P1 = [K; Q] K^T
//                       on the tensor cores, A and A_Q, the blocked inverse T,
//                       and on the tensor cores W = T diag(beta gamma) K and
//                       U' = T diag(beta) V; writes the state pass's operands
//                       ([Q^; W] with Q^ = diag(gamma) Q, K~^T, U', -A_Q,
//                       gamma), already in their shared-memory image.
//   state_kernel        per (sequence, value head) chain a cluster of CTAs,
//                       each owning a slice of the columns of H (d_v), held in
//                       tensor memory.  Per chunk two MMA steps: U = U' - W H
//                       (with -Q^ H in the same 128-row product), then
//                       H <- gamma_C H + K~^T U and O += A_Q U; an epilogue
//                       warp pair forms y, exchanging the per-token sums of
//                       o^2 across the cluster; a producer warp streams the
//                       next chunk's operands in by TMA.
//
// Every dense contraction is a tcgen05.mma chain with M = 128 (the transposed
// forms keep M at d_k or d_v), fp16 operands in 128-byte-swizzled K-major
// shared memory, fp32 accumulators in tensor memory; one thread issues,
// tcgen05.commit signals an mbarrier, and every wait is bounded.  Decays
// between two tokens are always exp(G_r - G_s) with r >= s.
//
// Operand precision.  Every computed operand is rounded to fp16 (3 more
// mantissa bits than bf16, same MMA rate and size).  The per-token RMSNorm
// magnifies the rounding error of rows whose o is small: with bf16 operands
// single outputs drifted by up to 6 % of max(1, |y|), with fp16 by under 1 %.
// All operands are bounded well inside the fp16 range (|x| <= ~4: unit-norm
// q, k, the SiLU-conv'd v of O(1) inputs, T diag(beta), W and the state).  The
// q.k and k.k products of P1 use a hi + lo split (P1 = hi.hi + hi.lo + lo.hi),
// which recovers ~22 bits for A and A_Q.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "gdn_common.cuh"
#include "../../include/gdn_trace.h"
#include "gdn_internal.h"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

constexpr int kC = 64;
constexpr int kD = 128;
constexpr int kPad = 66;  // fp32 64 x 64 matrices: padded rows (even: 8-byte aligned pairs)

// ---------------------------------------------------------------- workspace
// Per (chunk, value head), operand images the state pass copies straight into
// shared memory (fp16; SW128 K-major unless noted):
//   [Q^; W]  [128 rows][128 cols]: rows 0-63 Q^ = diag(gamma) Q, rows 64-127
//            W = T diag(beta gamma) K (one 128-row MMA operand)
//   K~^T     [128 i][64 m] = (diag(e^(G_C - G)) K)^T
//   U'       T diag(beta) V, plain row-major per state slice: [4][64 m][32]
//            (32 = the state pass's slice width)
//   -A_Q     [64 r][64 s], A_Q = D o (Q K^T), lower triangle with the diagonal
//   gamma    [64] fp32
constexpr uint32_t kVWQ = 0, kVKt = 32768, kVUp = 49152, kVAq = 65536, kVGam = 73728;
constexpr uint32_t kVSlot = 73984;
// The compact images of the one-CTA-per-chain state pass: nothing per value
// head that depends only on the q/k head.  Per (chunk, value head):
//   W        2 slabs x [64 rows][64 cols] (SW128), 16 KB
//   U'       as above, [4][64 m][32]
//   -A_Q     as above
//   gamma    [64] fp32;  decay-to-end e^(G_C - G_m) [64] fp32
// and per (chunk, q/k head): Q (2 slabs x [64][64], SW128, unscaled) and the
// K^T tile [128 i][64 m] (SW128) -- the state pass applies gamma to Q H and
// the decay to U itself.
constexpr uint32_t kCW = 0, kCUp = 16384, kCAq = 32768, kCGam = 40960, kCDec = 41216;
constexpr uint32_t kCSlot = 41472;
constexpr uint32_t kQQ = 0, kQKt = 16384, kQSlot = 32768;
static_assert(kCSlot % 256 == 0 && kCDec + 256 == kCSlot, "compact value-head slot");

struct Ws {
  int *chunk_base;   // [N + 1]: first chunk of each sequence; [N] = number of chunks
  int *seq_order;    // [N]: the sequences, longest first (by powers of two of their chunk counts); N > 1
  int4 *chunk_info;  // [max_chunks]: (sequence, first token, sequence start, tokens in the chunk)
  uint8_t *vs;       // [max_chunks][h_v] x kVSlot, or (compact) x kCSlot
  uint8_t *qs;       // compact: [max_chunks][h_qk] x kQSlot (after the value-head slots)
  int max_chunks;
  int compact;       // the images are the compact ones (one-CTA-per-chain state pass)
  const struct SegRun *runs;  // segment-parallel prefill: the state pass's chains (else null)
};

// One chain of the segment-parallel prefill's state passes: tokens [s0, s1)
// (chunk images from g0 on) of value head blockIdx.x % h_v.  The state starts
// from init (+ h * d_k * d_v; null: zeros) or, with kRunTransfer, from the
// identity with U' taken as zero (the segment's transfer matrix), and ends in
// final (+ h * d_k * d_v; may be null); with kRunOut the epilogue writes y.
enum : int { kRunOut = 1, kRunTransfer = 2 };
struct SegRun {
  int s0, s1, g0, flags;
  const float *init;
  float *final;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WsLayout {
  size_t base, order, info, vs, total;
  int max_chunks;
  WsLayout(int T, int N, int h_qk, int h_v) {
    max_chunks = (T + kC - 1) / kC + N;
    base = 0;
    order = align_up(sizeof(int) * (size_t)(N + 1), 256);
    info = align_up(order + sizeof(int) * (size_t)N, 1024);
    vs = align_up(info + sizeof(int4) * (size_t)max_chunks, 1024);
    // the larger of the two image layouts (split pass: kVSlot per value head; compact: kCSlot per
    // value head and kQSlot per q/k head)
    const size_t split = (size_t)h_v * kVSlot, compact = (size_t)h_v * kCSlot + (size_t)h_qk * kQSlot;
    total = vs + (size_t)max_chunks * (split > compact ? split : compact);
  }
};

// ---------------------------------------------------------------- helpers
__device__ __forceinline__ void mma_chain(uint32_t d, uint32_t a, int a_rows, int a_row0, uint32_t b, int b_rows,
                                          int b_row0, int ksteps, uint32_t idesc, bool acc) {
  for (int k = 0; k < ksteps; ++k)
    tc::mma16(d, tc::sdesc_kstep(a, a_rows, a_row0, k), tc::sdesc_kstep(b, b_rows, b_row0, k), idesc,
              (acc || k > 0) ? 1u : 0u);
}


// SiLU of a pair: x sigmoid(x) = h + h tanh(h), h = x / 2, with the hardware
// tanh (tanh.approx: absolute error about 2^-11, so |error| <= ~2^-11 |h|).
// Two multi-function-unit operations per pair instead of four (2^x and 1/x
// twice); on the prefill workloads the outputs' error against the oracle
// moved by under 1e-3 of the bound, and the prep ran 3 % faster.
constexpr float kLog2e = 1.4426950408889634f;
__device__ __forceinline__ float2 silu2(float2 x) {
  const float2 hx = tc::mul2(x, tc::splat2(0.5f));
  return tc::fma2(hx, make_float2(tc::tanh_approx(hx.x), tc::tanh_approx(hx.y)), hx);
}

__device__ __forceinline__ bool wait_all(uint64_t *bar, uint32_t &phase) {
  const bool ok = tc::mbar_wait(bar, phase & 1);
  ++phase;
  tc::fence_after_sync();
  return __syncthreads_or(!ok) != 0;
}

__device__ __forceinline__ void publish_operands() {
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
}

__device__ __forceinline__ uint2 pack4_f16(float a, float b, float c, float d) {
  return make_uint2(tc::pack_f16x2(a, b), tc::pack_f16x2(c, d));
}

// ================================================================ chunk table
// Chunk-count class of a sequence for the state pass's order: 1 + floor(log2(chunks)), 0 when empty.
__device__ __forceinline__ int length_class(int chunks) { return chunks > 0 ? 32 - __clz(chunks) : 0; }

__global__ void __launch_bounds__(1024) chunk_table_kernel(const PrefillParams p, Ws ws) {
  __shared__ int scan[1024];
  __shared__ int bad;
  __shared__ int cls_next[33];  // sequences per length class, then the next free place of each
  const int N = p.N, tid = threadIdx.x;
  tc::launch_dependents();  // the prep CTAs may take their places; they wait for this table
  if (tid == 0) bad = 0;
  const int per = (N + 1023) / 1024;
  const int n0 = min(N, tid * per), n1 = min(N, n0 + per);
  int cnt = 0;
  for (int n = n0; n < n1; ++n) {
    const int s0 = p.cu_seqlens[n], s1 = p.cu_seqlens[n + 1];
    if (s0 >= 0 && s1 >= s0 && s1 <= p.T) cnt += (s1 - s0 + kC - 1) / kC;
  }
  if (N > 1) {  // the state pass's order: length classes longest first, so long chains start first
    if (tid < 33) cls_next[tid] = 0;
    __syncthreads();
    for (int n = n0; n < n1; ++n) {
      const int s0 = p.cu_seqlens[n], s1 = p.cu_seqlens[n + 1];
      atomicAdd(&cls_next[length_class((s0 >= 0 && s1 >= s0 && s1 <= p.T) ? (s1 - s0 + kC - 1) / kC : 0)], 1);
    }
    __syncthreads();
    if (tid == 0) {
      int at = 0;
      for (int k = 32; k >= 0; --k) {
        const int c = cls_next[k];
        cls_next[k] = at;
        at += c;
      }
    }
    __syncthreads();
    for (int n = n0; n < n1; ++n) {  // the order inside a class does not matter for the results
      const int s0 = p.cu_seqlens[n], s1 = p.cu_seqlens[n + 1];
      const int c = (s0 >= 0 && s1 >= s0 && s1 <= p.T) ? (s1 - s0 + kC - 1) / kC : 0;
      ws.seq_order[atomicAdd(&cls_next[length_class(c)], 1)] = n;
    }
  }
  scan[tid] = cnt;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {  // inclusive scan
    const int v = tid >= off ? scan[tid - off] : 0;
    __syncthreads();
    scan[tid] += v;
    __syncthreads();
  }
  const int total = scan[1023];
  const bool overflow = total > ws.max_chunks;  // only possible with invalid cu_seqlens
  int run = scan[tid] - cnt;
  for (int n = n0; n < n1; ++n) {
    const int s0 = p.cu_seqlens[n], s1 = p.cu_seqlens[n + 1];
    const bool ok = s0 >= 0 && s1 >= s0 && s1 <= p.T;
    if (!ok) bad = 1;
    ws.chunk_base[n] = overflow ? 0 : run;
    if (ok) run += (s1 - s0 + kC - 1) / kC;
  }
  if (tid == 1023) ws.chunk_base[N] = overflow ? 0 : total;
  __syncthreads();
  if (tid == 0 && (bad || overflow)) set_status(p.status, kDevBadSeqlens);
  if (overflow) return;
  for (int g = tid; g < total; g += 1024) {  // sequence of chunk g by binary search
    int lo = 0, hi = N - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (ws.chunk_base[mid] <= g) lo = mid; else hi = mid - 1;
    }
    const int sq0 = p.cu_seqlens[lo], tq0 = sq0 + kC * (g - ws.chunk_base[lo]);
    ws.chunk_info[g] = make_int4(lo, tq0, sq0, min(kC, p.cu_seqlens[lo + 1] - tq0));
  }
}

// ================================================================ chunk prep
constexpr int kPrepThreads = 256;
// Shared memory of the prep kernel (byte offsets; SW128 tiles 1024-aligned).
//   [0, 64K): during the q/k phase the [K; Q] hi and lo fp16 tiles [128][128]
//     (the operands of K K^T and Q K^T).  Once those products are done, for
//     the two value heads of a pair: A, then T = (I + A)^-1 in place, fp32
//     [64][kPad] at P_AT0 / P_AT1, each later overwritten by its
//     [T diag(beta gamma); T diag(beta)] fp16 [128][64]; inverse scratch at
//     P_XF; the second head's V^T fp16 [128 j][64 m] at P_VT1.
//   [64K, 96K): K^T fp16 [128 i][64 m] at P_KT, the first head's V^T at P_VT0.
//   So [K^T; V^T] (first head, from P_KT) and [V^T; K^T] (second head, from
//   P_VT1) are each one 256-row B operand: one MMA gives both W and U'.
constexpr uint32_t P_KQ = 0;
constexpr uint32_t P_KQL = 32768;
constexpr uint32_t P_AT0 = 0, P_AT1 = 17408;
constexpr uint32_t P_XF = 34816;  // per head of the pair 4 KB
constexpr uint32_t P_VT1 = 49152, P_KT = 65536, P_VT0 = 81920;
constexpr int kMaxRep = kTcMaxRep;                    // value heads per q/k head
constexpr uint32_t P_VEC = 98304;                     // per value head: G, gamma, beta, decay-to-end
constexpr uint32_t P_RED = P_VEC + kMaxRep * 1024;
constexpr uint32_t P_MISC = P_RED + 64;
constexpr size_t kPrepSmem = P_MISC + 64 + 1024;
static_assert(P_AT1 >= P_AT0 + 64 * kPad * 4 && P_XF >= P_AT1 + 64 * kPad * 4, "A / T tiles");
static_assert(P_XF + 2 * 4096 <= P_VT1 && P_VT1 + 16384 == P_KT && P_KT + 16384 == P_VT0, "B operands");
static_assert(P_AT1 % 1024 == 0 && P_VT1 % 1024 == 0, "SW128 tiles 1024-aligned");
static_assert(P_VT0 + 16384 <= P_VEC, "regions");
static_assert(2 * (kPrepSmem + 1024) <= 233472, "two prep CTAs per SM");

constexpr uint32_t kIdN64 = tc::idesc_f16(128, 64);
constexpr uint32_t kIdN256 = tc::idesc_f16(128, 256);

// Raw rows for conv(4) of 8 output rows r0 .. r0+7 of the chunk: input rows
// r0-3 .. r0+7, 4 channels (x points at the first channel of token 0; bf16 row
// pitch `stride` elements) as packed bf16; rows past the chunk's end are 0, and
// so are the (at most three) rows before the sequence start unless `hist`
// points at the carried conv history of the 4 channels ([channel][3] bf16,
// oldest first: token s0 - 3 + m at m).  FULL: a whole chunk starting at
// least 3 tokens into its sequence (every row is a plain load).
template <bool FULL>
__device__ __forceinline__ void load_rows(const __nv_bfloat16 *x, size_t stride, int t0, int s0, int Lc, int r0,
                                          const __nv_bfloat16 *hist, uint2 (&xr)[11]) {
#pragma unroll
  for (int rr = 0; rr < 11; ++rr) {
    const int row = r0 - 3 + rr;
    const int t = t0 + row;
    if (FULL) {
      xr[rr] = *reinterpret_cast<const uint2 *>(x + (size_t)t * stride);
    } else if (t >= s0) {
      xr[rr] = row < Lc ? *reinterpret_cast<const uint2 *>(x + (size_t)t * stride) : make_uint2(0u, 0u);
    } else if (hist) {  // t >= t0 - 3 >= s0 - 3
      const uint16_t *h = reinterpret_cast<const uint16_t *>(hist) + (t - s0 + 3);
      xr[rr] = make_uint2((uint32_t)h[0] | ((uint32_t)h[3] << 16), (uint32_t)h[6] | ((uint32_t)h[9] << 16));
    } else {
      xr[rr] = make_uint2(0u, 0u);
    }
  }
}
// conv(4) + SiLU of the rows of load_rows, channels from conv_w row `ch`;
// channels in pairs, one packed fp32 instruction per pair.  FULL: every row is in the chunk.
template <bool FULL>
__device__ __forceinline__ void conv_silu(const uint2 (&xr)[11], const float *conv_w, int ch, int Lc, int r0,
                                          float (&y)[8][4]) {
  float4 w[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) w[c] = *reinterpret_cast<const float4 *>(conv_w + (size_t)(ch + c) * 4);
  float2 wp[2][4];  // [channel pair][tap]
#pragma unroll
  for (int pr = 0; pr < 2; ++pr) {
    wp[pr][0] = make_float2(w[2 * pr].x, w[2 * pr + 1].x);
    wp[pr][1] = make_float2(w[2 * pr].y, w[2 * pr + 1].y);
    wp[pr][2] = make_float2(w[2 * pr].z, w[2 * pr + 1].z);
    wp[pr][3] = make_float2(w[2 * pr].w, w[2 * pr + 1].w);
  }
  auto pair = [&](int rr, int pr) {  // channels 2 pr, 2 pr + 1 of input row rr (bf16 -> fp32 exactly)
    const uint32_t w32 = pr ? xr[rr].y : xr[rr].x;
    return make_float2(__uint_as_float(w32 << 16), __uint_as_float(w32 & 0xFFFF0000u));
  };
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const bool ok = FULL || r0 + r < Lc;
#pragma unroll
    for (int pr = 0; pr < 2; ++pr) {
      float2 a = tc::mul2(wp[pr][0], pair(r, pr));
      a = tc::fma2(wp[pr][1], pair(r + 1, pr), a);
      a = tc::fma2(wp[pr][2], pair(r + 2, pr), a);
      a = tc::fma2(wp[pr][3], pair(r + 3, pr), a);
      const float2 sv = silu2(a);
      y[r][2 * pr] = ok ? sv.x : 0.0f;
      y[r][2 * pr + 1] = ok ? sv.y : 0.0f;
    }
  }
}

// L2-normalise the 8 rows held by a warp (each lane holds 4 of the 128 channels).
__device__ __forceinline__ void l2norm_rows(float (&y)[8][4], int lane) {
  float ss[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const float2 y01 = make_float2(y[r][0], y[r][1]), y23 = make_float2(y[r][2], y[r][3]);
    const float2 s2 = tc::fma2(y23, y23, tc::mul2(y01, y01));
    ss[r] = s2.x + s2.y;
  }
  const float mine = reduce_scatter<8>(ss, lane);  // lane l: row l >> 2
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const float2 inv = tc::splat2(rsqrtf(__shfl_sync(0xffffffffu, mine, 4 * r) + kEpsL2));
    const float2 y01 = tc::mul2(make_float2(y[r][0], y[r][1]), inv), y23 = tc::mul2(make_float2(y[r][2], y[r][3]), inv);
    y[r][0] = y01.x; y[r][1] = y01.y; y[r][2] = y23.x; y[r][3] = y23.y;
  }
}

// upmap: the U' images as [slot][256 rows][32] fp16 (slot = chunk x h_v + value head), 64-byte swizzle:
// the staging's 16-byte chunk c of row m sits at c ^ ((m >> 1) & 3), the tensor memory accelerator's
// 64-byte pattern, so one 3-D store writes a head's 16 KB.
// NREP: the value heads per q/k head when fixed at compile time (2), else 0 (from p).
template <int NREP>
__global__ void __launch_bounds__(kPrepThreads, 2)
    chunk_prep_kernel(const PrefillParams p, const Ws ws, const __grid_constant__ CUtensorMap upmap) {
  // grid (chunk slots, q/k heads x value-head groups): a CTA takes up to kMaxRep of the value heads
  // of its q/k head (all of them unless h_v / h_qk > kMaxRep, where each group redoes the q/k part)
  const int ngrp = NREP ? 1 : (p.h_v / p.h_qk + kMaxRep - 1) / kMaxRep;
  const int g = blockIdx.x, hq = blockIdx.y / ngrp, vbase = kMaxRep * (blockIdx.y % ngrp);
  tc::grid_dependency_wait();  // the chunk table
  tc::launch_dependents();     // the state pass may be scheduled once every prep CTA has started
  const int total = ws.chunk_base[p.N];
  if (g >= total) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sbase = tc::smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int lr = tid & 127, gh = tid >> 7;
  const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
  const int h_v = p.h_v, h_qk = p.h_qk, rep = NREP ? NREP : h_v / h_qk, nrep = NREP ? NREP : min(kMaxRep, rep - vbase);
  const bool qk_images = vbase == 0;  // the group that writes the per-q/k-head images
  // TMEM: the 256-column W / U' accumulator at column 0; K K^T and Q K^T (64
  // columns) under it when the value heads come as one pair (their A is taken
  // before the first W / U' product), else beside it
  const uint32_t tmem_cols = nrep <= 2 ? 256u : 512u;
  const int COL_P1 = nrep <= 2 ? 0 : 256;

  const int4 info = ws.chunk_info[g];
  const int t0 = info.y, s0 = info.z, Lc = info.w;
  const bool full = Lc == kC && t0 - 3 >= s0;  // a whole chunk with no sequence start in its conv window
  // conv history of channel ch for this thread's 4 channels (only the first chunk of a sequence reads it)
  const size_t conv_ch = 2 * (size_t)h_qk * kD + (size_t)h_v * kD;
  const __nv_bfloat16 *hist0 =
      (p.init_conv && t0 == s0) ? static_cast<const __nv_bfloat16 *>(p.init_conv) + (size_t)info.x * conv_ch * 3 : nullptr;
  auto hist = [&](int ch) { return hist0 ? hist0 + (size_t)ch * 3 : nullptr; };

  // per value head vv: G at sG[256 vv], gamma at +64, beta at +128, decay-to-end at +192
  float *sG = reinterpret_cast<float *>(sm + P_VEC);
  float *const sGall = sG;
  float *carry = reinterpret_cast<float *>(sm + P_RED);
  uint64_t *bar = reinterpret_cast<uint64_t *>(sm + P_MISC);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + P_MISC + 8);

  const __nv_bfloat16 *xq = static_cast<const __nv_bfloat16 *>(p.q);
  const __nv_bfloat16 *xk = static_cast<const __nv_bfloat16 *>(p.k);
  const __nv_bfloat16 *xv = static_cast<const __nv_bfloat16 *>(p.v);
  const __nv_bfloat16 *xa = static_cast<const __nv_bfloat16 *>(p.a);
  const __nv_bfloat16 *xb = static_cast<const __nv_bfloat16 *>(p.b);
  const size_t qk_stride = (size_t)h_qk * kD, v_stride = (size_t)h_v * kD;

  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, tmem_cols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(bar, 1);
    tc::fence_mbar_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  uint32_t phase = 0;
  bool failed = false;

  const int r0 = 8 * warp, c0 = 4 * lane;  // conv: this thread's rows and channels
  const bool compact = ws.compact != 0;
  auto v_slot_of = [&](int vv) {
    return ws.vs + ((size_t)g * h_v + hq * rep + vbase + vv) * (compact ? kCSlot : kVSlot);
  };
  uint8_t *const q_slot = ws.qs + ((size_t)g * h_qk + hq) * kQSlot;  // compact only

  // the v rows of the first pair into L2 while the q/k rows are worked on
  auto prefetch_v = [&](int vv) {
    const int t = t0 - 3 + tid;
    if (tid < kC + 3 && t >= s0 && t < t0 + Lc)
      tc::prefetch_l2(xv + (size_t)t * v_stride + (size_t)(hq * rep + vbase + vv) * kD, kD * 2);
  };
  prefetch_v(0);

  // the q and k rows of the conv: loads in flight over the gates below
  uint2 xrq[11], xrk[11];
  if (full) {
    load_rows<true>(xq + hq * kD + c0, qk_stride, t0, s0, Lc, r0, nullptr, xrq);
    load_rows<true>(xk + hq * kD + c0, qk_stride, t0, s0, Lc, r0, nullptr, xrk);
  } else {
    load_rows<false>(xq + hq * kD + c0, qk_stride, t0, s0, Lc, r0, hist(hq * kD + c0), xrq);
    load_rows<false>(xk + hq * kD + c0, qk_stride, t0, s0, Lc, r0, hist(h_qk * kD + hq * kD + c0), xrk);
  }

  // ---------------- gates of every value head and their running sums inside the chunk
  for (int v0 = 0; v0 < nrep; v0 += 4) {
    const int vv = v0 + (tid >> 6), r = tid & 63;
    float gsum = 0.0f;
    if (vv < nrep) {
      const int h = hq * rep + vbase + vv;
      float gg = 0.0f, be = 0.0f;
      if (r < Lc) {
        const size_t gi = (size_t)(t0 + r) * h_v + h;
        gg = gate_g(__bfloat162float(xa[gi]), expf(p.A_log[h]), p.dt_bias[h]);
        be = sigmoid_f(__bfloat162float(xb[gi]));
      }
      gsum = gg;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, gsum, off);
        if (lane >= off) gsum += y;
      }
      if (r == 31) carry[vv & 3] = gsum;
      sG[vv * 256 + 128 + r] = be;
    }
    __syncthreads();
    if (vv < nrep) {
      if (r >= 32) gsum += carry[vv & 3];
      sG[vv * 256 + r] = gsum;
      const float gm = expf(gsum);
      sG[vv * 256 + 64 + r] = gm;
      *reinterpret_cast<float *>(v_slot_of(vv) + (compact ? kCGam : kVGam) + 4 * r) = gm;
    }
    __syncthreads();
    if (vv < nrep) {
      const float dec = expf(sG[vv * 256 + 63] - sG[vv * 256 + r]);
      sG[vv * 256 + 192 + r] = dec;
      if (compact) *reinterpret_cast<float *>(v_slot_of(vv) + kCDec + 4 * r) = dec;
    }
    __syncthreads();
  }

  // ---------------- q and k: conv + SiLU + L2 norm -> [K; Q] hi / lo tiles, K^T tile, Q^ images
  {
    float y[8][4], kreg[8][4];
    {
      if (nrep > 1) prefetch_v(1);
      if (full) conv_silu<true>(xrq, p.conv_w, hq * kD + c0, Lc, r0, y);
      else conv_silu<false>(xrq, p.conv_w, hq * kD + c0, Lc, r0, y);
    }
    l2norm_rows(y, lane);
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const uint2 hi = pack4_f16(y[r][0], y[r][1], y[r][2], y[r][3]);
      const __half2 h01 = *reinterpret_cast<const __half2 *>(&hi.x), h23 = *reinterpret_cast<const __half2 *>(&hi.y);
      const uint2 lo = pack4_f16(y[r][0] - __low2float(h01), y[r][1] - __high2float(h01),
                                 y[r][2] - __low2float(h23), y[r][3] - __high2float(h23));
      const uint32_t off = tc::sw128_offset(128, 64 + r0 + r, c0);
      *reinterpret_cast<uint2 *>(sm + P_KQ + off) = hi;
      *reinterpret_cast<uint2 *>(sm + P_KQL + off) = lo;
    }
    if (compact) {
      // Q, once per q/k head: its two 64-row SW128 slabs are rows 64-127 of the hi tile's slabs (the same
      // fp16 values, the same swizzle), copied below
    } else {
      for (int vv = 0; vv < nrep; ++vv) {  // Q^ = diag(gamma) Q: rows 0-63 of the [Q^; W] image
        const float *gam = sG + vv * 256 + 64;
        uint8_t *dst = v_slot_of(vv) + kVWQ;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const float2 gr = tc::splat2(gam[r0 + r]);
          const float2 q01 = tc::mul2(gr, make_float2(y[r][0], y[r][1])),
                       q23 = tc::mul2(gr, make_float2(y[r][2], y[r][3]));
          *reinterpret_cast<uint2 *>(dst + tc::sw128_offset(128, r0 + r, c0)) = pack4_f16(q01.x, q01.y, q23.x, q23.y);
        }
      }
    }
    if (full) conv_silu<true>(xrk, p.conv_w, h_qk * kD + hq * kD + c0, Lc, r0, kreg);
    else conv_silu<false>(xrk, p.conv_w, h_qk * kD + hq * kD + c0, Lc, r0, kreg);
    l2norm_rows(kreg, lane);
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const uint2 hi = pack4_f16(kreg[r][0], kreg[r][1], kreg[r][2], kreg[r][3]);
      const __half2 h01 = *reinterpret_cast<const __half2 *>(&hi.x), h23 = *reinterpret_cast<const __half2 *>(&hi.y);
      const uint2 lo = pack4_f16(kreg[r][0] - __low2float(h01), kreg[r][1] - __high2float(h01),
                                 kreg[r][2] - __low2float(h23), kreg[r][3] - __high2float(h23));
      const uint32_t off = tc::sw128_offset(128, r0 + r, c0);
      *reinterpret_cast<uint2 *>(sm + P_KQ + off) = hi;
      *reinterpret_cast<uint2 *>(sm + P_KQL + off) = lo;
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {  // K^T tile (the K half of the B operand of W)
      float kt[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) kt[r] = kreg[r][c];
      tc::st_chunk_f16(sm + P_KT + tc::sw128_chunk(128, c0 + c, warp), kt);
    }
  }
  publish_operands();

  // ---------------- P1 = [K; Q] K^T (hi.hi + hi.lo + lo.hi): rows 0..63 K K^T, 64..127 Q K^T
  if (tid == 0) {
    mma_chain(tmem + COL_P1, sbase + P_KQ, 128, 0, sbase + P_KQ, 128, 0, 8, kIdN64, false);
    mma_chain(tmem + COL_P1, sbase + P_KQ, 128, 0, sbase + P_KQL, 128, 0, 8, kIdN64, true);
    mma_chain(tmem + COL_P1, sbase + P_KQL, 128, 0, sbase + P_KQ, 128, 0, 8, kIdN64, true);
    tc::mma_commit(bar);
    if (compact && qk_images) {  // the per-q/k-head images: Q (from the hi tile) and the K^T tile
      tc::bulk_s2g(q_slot + kQQ, sm + P_KQ + 8192, 8192);
      tc::bulk_s2g(q_slot + kQQ + 8192, sm + P_KQ + 16384 + 8192, 8192);
      tc::bulk_s2g(q_slot + kQKt, sm + P_KT, 16384);
      tc::bulk_commit();
    }
  }

  // ---------------- the value heads, two at a time
  for (int grp = 0; grp < nrep && !failed; grp += 2) {
    const int nh = min(2, nrep - grp);
    auto AT = [&](int hh) { return reinterpret_cast<float *>(sm + (hh ? P_AT1 : P_AT0)); };
    auto XF = [&](int hh) { return reinterpret_cast<float *>(sm + P_XF + (hh ? 4096 : 0)); };

    // v: conv + SiLU -> V^T tiles; both heads' rows in flight at once
    {
      uint2 xr[11];
      float y[8][4];
      const int vch0 = 2 * h_qk * kD + (hq * rep + vbase + grp) * kD + c0;  // conv channel of the first head
      if (full) {
        load_rows<true>(xv + (size_t)(hq * rep + vbase + grp) * kD + c0, v_stride, t0, s0, Lc, r0, nullptr, xr);
        conv_silu<true>(xr, p.conv_w, vch0, Lc, r0, y);
      } else {
        load_rows<false>(xv + (size_t)(hq * rep + vbase + grp) * kD + c0, v_stride, t0, s0, Lc, r0, hist(vch0), xr);
        conv_silu<false>(xr, p.conv_w, vch0, Lc, r0, y);
      }
      // the second head's rows in flight over the first head's stores and the wait below
      if (nh > 1) {
        if (full)
          load_rows<true>(xv + (size_t)(hq * rep + vbase + grp + 1) * kD + c0, v_stride, t0, s0, Lc, r0, nullptr, xr);
        else
          load_rows<false>(xv + (size_t)(hq * rep + vbase + grp + 1) * kD + c0, v_stride, t0, s0, Lc, r0,
                           hist(vch0 + kD), xr);
      }
      if (grp + 2 < nrep) {
        prefetch_v(grp + 2);
        if (grp + 3 < nrep) prefetch_v(grp + 3);
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // first head: its tile is not under the K K^T / Q K^T operands
        float col[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) col[r] = y[r][c];
        tc::st_chunk_f16(sm + P_VT0 + tc::sw128_chunk(128, c0 + c, warp), col);
      }
      if (grp == 0 && tid == 0 && compact && qk_images) tc::bulk_wait_read();  // before the tiles are reused
      if (grp == 0 && wait_all(bar, phase)) { failed = true; break; }  // K K^T and Q K^T are done
      if (nh > 1) {
        if (full) conv_silu<true>(xr, p.conv_w, vch0 + kD, Lc, r0, y);
        else conv_silu<false>(xr, p.conv_w, vch0 + kD, Lc, r0, y);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float col[8];
#pragma unroll
          for (int r = 0; r < 8; ++r) col[r] = y[r][c];
          tc::st_chunk_f16(sm + P_VT1 + tc::sw128_chunk(128, c0 + c, warp), col);
        }
      }
    }

    // A (fp32, strictly lower, zero elsewhere) and -A_Q (image) of both heads
#pragma unroll 1
    for (int hh = 0; hh < nh; ++hh) {
      const float *sGh = sGall + (grp + hh) * 256;
      float v[32];
      tc::tmem_ld32(tmem + lane_off + COL_P1 + 32 * gh, v);
      float2 Gs[16];  // shared-memory reads before the stores below
#pragma unroll
      for (int q = 0; q < 16; ++q) Gs[q] = *reinterpret_cast<const float2 *>(sGh + 32 * gh + 2 * q);
      const int r = lr & 63;
      const float2 Gr = tc::splat2(sGh[r]);
      if (lr < 64) {
        const float2 br = tc::splat2(sGh[128 + r]);
#pragma unroll
        for (int q = 0; q < 16; ++q) {  // beta_r e^(G_r - G_s) (K K^T)_rs for s < r
          const float2 d = tc::mul2(tc::sub2(Gr, Gs[q]), tc::splat2(kLog2e));
          const float2 e = tc::mul2(tc::mul2(br, make_float2(tc::ex2_approx(d.x), tc::ex2_approx(d.y))),
                                    make_float2(v[2 * q], v[2 * q + 1]));
          const int s = 32 * gh + 2 * q;
          v[2 * q] = (s < r) ? e.x : 0.0f;
          v[2 * q + 1] = (s + 1 < r) ? e.y : 0.0f;
        }
        float *row = AT(hh) + r * kPad + 32 * gh;
#pragma unroll
        for (int q = 0; q < 32; q += 2) *reinterpret_cast<float2 *>(row + q) = make_float2(v[q], v[q + 1]);
      } else {
#pragma unroll
        for (int q = 0; q < 16; ++q) {  // -A_Q = -e^(G_r - G_s) (Q K^T)_rs for s <= r
          const float2 d = tc::mul2(tc::sub2(Gr, Gs[q]), tc::splat2(kLog2e));
          const float2 e = tc::mul2(make_float2(-tc::ex2_approx(d.x), -tc::ex2_approx(d.y)),
                                    make_float2(v[2 * q], v[2 * q + 1]));
          const int s = 32 * gh + 2 * q;
          v[2 * q] = (s <= r) ? e.x : 0.0f;
          v[2 * q + 1] = (s + 1 <= r) ? e.y : 0.0f;
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)  // staged in the image's layout (the inverse's scratch is free)
          tc::st_chunk_f16(sm + P_XF + tc::sw128_chunk(64, r, 4 * gh + cc), v + 8 * cc);
        // warps 2 and 6 hold rows 0-31 of -A_Q, warps 3 and 7 rows 32-63: each pair's 4 KB of the image,
        // contiguous, goes by one bulk copy once the pair (synchronised among its own 64 threads) has staged it
        tc::fence_async_smem();
        const int pr = warp & 1, t = 32 * (warp >> 2) + lane;
        tc::named_barrier(1 + pr, 64);
        if (t == 0) {
          tc::bulk_s2g(v_slot_of(grp + hh) + (compact ? kCAq : kVAq) + 4096 * pr, sm + P_XF + 4096 * pr, 4096);
          tc::bulk_commit();
        }
        if (hh + 1 < nh) {  // read before the next head's staging
          if (t == 0) tc::bulk_wait_read();
          tc::named_barrier(1 + pr, 64);
        }
      }
    }
    if (lr >= 64 && 32 * (warp >> 2) + lane == 0) tc::bulk_wait_read();  // before the inverse's scratch goes there
    tc::fence_before_sync();
    __syncthreads();

    // T = (I + A)^-1 of both heads, in place, by recursive doubling on the unit lower-triangular I + A.
    // (a) the four diagonal 16 x 16 blocks by forward substitution, one column per thread
    {
      float x[16];
      const int hh = tid >> 6, bb = (tid >> 4) & 3, s = tid & 15;
      const bool act = hh < nh;
      if (tid >= 128 && !compact) {  // meanwhile: the K~^T = (diag(e^(G_C - G)) K)^T images of the pair, from the
                                // K^T tile (the image has its SW128 layout), 16-byte chunks in order
        for (int h2 = 0; h2 < nh; ++h2) {
          const float *dec = sGall + (grp + h2) * 256 + 192;
          uint8_t *dst = v_slot_of(grp + h2) + kVKt;
#pragma unroll 4
          for (int k = 0; k < 8; ++k) {
            const int q = tid - 128 + 128 * k;              // chunk q: row i = q / 8, physical position q % 8
            const int mc = (q & 7) ^ ((q >> 3) & 7);        // its columns m = 8 mc .. 8 mc + 7
            const uint4 raw = *reinterpret_cast<const uint4 *>(sm + P_KT + 16 * q);
            const float4 d0 = *reinterpret_cast<const float4 *>(dec + 8 * mc);
            const float4 d1 = *reinterpret_cast<const float4 *>(dec + 8 * mc + 4);
            const float2 k0 = tc::mul2(__half22float2(*reinterpret_cast<const __half2 *>(&raw.x)), make_float2(d0.x, d0.y));
            const float2 k1 = tc::mul2(__half22float2(*reinterpret_cast<const __half2 *>(&raw.y)), make_float2(d0.z, d0.w));
            const float2 k2 = tc::mul2(__half22float2(*reinterpret_cast<const __half2 *>(&raw.z)), make_float2(d1.x, d1.y));
            const float2 k3 = tc::mul2(__half22float2(*reinterpret_cast<const __half2 *>(&raw.w)), make_float2(d1.z, d1.w));
            *reinterpret_cast<uint4 *>(dst + 16 * q) = make_uint4(tc::pack_f16x2(k0.x, k0.y), tc::pack_f16x2(k1.x, k1.y),
                                                                tc::pack_f16x2(k2.x, k2.y), tc::pack_f16x2(k3.x, k3.y));
          }
        }
      }
      if (act) {
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          const float *arow = AT(hh) + (16 * bb + r) * kPad + 16 * bb;
          float acc0 = (r == s) ? 1.0f : 0.0f, acc1 = 0.0f;
#pragma unroll
          for (int m = 0; m + 1 < r; m += 2) {
            acc0 = fmaf(-arow[m], x[m], acc0);
            acc1 = fmaf(-arow[m + 1], x[m + 1], acc1);
          }
          if (r & 1) acc0 = fmaf(-arow[r - 1], x[r - 1], acc0);
          x[r] = acc0 + acc1;
        }
      }
      __syncthreads();  // every column is solved before the blocks are overwritten
      if (act) {
#pragma unroll
        for (int r = 0; r < 16; ++r) AT(hh)[(16 * bb + r) * kPad + 16 * bb + s] = x[r];
      }
    }
    __syncthreads();
    // (b) T_10 = -T_11 (A_10 T_00) and T_32 = -T_33 (A_32 T_22): two elements per thread and head
    //     (the diagonal blocks of T hold zeros above their diagonal)
#pragma unroll 1
    for (int hh = 0; hh < nh; ++hh) {
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int e = tid + kPrepThreads * it;
        const int blk = e >> 8, r = (e >> 4) & 15, s = e & 15, o = 32 * blk;
        const float *arow = AT(hh) + (o + 16 + r) * kPad + o;
        const float *tcol = AT(hh) + o * kPad + o + s;
        float2 acc = make_float2(0.0f, 0.0f);  // even and odd k
#pragma unroll
        for (int k = 0; k < 16; k += 2)
          acc = tc::fma2(*reinterpret_cast<const float2 *>(arow + k), make_float2(tcol[k * kPad], tcol[(k + 1) * kPad]),
                         acc);
        XF(hh)[e] = acc.x + acc.y;
      }
    }
    __syncthreads();
#pragma unroll 1
    for (int hh = 0; hh < nh; ++hh) {
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int e = tid + kPrepThreads * it;
        const int blk = e >> 8, r = (e >> 4) & 15, s = e & 15, o = 32 * blk;
        const float *trow = AT(hh) + (o + 16 + r) * kPad + o + 16;
        const float *xf = XF(hh) + blk * 256 + s;
        float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < 16; k += 2)
          acc = tc::fma2(*reinterpret_cast<const float2 *>(trow + k), make_float2(xf[k * 16], xf[(k + 1) * 16]), acc);
        AT(hh)[(o + 16 + r) * kPad + o + s] = -(acc.x + acc.y);  // over A_10 / A_32, read above
      }
    }
    __syncthreads();
    // (c) the lower-left 32 x 32 block T_21 = -T_2 (A_21 T_1); threads 128 hh .. 128 hh + 127 take
    //     head hh, a 2 x 4 tile each.  T_1 and T_2 are lower triangular: (A_21 T_1)[., c] sums over
    //     k >= c and (T_2 Y)[r, .] over k <= r, so each warp's loop starts (first product: its columns
    //     share a lower bound) or stops (second: its rows share an upper bound) where its tile allows
    {
      const int hh = tid >> 7, t = tid & 127;
      const bool act = hh < nh;
      if (act) {
        const int rr = 2 * (t & 15), cc = 4 * (t >> 4), k0 = 8 * ((t >> 5) & 3);  // k0: the warp's first column
        const float *At = AT(hh);
        const float *a0 = At + (32 + rr) * kPad, *a1 = a0 + kPad;
        float2 y0a = make_float2(0.0f, 0.0f), y0b = y0a, y1a = y0a, y1b = y0a;  // rows rr, rr + 1
#pragma unroll 4
        for (int k = k0; k < 32; k += 2) {
          const float2 av = *reinterpret_cast<const float2 *>(a0 + k), bv = *reinterpret_cast<const float2 *>(a1 + k);
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const float *trow = At + (k + kk) * kPad + cc;
            const float2 t01 = *reinterpret_cast<const float2 *>(trow), t23 = *reinterpret_cast<const float2 *>(trow + 2);
            const float2 x = tc::splat2(kk ? av.y : av.x), z = tc::splat2(kk ? bv.y : bv.x);
            y0a = tc::fma2(x, t01, y0a);
            y0b = tc::fma2(x, t23, y0b);
            y1a = tc::fma2(z, t01, y1a);
            y1b = tc::fma2(z, t23, y1b);
          }
        }
        *reinterpret_cast<float4 *>(XF(hh) + rr * 32 + cc) = make_float4(y0a.x, y0a.y, y0b.x, y0b.y);
        *reinterpret_cast<float4 *>(XF(hh) + (rr + 1) * 32 + cc) = make_float4(y1a.x, y1a.y, y1b.x, y1b.y);
      }
      __syncthreads();
      if (act) {
        const int rr = 2 * (t >> 3), cc = 4 * (t & 7), k1 = 8 * ((t >> 5) & 3) + 8;  // k1: past the warp's last row
        float *At = AT(hh);
        const float *t0r = At + (32 + rr) * kPad + 32, *t1r = t0r + kPad;
        float2 z0a = make_float2(0.0f, 0.0f), z0b = z0a, z1a = z0a, z1b = z0a;
#pragma unroll 4
        for (int k = 0; k < k1; k += 2) {
          const float2 pv = *reinterpret_cast<const float2 *>(t0r + k), qv = *reinterpret_cast<const float2 *>(t1r + k);
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const float4 yk = *reinterpret_cast<const float4 *>(XF(hh) + (k + kk) * 32 + cc);
            const float2 x = tc::splat2(kk ? pv.y : pv.x), z = tc::splat2(kk ? qv.y : qv.x);
            z0a = tc::fma2(x, make_float2(yk.x, yk.y), z0a);
            z0b = tc::fma2(x, make_float2(yk.z, yk.w), z0b);
            z1a = tc::fma2(z, make_float2(yk.x, yk.y), z1a);
            z1b = tc::fma2(z, make_float2(yk.z, yk.w), z1b);
          }
        }
        float *o0 = At + (32 + rr) * kPad + cc, *o1 = o0 + kPad;
        *reinterpret_cast<float2 *>(o0) = make_float2(-z0a.x, -z0a.y);
        *reinterpret_cast<float2 *>(o0 + 2) = make_float2(-z0b.x, -z0b.y);
        *reinterpret_cast<float2 *>(o1) = make_float2(-z1a.x, -z1a.y);
        *reinterpret_cast<float2 *>(o1 + 2) = make_float2(-z1b.x, -z1b.y);
      }
    }
    // [T diag(beta gamma); T diag(beta)] of each head over its own T (read first)
#pragma unroll 1
    for (int hh = 0; hh < nh; ++hh) {
      const int r = tid & 63, oq = tid >> 6;  // columns [16 oq, 16 oq + 16)
      const float *sGh = sGall + (grp + hh) * 256;
      uint32_t pa[8], pb[8];  // fp16 pairs
      __syncthreads();  // T complete (first head) / the previous head's stores done
#pragma unroll
      for (int e = 0; e < 16; e += 2) {
        float b2[2], a2[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int m = 16 * oq + e + i;
          const float t = (m <= r) ? AT(hh)[r * kPad + m] : 0.0f;
          b2[i] = t * sGh[128 + m];
          a2[i] = b2[i] * sGh[64 + m];
        }
        pa[e >> 1] = tc::pack_f16x2(a2[0], a2[1]);
        pb[e >> 1] = tc::pack_f16x2(b2[0], b2[1]);
      }
      __syncthreads();
      uint8_t *tbs = reinterpret_cast<uint8_t *>(AT(hh));
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int q = 4 * half;
        *reinterpret_cast<uint4 *>(tbs + tc::sw128_chunk(128, r, 2 * oq + half)) =
            make_uint4(pa[q], pa[q + 1], pa[q + 2], pa[q + 3]);
        *reinterpret_cast<uint4 *>(tbs + tc::sw128_chunk(128, 64 + r, 2 * oq + half)) =
            make_uint4(pb[q], pb[q + 1], pb[q + 2], pb[q + 3]);
      }
    }
    publish_operands();

    // ---------------- per head: [T diag(beta gamma); T diag(beta)] times the 256-row B operand
    //   first head:  B = [K^T; V^T]: W = T diag(beta gamma) K in rows 0-63, columns 0-127,
    //                U' = T diag(beta) V in rows 64-127, columns 128-255
    //   second head: B = [V^T; K^T]: the same with the column halves swapped
    // Each head's W and U' are staged in shared memory (over its own operands, which the product has
    // read) and stored to their images in order, while the next head's product runs.
    auto issue_wu = [&](int hh) {
      if (tid == 0) {
        mma_chain(tmem, sbase + (hh ? P_AT1 : P_AT0), 128, 0, sbase + (hh ? P_VT1 : P_KT), 256, 0, 4, kIdN256,
                  false);
        tc::mma_commit(bar);
      }
    };
    issue_wu(0);
#pragma unroll 1
    for (int hh = 0; hh < nh; ++hh) {
      if (wait_all(bar, phase)) { failed = true; break; }
      uint8_t *stw = sm + (hh ? P_AT1 : P_AT0);  // W staging: the image's two 8 KB slab halves (rows 64-127)
      uint8_t *stu = sm + (hh ? P_VT1 : P_VT0);  // U' staging: [4 slices][64 m][32 j], chunks permuted per row
      const int wcol = hh ? 128 : 0, half = warp >> 2;  // this warp's 64 columns of W or U'
      if ((warp & 3) < 2) {  // TMEM lanes 0-63: W
        const int r = 32 * (warp & 3) + lane;
#pragma unroll
        for (int c32 = 0; c32 < 2; ++c32) {
          float w[32];
          tc::tmem_ld32(tmem + lane_off + wcol + 64 * half + 32 * c32, w);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)
            tc::st_chunk_f16(stw + half * 8192 + tc::sw128_chunk(64, r, 4 * c32 + cc), w + 8 * cc);
        }
      } else {  // TMEM lanes 64-127: U'
        const int m = 32 * (warp & 3) - 64 + lane;
#pragma unroll
        for (int c32 = 0; c32 < 2; ++c32) {
          float u[32];
          tc::tmem_ld32(tmem + lane_off + (128 - wcol) + 64 * half + 32 * c32, u);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)  // state columns 64 half + 32 c32 + 8 cc .. + 7: slice 2 half + c32
            tc::st_chunk_f16(stu + (2 * half + c32) * 4096 + m * 64 + ((cc ^ ((m >> 1) & 3)) << 4), u + 8 * cc);
        }
      }
      tc::fence_async_smem();  // the stagings are read by the tensor memory accelerator
      tc::fence_before_sync();
      __syncthreads();  // staged, and the accumulator is read: the next product may overwrite it
      tc::fence_after_sync();
      if (hh + 1 < nh) issue_wu(hh + 1);
      if (tid == 0) {  // W: the staged bytes are the image's, in order; U': one swizzled 3-D store
        uint8_t *v_slot = v_slot_of(grp + hh);
        if (compact) {
          tc::bulk_s2g(v_slot + kCW, stw, 16384);
        } else {  // the W rows 64-127 of the two slabs of [Q^; W]
          tc::bulk_s2g(v_slot + kVWQ + 8192, stw, 8192);
          tc::bulk_s2g(v_slot + kVWQ + 24576, stw + 8192, 8192);
        }
        tc::tma_store_3d(&upmap, 0, 0, g * h_v + hq * rep + vbase + grp + hh, stu);
        tc::bulk_commit();
      }
    }
    if (grp + 2 < nrep) {  // the stagings are read before the next pair's tiles go there
      if (tid == 0) tc::bulk_wait_read();
      __syncthreads();
    }
  }
  if (failed && tid == 0) set_status(p.status, kDevTimeout);
  tc::bulk_wait_all();  // this thread's image stores are done before the CTA's shared memory goes
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, tmem_cols);
}

// ================================================================ state pass
// The columns j of H = S^T (d_v) evolve independently, so each (sequence,
// value head) chain is split over a cluster of kSlices CTAs, CTA `sv` owning
// columns [kBV sv, kBV sv + kBV).  Per chunk, with H the slice entering it:
//   MMA 1:  D_U  = [Q^; W] (-H)            rows 0-63: -Q^ H,  rows 64-127: -W H
//           U    = U' + D_U[64:128]         (fp32, then the fp16 operand U^T)
//   MMA 2:  D_H += K~^T U                   (D_H scaled by gamma_C before)
//           D_U += [-A_Q; *] U              (rows 0-63 become -O; rows 64-127 unused)
// Every product has M = 128 rows and N = kBV columns.  tcgen05.mma issues at
// a fixed cost per instruction, so the critical path per chunk is kept to
// MMA 1 (8 instructions) and the K~^T U half of MMA 2 (4); the A_Q U half is
// issued by a second thread (ST >= 2: the copy warp, once the K~^T U half is
// in, so that half runs first on the tensor core).  Warps 0-7 run the chain
// (each TMEM lane by two warps, one per half of the columns), warps 8-9 the
// epilogue one chunk behind (exchanging per-token partial sums of o^2 with the
// other CTAs of the cluster through st.async into their shared memory), warp
// 10 issues the operand copies.
// ST = 0: one buffer per operand set, refilled as soon as each set is consumed
// (two CTAs per SM).  ST >= 2: a ring of ST whole per-chunk operand sets
// ([Q^; W], K~^T, -A_Q, U' slice, gamma), so the copies of the next chunks
// stream in while one is computed (one CTA per SM).
template <int NS, int ST>
struct StateCfg {
  static constexpr int kSlices = NS;                    // CTAs per chain
  static constexpr int kBV = kD / NS;                   // state columns per CTA
  static constexpr int kCG = 2;                         // column groups of the chain warps
  static constexpr int kCols = kBV / kCG;               // columns per chain thread
  static constexpr int kMainWarps = 4 * kCG;            // TMEM lane quarters x column groups
  static constexpr int kMainThreads = 32 * kMainWarps, kEpiThreads = 64;
  static constexpr int kEpiWarp = kMainWarps, kProdWarp = kMainWarps + 2;
  static constexpr int kThreads = 32 * (kMainWarps + 3);
  static constexpr int kMinBlocks = ST == 0 ? 2 : 1;
  // one operand set: [Q^; W] (32 KB), K~^T (16 KB), -A_Q (8 KB; rows 64-127 of its
  // 128-row operand read the next 8 KB, unused), U' [64 m][kBV] fp16, gamma [64]
  static constexpr uint32_t R_WQ = 0, R_KT = 32768, R_AQ = 49152, R_UP = 57344;
  static constexpr uint32_t R_GAM = R_UP + kBV * 128;
  static constexpr uint32_t kStage = (R_GAM + 256 + 1023) / 1024 * 1024;
  static constexpr uint32_t kSets = ST == 0 ? 1 : ST;
  static constexpr uint32_t S_NH = kSets * kStage;      // -H^T fp16 [kBV j][128 i]
  static constexpr uint32_t S_NU = S_NH + kBV * 256;    // U^T fp16 [kBV j][64 m]
  static constexpr uint32_t S_Z = S_NU + kBV * 128;     // z [2][64 t][kBV] bf16 (TMA), two chunks ahead
  static constexpr uint32_t S_Y = S_Z + 2 * kBV * 128;  // y [64 t][kBV] bf16 (TMA store)
  static constexpr uint32_t S_WN = S_Y + kBV * 128;     // norm_w of this slice [kBV]
  static constexpr uint32_t S_PART = S_WN + kBV * 4;    // partial sums of o^2 [2][kSlices][64]
  static constexpr uint32_t S_MISC = S_PART + 2 * kSlices * 64 * 4;
  static constexpr size_t kSmem = S_MISC + 256 + 1024;
  // barriers: chain, epilogue, then the operand-set ones of the buffering scheme
  static constexpr int B_M1 = 0, B_M2 = 1, B_Z = 2 /* [2] */, B_ORDY = 4, B_ODONE = 6, B_PART = 8, B_SETS = 10;
  // ST >= 2: after full[ST] and empty[ST], "U published" (chain -> copy warp) and "-A_Q U done"
  static constexpr int B_UPUB = B_SETS + 2 * ST, B_AQ = B_UPUB + 1;
  static constexpr int kBars = B_SETS + (ST == 0 ? 4 : 2 * ST + 2);
  // tensor memory: H slice (fp32, lanes i), D_U in two buffers (chunk c's
  // epilogue reads one while chunk c+1's first product writes the other)
  static constexpr int COL_H = 0, COL_U = kBV;
  static constexpr uint32_t kTmemCols = 3 * kBV <= 128 ? 128 : 3 * kBV <= 256 ? 256 : 512;
  static constexpr uint32_t kIdN = tc::idesc_f16(128, kBV);
  static_assert(S_NH % 1024 == 0 && S_NU % 1024 == 0 && kStage % 1024 == 0, "SW128 tiles");
  static_assert(kSets * kStage - kStage + R_AQ + 16384 <= S_MISC, "rows 64-127 of the -A_Q operand stay inside");
  static_assert(S_Z % 128 == 0 && S_Y % 128 == 0, "TMA boxes 128-byte aligned");
  static_assert(kMinBlocks * (kSmem + 1024) <= 233472 && kSmem <= 232448, "shared memory budget");
  static_assert(kBars * 8 + 4 <= 256, "barrier block");
  static_assert(kCols == 8 || kCols == 16 || kCols == 32, "TMEM access widths");
};
constexpr int kBarMain = 1, kBarEpi = 2;

// tcgen05.ld / st of NC consecutive columns (32 lanes x 32 bit), NC = 8, 16 or 32
[[maybe_unused]] __device__ __forceinline__ void tmem_ld_cols(uint32_t a, float (&v)[8]) { tc::tmem_ld8(a, v); }
[[maybe_unused]] __device__ __forceinline__ void tmem_st_cols(uint32_t a, const float (&v)[8]) {
  tc::tmem_st8_nowait(a, v);
  tc::tmem_st_wait();
}
[[maybe_unused]] __device__ __forceinline__ void tmem_st_cols_nowait(uint32_t a, const float (&v)[8]) {
  tc::tmem_st8_nowait(a, v);
}
[[maybe_unused]] __device__ __forceinline__ void tmem_ld_cols(uint32_t a, float (&v)[32]) { tc::tmem_ld32(a, v); }
[[maybe_unused]] __device__ __forceinline__ void tmem_ld_cols(uint32_t a, float (&v)[16]) { tc::tmem_ld16(a, v); }
[[maybe_unused]] __device__ __forceinline__ void tmem_st_cols(uint32_t a, const float (&v)[32]) { tc::tmem_st32(a, v); }
[[maybe_unused]] __device__ __forceinline__ void tmem_st_cols(uint32_t a, const float (&v)[16]) { tc::tmem_st16(a, v); }
[[maybe_unused]] __device__ __forceinline__ void tmem_st_cols_nowait(uint32_t a, const float (&v)[32]) {
  tc::tmem_st32_nowait(a, v);
}
[[maybe_unused]] __device__ __forceinline__ void tmem_st_cols_nowait(uint32_t a, const float (&v)[16]) {
  tc::tmem_st16_nowait(a, v);
}

template <int NS, int ST>
__global__ void __launch_bounds__(StateCfg<NS, ST>::kThreads, StateCfg<NS, ST>::kMinBlocks)
    state_kernel(const PrefillParams p, const Ws ws, const __grid_constant__ CUtensorMap zmap,
                 const __grid_constant__ CUtensorMap omap) {
  using C = StateCfg<NS, ST>;
  constexpr int kSlices = C::kSlices, kBV = C::kBV, kCols = C::kCols;
  constexpr int kMainThreads = C::kMainThreads, kEpiThreads = C::kEpiThreads, kStateThreads = C::kThreads;
  constexpr uint32_t S_NH = C::S_NH, S_NU = C::S_NU, S_Z = C::S_Z, S_Y = C::S_Y, S_WN = C::S_WN,
                     S_PART = C::S_PART, S_MISC = C::S_MISC;
  // operand set of the chain's chunk c (a ring slot when ST >= 2)
  auto set_of = [](int c) -> uint32_t { return ST == 0 ? 0u : C::kStage * (uint32_t)(c % (ST == 0 ? 1 : ST)); };
  constexpr int COL_H = C::COL_H, COL_U = C::COL_U;
  constexpr uint32_t kStateTmemCols = C::kTmemCols, kIdNBV = C::kIdN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sbase = tc::smem_u32(sm);
  const int h_v = p.h_v;
  const int chain = blockIdx.x / kSlices;  // chains go sequence by sequence, longest sequences first
  const int sv = (int)tc::cluster_ctarank();
  const int h = chain % h_v;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
  const int j0 = kBV * sv;  // first state column of this CTA
  int s0 = p.cu_seqlens[chain / h_v], s1 = p.cu_seqlens[chain / h_v + 1];  // one sequence: it is n = 0

  uint64_t *bar = reinterpret_cast<uint64_t *>(sm + S_MISC);
  uint64_t *bar_m1 = bar + C::B_M1, *bar_m2 = bar + C::B_M2, *bar_z = bar + C::B_Z;
  uint64_t *bar_oready = bar + C::B_ORDY, *bar_odone = bar + C::B_ODONE, *bar_part = bar + C::B_PART;  // [2] each
  // ST = 0: set 1 ([Q^; W], U', gamma) and set 2 (K~^T, -A_Q) full, MMA 2's second half done, U step done;
  // ST >= 2: full[ST], empty[ST] (empty completes when both halves of MMA 2 have read the set)
  uint64_t *bar_s1 = bar + C::B_SETS, *bar_s2 = bar + C::B_SETS + 1, *bar_m2b = bar + C::B_SETS + 2;
  uint64_t *bar_udone = bar + C::B_SETS + 3;
  uint64_t *bar_full = bar + C::B_SETS, *bar_empty = bar + C::B_SETS + (ST == 0 ? 0 : ST);
  uint64_t *bar_upub = bar + (ST == 0 ? 0 : C::B_UPUB), *bar_aq = bar + (ST == 0 ? 0 : C::B_AQ);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + S_MISC + 8 * C::kBars);
  float *sWn = reinterpret_cast<float *>(sm + S_WN);
  __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out);

  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, kStateTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < C::kBars; ++i)
      tc::mbar_init(bar + i, (ST != 0 && i >= C::B_SETS + ST && i < C::B_SETS + 2 * ST) ? 2 : 1);
    tc::fence_mbar_init();
    tc::prefetch_tmap(&zmap);
    tc::prefetch_tmap(&omap);
  }
  for (int j = tid; j < kBV; j += kStateThreads) sWn[j] = p.norm_w[j0 + j];
  tc::fence_before_sync();
  tc::cluster_sync();  // every CTA's barriers are initialised before any peer signals them
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  bool failed = false;

  tc::grid_dependency_wait();  // the chunk table and the operand images
  const int n = p.N > 1 ? ws.seq_order[chain / h_v] : chain / h_v;
  if (n != chain / h_v) {
    s0 = p.cu_seqlens[n];
    s1 = p.cu_seqlens[n + 1];
  }
  bool valid = s0 >= 0 && s1 >= s0 && s1 <= p.T;  // else reported by the chunk table
  const int g0 = valid ? ws.chunk_base[n] : 0, g1 = valid ? ws.chunk_base[n + 1] : 0;
  if (valid && g1 - g0 != (s1 - s0 + kC - 1) / kC) valid = false;  // table overflow, reported
  const int nch = valid ? g1 - g0 : 0;
  auto slot = [&](int gg) { return ws.vs + ((size_t)gg * h_v + h) * kVSlot; };

  if (warp < C::kMainWarps) {
    // ======================= state chain: TMEM lane i, columns [kCols gh, kCols gh + kCols)
    const int i = 32 * (warp & 3) + lane, gh = warp >> 2, jc = kCols * gh;
    uint32_t ph_s1 = 0, ph_s2 = 0, ph_m1 = 0, ph_m2 = 0;
    auto wait_main = [&](uint64_t *b, uint32_t &phase) {
      const bool ok = tc::mbar_wait(b, phase & 1);
      ++phase;
      tc::fence_after_sync();
      return tc::named_barrier_or(kBarMain, kMainThreads, !ok);
    };
    auto publish_main = [&]() {
      tc::fence_async_smem();
      tc::fence_before_sync();
      tc::named_barrier(kBarMain, kMainThreads);
      tc::fence_after_sync();
    };
    // H (fp32, TMEM) -> -H^T fp16 operand; then H <- gamma_C H for the coming update
    auto copy_and_scale = [&](float gC) {
      float v[kCols], w[kCols];
      tmem_ld_cols(tmem + lane_off + COL_H + jc, v);
#pragma unroll
      for (int j = 0; j < kCols; ++j) w[j] = v[j] * gC;
      tmem_st_cols_nowait(tmem + lane_off + COL_H + jc, w);  // completes while the copy is written
      __half *nh = reinterpret_cast<__half *>(sm + S_NH);
#pragma unroll
      for (int j = 0; j < kCols; ++j) nh[tc::sw128_offset(kBV, jc + j, i) >> 1] = __float2half_rn(-v[j]);
      tc::tmem_st_wait();
    };

    // ---------------- initial state slice -> TMEM H
    const size_t st_off = ((size_t)n * h_v + h) * kD * kD + (size_t)i * kD + j0 + jc;
    {
      float v[kCols];
#pragma unroll
      for (int q = 0; q < kCols; q += 4) {
        const float4 f = p.init_state ? *reinterpret_cast<const float4 *>(p.init_state + st_off + q)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
        v[q] = f.x; v[q + 1] = f.y; v[q + 2] = f.z; v[q + 3] = f.w;
      }
      tmem_st_cols(tmem + lane_off + COL_H + jc, v);
    }
    // gamma_C of the chain's chunk c, from its operand set
    auto gamma_c = [&](int c) { return reinterpret_cast<const float *>(sm + set_of(c) + C::R_GAM)[kC - 1]; };
    // wait for the operand set of chunk c (ST = 0: set 1 only; set 2 is waited before MMA 2)
    auto wait_set = [&](int c) {
      if constexpr (ST == 0) return wait_main(bar_s1, ph_s1);
      uint32_t par = (uint32_t)(c / (ST == 0 ? 1 : ST)) & 1;
      return wait_main(bar_full + c % (ST == 0 ? 1 : ST), par);
    };
    // the same wait, this thread only (the caller joins the chain's barrier)
    auto set_arrived = [&](int c) -> bool {
      if constexpr (ST == 0) {
        const bool ok = tc::mbar_wait(bar_s1, ph_s1 & 1);
        ++ph_s1;
        return ok;
      }
      return tc::mbar_wait(bar_full + c % (ST == 0 ? 1 : ST), (uint32_t)(c / (ST == 0 ? 1 : ST)) & 1);
    };
    if (nch > 0) {
      if (wait_set(0)) failed = true;
      else copy_and_scale(gamma_c(0));
    }
    publish_main();

    for (int c = 0; c < nch && !failed; ++c) {
      const int buf = c & 1;
      const uint32_t d_u = tmem + COL_U + kBV * buf;  // chunk c-2's -O read from it: waited below

      const uint32_t set = set_of(c);  // this chunk's operand set
      // ---------------- MMA 1: D_U = [Q^; W] (-H)
      if (tid == 0) {
        for (int k = 0; k < 8; ++k)
          tc::mma16(d_u, tc::sdesc_kstep(sbase + set + C::R_WQ, 128, 0, k), tc::sdesc_kstep(sbase + S_NH, kBV, 0, k),
                    kIdNBV, k > 0 ? 1u : 0u);
        tc::mma_commit(bar_m1);
      }
      {  // MMA 1 done; ring form: the previous chunk's -A_Q U (copy warp) has read U^T, rewritten below
        bool ok = tc::mbar_wait(bar_m1, ph_m1 & 1);
        ++ph_m1;
        if constexpr (ST != 0)
          if (c >= 1) ok = tc::mbar_wait(bar_aq, (uint32_t)(c - 1) & 1) && ok;
        tc::fence_after_sync();
        if (tc::named_barrier_or(kBarMain, kMainThreads, !ok)) { failed = true; break; }
      }
      if (warp & 2) {  // U = U' + D_U rows 64-127 -> U^T fp16 operand
        const int m = i - 64;
        float u[kCols];
        tmem_ld_cols(d_u + lane_off + jc, u);
        const uint4 *up = reinterpret_cast<const uint4 *>(sm + set + C::R_UP + m * kBV * 2 + jc * 2);
        __half *nu = reinterpret_cast<__half *>(sm + S_NU);
#pragma unroll
        for (int q = 0; q < kCols / 8; ++q) {
          const uint4 raw = up[q];
          const __half2 *hp = reinterpret_cast<const __half2 *>(&raw);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __half22float2(hp[e]);
            u[8 * q + 2 * e] += f.x;
            u[8 * q + 2 * e + 1] += f.y;
          }
        }
#pragma unroll
        for (int j = 0; j < kCols; ++j) nu[tc::sw128_offset(kBV, jc + j, m) >> 1] = __float2half_rn(u[j]);
      }
      publish_main();
      if constexpr (ST == 0) {
        if (tid == 0) tc::mbar_arrive(bar_udone);  // U' and [Q^; W] of this chunk are consumed
        if (wait_main(bar_s2, ph_s2)) { failed = true; break; }
      }

      // ---------------- MMA 2: D_H += K~^T U (critical);  D_U += [-A_Q; *] U (second issuer: with the
      //                  ring, the copy warp, once these four are in, so they run first on the tensor core)
      if (tid == 0) {
        for (int k = 0; k < 4; ++k)
          tc::mma16(tmem + COL_H, tc::sdesc_kstep(sbase + set + C::R_KT, 128, 0, k),
                    tc::sdesc_kstep(sbase + S_NU, kBV, 0, k), kIdNBV, 1u);
        tc::mma_commit(bar_m2);
        if constexpr (ST != 0) {
          tc::mma_commit(bar_empty + c % (ST == 0 ? 1 : ST));
          tc::mbar_arrive(bar_upub);
        }
      } else if (ST == 0 && tid == 32) {
        for (int k = 0; k < 4; ++k)
          tc::mma16(d_u, tc::sdesc_kstep(sbase + set + C::R_AQ, 128, 0, k), tc::sdesc_kstep(sbase + S_NU, kBV, 0, k),
                    kIdNBV, 1u);
        tc::mma_commit(bar_m2b);
        tc::mma_commit(bar_oready + buf);
      }
      {  // MMA 2 done and chunk c+1's operand set in: one barrier for both
        bool ok = tc::mbar_wait(bar_m2, ph_m2 & 1);
        ++ph_m2;
        if (c + 1 < nch) ok = set_arrived(c + 1) && ok;
        tc::fence_after_sync();
        if (tc::named_barrier_or(kBarMain, kMainThreads, !ok)) { failed = true; break; }
      }
      if (c + 1 < nch) copy_and_scale(gamma_c(c + 1));
      {  // publish chunk c+1's -H^T; the epilogue has read chunk c-1's -O (chunk c+1 reuses its buffer)
        bool ok = true;
        if (c >= 1 && c + 1 < nch) ok = tc::mbar_wait(bar_odone + ((c + 1) & 1), ((c - 1) >> 1) & 1);
        tc::fence_async_smem();
        tc::fence_before_sync();
        const bool bad = tc::named_barrier_or(kBarMain, kMainThreads, !ok);
        tc::fence_after_sync();
        if (bad) { failed = true; break; }
      }
    }

    if (failed) {
      if (tid == 0) set_status(p.status, kDevTimeout);
    } else if (valid && p.final_state) {
      float v[kCols];
      tmem_ld_cols(tmem + lane_off + COL_H + jc, v);
#pragma unroll
      for (int q = 0; q < kCols; q += 4)
        *reinterpret_cast<float4 *>(p.final_state + st_off + q) = make_float4(v[q], v[q + 1], v[q + 2], v[q + 3]);
    }
  } else if (warp < C::kEpiWarp + 2) {
    // ======================= RMSNormGated epilogue (two warps; thread m owns token row m of the chunk)
    // buffer c & 1 of each two-buffer barrier completes for chunk c in phase (c >> 1) & 1
    const int m = tid - kMainThreads;
    int z_issued = 0, z_done = 0;  // z loads issued / waited for (chunks [0, z_issued))
    const float scale = rsqrtf((float)kD);
    auto issue_z = [&](int cc) {  // z of chunk cc into buffer cc & 1
      if (m == 0) {
        tc::mbar_arrive_expect_tx(bar_z + (cc & 1), 64 * kBV * 2);
        tc::tma_load_2d(sm + S_Z + (cc & 1) * kBV * 128, &zmap, h * kD + j0, s0 + kC * cc, bar_z + (cc & 1));
      }
      z_issued = cc + 1;
    };
    auto wait_epi = [&](uint64_t *b, uint32_t parity, bool cluster) {
      const bool ok = cluster ? tc::mbar_wait_cluster(b, parity) : tc::mbar_wait(b, parity);
      tc::fence_after_sync();
      return tc::named_barrier_or(kBarEpi, kEpiThreads, !ok);
    };
    // this thread's partial sum goes to slot [buf][sv][m] of every CTA of the cluster
    const uint32_t part_local = tc::smem_u32(sm + S_PART) + 4u * (uint32_t)(sv * 64 + m);
    if (nch > 0) issue_z(0);
    if (nch > 1) issue_z(1);
    for (int c = 0; c < nch; ++c) {
      const int buf = c & 1;
      const uint32_t par = (c >> 1) & 1;
      const uint32_t d_u = tmem + lane_off + COL_U + kBV * buf;
      const int t0 = s0 + kC * c;
      const int Lc = min(kC, s1 - t0);
      if (wait_epi(bar_oready + buf, par, false)) { failed = true; break; }
      constexpr int kEw = kBV < 32 ? kBV : 32;  // TMEM columns per epilogue load
      float ss = 0.0f;
#pragma unroll
      for (int c32 = 0; c32 < kBV; c32 += kEw) {
        float o[kEw];
        tmem_ld_cols(d_u + c32, o);
#pragma unroll
        for (int j = 0; j < kEw; ++j) ss = fmaf(o[j], o[j], ss);
      }
      ss *= scale * scale;
      if (m == 0) tc::mbar_arrive_expect_tx(bar_part + buf, kSlices * 64 * 4);
      const uint32_t off = 4u * (uint32_t)(buf * kSlices * 64);
      for (int r = 0; r < kSlices; ++r)
        tc::st_async_f32(tc::mapa(part_local + off, r), ss, tc::mapa(tc::smem_u32(bar_part + buf), r));
      if (wait_epi(bar_part + buf, par, true)) { failed = true; break; }
      const float *part = reinterpret_cast<const float *>(sm + S_PART) + buf * kSlices * 64;
      float tot = 0.0f;
#pragma unroll
      for (int r = 0; r < kSlices; ++r) tot += part[r * 64 + m];
      const float inv = -scale * rsqrtf(tot * (1.0f / kD) + kEpsRms);  // o = -scale D_U
      if (wait_epi(bar_z + buf, par, false)) { failed = true; break; }
      z_done = c + 1;
      tc::bulk_wait_read();  // this thread's earlier y copies have left S_Y
      tc::named_barrier(kBarEpi, kEpiThreads);
#pragma unroll
      for (int c32 = 0; c32 < kBV; c32 += kEw) {
        float o[kEw];
        tmem_ld_cols(d_u + c32, o);
        const uint4 *zrow = reinterpret_cast<const uint4 *>(sm + S_Z + buf * kBV * 128 + m * kBV * 2 + c32 * 2);
#pragma unroll
        for (int q = 0; q < kEw / 8; ++q) {
          const uint4 zz = zrow[q];
          const uint32_t zw[4] = {zz.x, zz.y, zz.z, zz.w};
          float y8[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float za = __uint_as_float(zw[e] << 16), zb = __uint_as_float(zw[e] & 0xFFFF0000u);
            const int j = c32 + 8 * q + 2 * e;
            // silu(z) = z (1 + tanh(z / 2)) / 2 with the hardware tanh: its ~2^-11
            // error scales one output element, well inside the output rounding
            y8[2 * e] = o[8 * q + 2 * e] * inv * sWn[j] * (0.5f * za) * (1.0f + tc::tanh_approx(0.5f * za));
            y8[2 * e + 1] = o[8 * q + 2 * e + 1] * inv * sWn[j + 1] * (0.5f * zb) * (1.0f + tc::tanh_approx(0.5f * zb));
          }
          *reinterpret_cast<uint4 *>(sm + S_Y + m * kBV * 2 + (c32 + 8 * q) * 2) =
              make_uint4(tc::pack_bf16x2(y8[0], y8[1]), tc::pack_bf16x2(y8[2], y8[3]), tc::pack_bf16x2(y8[4], y8[5]),
                         tc::pack_bf16x2(y8[6], y8[7]));
        }
      }
      tc::fence_before_sync();
      tc::fence_async_smem();
      tc::named_barrier(kBarEpi, kEpiThreads);
      if (m == 0) tc::mbar_arrive(bar_odone + buf);  // -O of this buffer is read
      if (c + 2 < nch) issue_z(c + 2);                // into the z buffer just consumed
      if (Lc == kC) {
        if (m == 0) {
          tc::tma_store_2d(&omap, h * kD + j0, t0, sm + S_Y);
          tc::bulk_commit();
        }
      } else if (m < Lc) {  // a sequence's last, short chunk: only its own rows
        tc::bulk_s2g(out + ((size_t)(t0 + m) * h_v + h) * kD + j0, sm + S_Y + m * kBV * 2, kBV * 2);
        tc::bulk_commit();
      }
    }
    tc::bulk_wait_all();
    if (failed) {
      if (m == 0) set_status(p.status, kDevTimeout);
      for (int cc = z_done; cc < z_issued; ++cc) tc::mbar_wait(bar_z + (cc & 1), (cc >> 1) & 1);
    }
  } else if (warp == C::kProdWarp) {
    if constexpr (ST == 0) {
      // ======================= operand copies (one lane), each set as soon as its buffers are free
      uint32_t ph = 0;
      int n1 = 0, n2 = 0;  // sets issued
      auto issue_s1 = [&](int gg) {  // [Q^; W], U' slice, gamma
        tc::mbar_arrive_expect_tx(bar_s1, 32768 + 64 * kBV * 2 + 256);
        tc::bulk_g2s(sm + C::R_WQ, slot(gg) + kVWQ, 32768, bar_s1);
        tc::bulk_g2s(sm + C::R_UP, slot(gg) + kVUp + (size_t)sv * 64 * kBV * 2, 64 * kBV * 2, bar_s1);
        tc::bulk_g2s(sm + C::R_GAM, slot(gg) + kVGam, 256, bar_s1);
        ++n1;
      };
      auto issue_s2 = [&](int gg) {  // K~^T, -A_Q
        tc::mbar_arrive_expect_tx(bar_s2, 16384 + 8192);
        tc::bulk_g2s(sm + C::R_KT, slot(gg) + kVKt, 16384, bar_s2);
        tc::bulk_g2s(sm + C::R_AQ, slot(gg) + kVAq, 8192, bar_s2);
        ++n2;
      };
      if (lane == 0 && nch > 0) {
        issue_s1(g0);
        issue_s2(g0);
        if (nch > 1) {
          tc::prefetch_l2(slot(g0 + 1) + kVWQ, 32768 + 16384);
          tc::prefetch_l2(slot(g0 + 1) + kVUp + (size_t)sv * 64 * kBV * 2, 64 * kBV * 2);
          tc::prefetch_l2(slot(g0 + 1) + kVAq, 8192 + 256);
        }
        for (int c = 0; c + 1 < nch; ++c) {
          // chunk c's MMA 1 and U' are consumed (the chain signals after MMA 1 and the U step)
          if (!tc::mbar_wait(bar_udone, ph & 1)) { failed = true; break; }
          issue_s1(g0 + c + 1);
          if (c + 2 < nch) {  // the chunk after: into L2 now, so its copies later come from there
            tc::prefetch_l2(slot(g0 + c + 2) + kVWQ, 32768 + 16384);
            tc::prefetch_l2(slot(g0 + c + 2) + kVUp + (size_t)sv * 64 * kBV * 2, 64 * kBV * 2);
            tc::prefetch_l2(slot(g0 + c + 2) + kVAq, 8192 + 256);
          }
          // chunk c's MMA 2 (both halves) has read K~^T and -A_Q
          if (!tc::mbar_wait(bar_m2, ph & 1) || !tc::mbar_wait(bar_m2b, ph & 1)) { failed = true; break; }
          issue_s2(g0 + c + 1);
          ++ph;
        }
        if (failed) set_status(p.status, kDevTimeout);
        // copies in flight must land before the CTA's shared memory goes away
        // (the last set of each kind; set k completes phase k of its barrier)
        if (n1 > 0) tc::mbar_wait(bar_s1, (uint32_t)(n1 - 1) & 1);
        if (n2 > 0) tc::mbar_wait(bar_s2, (uint32_t)(n2 - 1) & 1);
      }
    } else if (lane == 0 && nch > 0) {
      // ======================= operand copies (one lane): the set of chunk c into ring slot c % ST as soon
      // as MMA 2 of chunk c - ST has read it; and MMA 2's -A_Q U of every chunk, issued once the chain's
      // K~^T U is in (a waiter here lags its signaller by at most one use: the chain waits for chunk c's
      // -A_Q U before it publishes chunk c + 1's U)
      constexpr int kST = ST == 0 ? 1 : ST;
      int issued = 0;
      auto issue_set = [&](int c) {
        const int r = c % kST;
        uint8_t *dst = sm + set_of(c);
        const uint8_t *src = slot(g0 + c);
        tc::mbar_arrive_expect_tx(bar_full + r, 32768 + 16384 + 8192 + 64 * kBV * 2 + 256);
        tc::bulk_g2s(dst + C::R_WQ, src + kVWQ, 32768 + 16384, bar_full + r);  // [Q^; W] and K~^T
        tc::bulk_g2s(dst + C::R_AQ, src + kVAq, 8192, bar_full + r);
        tc::bulk_g2s(dst + C::R_UP, src + kVUp + (size_t)sv * 64 * kBV * 2, 64 * kBV * 2, bar_full + r);
        tc::bulk_g2s(dst + C::R_GAM, src + kVGam, 256, bar_full + r);
        issued = c + 1;
      };
      for (int c = 0; c < kST && c < nch; ++c) issue_set(c);
      for (int c = 0; c < nch; ++c) {
        if (!tc::mbar_wait(bar_upub, (uint32_t)c & 1)) { failed = true; break; }
        tc::fence_after_sync();
        const uint32_t d_u = tmem + COL_U + kBV * (c & 1), set = set_of(c);
        for (int k = 0; k < 4; ++k)
          tc::mma16(d_u, tc::sdesc_kstep(sbase + set + C::R_AQ, 128, 0, k), tc::sdesc_kstep(sbase + S_NU, kBV, 0, k),
                    kIdNBV, 1u);
        tc::mma_commit(bar_empty + c % kST);
        tc::mma_commit(bar_oready + (c & 1));
        tc::mma_commit(bar_aq);
        if (c + kST < nch) {
          if (!tc::mbar_wait(bar_empty + c % kST, (uint32_t)(c / kST) & 1)) { failed = true; break; }
          issue_set(c + kST);
        }
      }
      if (failed) set_status(p.status, kDevTimeout);
      // copies in flight must land before the CTA's shared memory goes away
      for (int c = issued - kST < 0 ? 0 : issued - kST; c < issued; ++c)
        tc::mbar_wait(bar_full + c % kST, (uint32_t)(c / kST) & 1);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kStateTmemCols);
  tc::cluster_sync();  // no CTA leaves while a peer may still store into its shared memory
}

// ================================================================ state pass, transposed
// One CTA per (sequence, value head) chain, owning the whole state, on the
// compact images.  The state is kept transposed, S = H^T (lanes j over d_v,
// columns i over d_k, fp32 in tensor memory), so both products of a chunk
// take their A operand straight from tensor memory (fp16 copies written there
// by the chain warps) and run at N = 128:
//   MMA 1:  D1 = (-S) [Q; W]^T          columns 0-63: -(Q H)^T, 64-127: -(W H)^T
//           U^T = U'^T + D1[:, 64:128]   (fp32), then two fp16 copies in tensor
//           memory: U^T diag(d) (d_m = e^(G_C - G_m), the decay to the chunk's
//           end) and U^T itself
//   MMA 2:  S  += (U^T diag(d)) K        (S scaled by gamma_C before; K from the
//                                          unscaled K^T image: this is K~^T U)
//           O2  = U^T (-A_Q)^T           (-(A_Q U)^T)
//   y:      o_r = -scale (gamma_r D1[:, r] + O2[:, r]),  y = o / rms(o) w silu(z)
// 16 tcgen05.mma per chunk (8 + 4 + 4) against 64 when the columns of H are
// split over four CTAs, and no shared-memory round trip for the operands the
// chain computes.  Warps 0-7 run the chain (warp w: TMEM lanes 32 (w & 3), half
// w >> 2 of the columns), warps 8-15 the RMSNormGated epilogue one chunk behind
// (thread = state column j, warp half = 32 of the chunk's tokens; the
// per-token sums of o^2 reduced across lanes and warps).  The MMA-issuing
// thread also streams the operand sets in by TMA, a ring of two: set c + 2
// goes into the slot of chunk c right after MMA 1 of chunk c + 1 is issued
// (MMAs complete in issue order, so chunk c's products have then read it).
namespace ts {
constexpr int kChainWarps = 8, kEpiWarps = 8;
constexpr int kChainThreads = 32 * kChainWarps, kEpiThreads = 32 * kEpiWarps;
constexpr int kThreads = 32 * (kChainWarps + kEpiWarps);
constexpr int kSets = 2;
// one operand set: [Q; W] (two slabs of [64 Q rows; 64 W rows], 32 KB), K^T (16 KB), -A_Q (8 KB),
// U' of every column (16 KB), gamma and the decays to the chunk's end (256 B each)
constexpr uint32_t R_WQ = 0, R_KT = 32768, R_AQ = 49152, R_UP = 57344, R_GAM = 73728, R_DEC = 73984;
constexpr uint32_t kSetBytes = 32768 + 16384 + 8192 + 16384 + 512;
constexpr uint32_t kStage = 75776;                      // 74 KB, 1024-aligned
constexpr uint32_t S_Z = kSets * kStage;                // z [2][64 t][128] bf16 (TMA)
constexpr uint32_t S_Y = S_Z + 2 * 16384;               // y [64 t][128] bf16 (TMA store)
constexpr uint32_t S_WN = S_Y + 16384;                  // norm_w [128]
constexpr uint32_t S_PART = S_WN + 512;                 // sums of o^2 [4 lane quarters][64 tokens]
constexpr uint32_t S_INV = S_PART + 1024;               // 1 / rms per token [64]
constexpr uint32_t S_MISC = S_INV + 256;
constexpr size_t kSmem = S_MISC + 256 + 1024;
// barriers: full[2], empty[2], m1, m2, oready, odone, z[2]
constexpr int B_FULL = 0, B_EMPTY = 2, B_M1 = 4, B_M2 = 5, B_ORDY = 6, B_ODONE = 7, B_Z = 8, kBars = 10;
// tensor memory: S, D1, O2, the fp16 -S (64 columns), U^T diag(d) and U^T (32 columns each)
constexpr uint32_t COL_S = 0, COL_D = 128, COL_O2 = 256, COL_AS = 320, COL_AU = 384, COL_AU2 = 416;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kId128 = tc::idesc_f16(128, 128), kId64 = tc::idesc_f16(128, 64);
static_assert(R_DEC + 256 <= kStage && kStage % 1024 == 0 && R_WQ + kSetBytes == R_DEC + 256, "operand set");
static_assert(kSmem <= 232448, "shared memory budget (one CTA per SM)");
static_assert(kBars * 8 + 4 <= 256, "barrier block");
static_assert(COL_AU2 + 32 <= kTmemCols, "tensor memory");
constexpr int kBarChain = 3, kBarEpiTs = 4;
}  // namespace ts

__global__ void __launch_bounds__(ts::kThreads, 1)
    state_ts_kernel(const PrefillParams p, const Ws ws, const __grid_constant__ CUtensorMap zmap,
                    const __grid_constant__ CUtensorMap omap) {
  using namespace ts;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sbase = tc::smem_u32(sm);
  const int h_v = p.h_v, h_qk = p.h_qk, hq = (blockIdx.x % h_v) / (h_v / h_qk);
  const int chain = blockIdx.x, h = chain % h_v;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
  uint64_t *bar = reinterpret_cast<uint64_t *>(sm + S_MISC);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + S_MISC + 8 * kBars);
  float *sWn = reinterpret_cast<float *>(sm + S_WN);
  __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out);

  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < kBars; ++i) tc::mbar_init(bar + i, 1);
    tc::fence_mbar_init();
    tc::prefetch_tmap(&zmap);
    tc::prefetch_tmap(&omap);
  }
  for (int j = tid; j < kD; j += kThreads) sWn[j] = p.norm_w[j];
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  bool failed = false;

  tc::grid_dependency_wait();  // the chunk table and the operand images
  int n = 0, s0, s1, g0, nch, flags = kRunOut;
  bool valid;
  const float *init_base;  // this chain's state in and out: [d_k][d_v], or null
  float *final_base;
  if (ws.runs) {  // a chain of the segment-parallel prefill
    const SegRun run = ws.runs[chain / h_v];
    s0 = run.s0; s1 = run.s1; g0 = run.g0; flags = run.flags;
    valid = s1 >= s0;
    nch = valid ? (s1 - s0 + kC - 1) / kC : 0;
    init_base = run.init ? run.init + (size_t)h * kD * kD : nullptr;
    final_base = run.final ? run.final + (size_t)h * kD * kD : nullptr;
  } else {
    n = p.N > 1 ? ws.seq_order[chain / h_v] : chain / h_v;
    s0 = p.cu_seqlens[n];
    s1 = p.cu_seqlens[n + 1];
    valid = s0 >= 0 && s1 >= s0 && s1 <= p.T;  // else reported by the chunk table
    g0 = valid ? ws.chunk_base[n] : 0;
    const int g1 = valid ? ws.chunk_base[n + 1] : 0;
    if (valid && g1 - g0 != (s1 - s0 + kC - 1) / kC) valid = false;  // table overflow, reported
    nch = valid ? g1 - g0 : 0;
    init_base = p.init_state ? p.init_state + ((size_t)n * h_v + h) * kD * kD : nullptr;
    final_base = p.final_state ? p.final_state + ((size_t)n * h_v + h) * kD * kD : nullptr;
  }
  const bool transfer = (flags & kRunTransfer) != 0, with_out = (flags & kRunOut) != 0;
  auto vslot = [&](int gg) { return ws.vs + ((size_t)gg * h_v + h) * kCSlot; };
  auto qslot = [&](int gg) { return ws.qs + ((size_t)gg * h_qk + hq) * kQSlot; };
  auto set_at = [](int c) -> uint32_t { return kStage * (uint32_t)(c % kSets); };

  int issued = 0;  // operand sets issued (thread 0)
  auto issue_set = [&](int c) {
    uint8_t *dst = sm + set_at(c);
    const uint8_t *v = vslot(g0 + c), *q = qslot(g0 + c);
    uint64_t *full = bar + B_FULL + c % kSets;
    tc::mbar_arrive_expect_tx(full, kSetBytes);
    tc::bulk_g2s(dst + R_WQ, q + kQQ, 8192, full);                   // slab 0: Q rows 0-63
    tc::bulk_g2s(dst + R_WQ + 8192, v + kCW, 8192, full);            //         W rows 64-127
    tc::bulk_g2s(dst + R_WQ + 16384, q + kQQ + 8192, 8192, full);    // slab 1: Q
    tc::bulk_g2s(dst + R_WQ + 24576, v + kCW + 8192, 8192, full);    //         W
    tc::bulk_g2s(dst + R_KT, q + kQKt, 16384, full);
    tc::bulk_g2s(dst + R_AQ, v + kCAq, 8192, full);
    tc::bulk_g2s(dst + R_UP, v + kCUp, 16384, full);
    tc::bulk_g2s(dst + R_GAM, v + kCGam, 512, full);                  // gamma and the decays
    if (c + 1 < nch) {  // the set after: into L2 now
      tc::prefetch_l2(vslot(g0 + c + 1), kCSlot);
      tc::prefetch_l2(qslot(g0 + c + 1), kQSlot);
    }
    issued = c + 1;
  };
  if (tid == 0)
    for (int c = 0; c < kSets && c < nch; ++c) issue_set(c);

  if (warp < kChainWarps) {
    // ======================= the chain: lane j = 32 (warp & 3) + lane, columns half hf
    const int hf = warp >> 2, j = 32 * (warp & 3) + lane;
    const size_t st_base = j;  // element (i, j) of the chain's state at + i * kD
    // every chain thread waits on the mbarriers itself; a wait that runs out is
    // ORed into the next barrier the chain passes anyway (its publish)
    bool ok = true;
    auto publish_chain = [&]() {  // tensor-memory stores of every chain thread are done; true: a wait failed
      tc::tmem_st_wait();
      tc::fence_before_sync();
      const bool bad = tc::named_barrier_or(kBarChain, kChainThreads, !ok);
      tc::fence_after_sync();
      return bad;
    };
    // shared-memory descriptors of each ring slot's operands at K step 0; step k adds
    // (k >> 2) R 128 + (k & 3) 32 bytes, i.e. (k >> 2) R 8 + 2 (k & 3) in the 16-byte address field
    static_assert(kSets == 2, "two ring slots");
    const uint64_t desc_wq0 = tc::sdesc_sw128(sbase + R_WQ), desc_wq1 = tc::sdesc_sw128(sbase + kStage + R_WQ);
    const uint64_t desc_kt0 = tc::sdesc_sw128(sbase + R_KT), desc_kt1 = tc::sdesc_sw128(sbase + kStage + R_KT);
    {  // initial state slice: S[j][i] = H[i][j], columns [64 hf, 64 hf + 64)
      float v[32];
#pragma unroll 1
      for (int c32 = 0; c32 < 2; ++c32) {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int i = 64 * hf + 32 * c32 + e;
          v[e] = transfer ? (i == j ? 1.0f : 0.0f) : init_base ? init_base[st_base + (size_t)i * kD] : 0.0f;
        }
        tc::tmem_st32_nowait(tmem + lane_off + COL_S + 64 * hf + 32 * c32, v);
      }
    }
    if (publish_chain()) failed = true;
    for (int c = 0; c < nch && !failed; ++c) {
      const int rs = c % kSets;
      const uint32_t set = set_at(c);
      ok = tc::mbar_wait(bar + B_FULL + rs, (uint32_t)(c / kSets) & 1) && ok;
      // ---- S -> gamma_C S in place, and its fp16 negative as the A operand of MMA 1
      {
        const float gC = reinterpret_cast<const float *>(sm + set + R_GAM)[kC - 1];
        uint32_t r0[32], r1[32];  // both loads in flight before the wait
        tc::tmem_ld32_issue(tmem + lane_off + COL_S + 64 * hf, r0);
        tc::tmem_ld32_issue(tmem + lane_off + COL_S + 64 * hf + 32, r1);
        tc::tmem_ld_wait_regs(r0);
        tc::tmem_ld_wait_regs(r1);
        auto convert = [&](uint32_t (&r)[32], uint32_t col) {
          float pk[16], w[32];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = __uint_as_float(tc::pack_f16x2(-__uint_as_float(r[2 * e]), -__uint_as_float(r[2 * e + 1])));
          tc::tmem_st16_nowait(tmem + lane_off + COL_AS + col / 2, pk);
#pragma unroll
          for (int e = 0; e < 32; ++e) w[e] = __uint_as_float(r[e]) * gC;
          tc::tmem_st32_nowait(tmem + lane_off + COL_S + col, w);
        };
        convert(r0, 64 * hf);
        convert(r1, 64 * hf + 32);
      }
      if (publish_chain()) { failed = true; break; }
      // ---- MMA 1 (D1 and O2 of chunk c - 1 have been read by the epilogue)
      if (tid == 0) {
        bool ok0 = true;
        if (c >= 1) ok0 = tc::mbar_wait(bar + B_ODONE, (uint32_t)(c - 1) & 1);
        if (!ok0) set_status(p.status, kDevTimeout);
        tc::fence_after_sync();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          tc::mma16_ts(tmem + COL_D, tmem + COL_AS + 8 * k,
                       (rs ? desc_wq1 : desc_wq0) + (uint64_t)((k >> 2) * 128 * 8 + 2 * (k & 3)), kId128,
                       k > 0 ? 1u : 0u);
        tc::mma_commit(bar + B_M1);
        // the slot of chunk c - 1 is free once its products are done (before this MMA 1 completes): refill it
        if (c >= 1 && c + 1 < nch) {
          if (tc::mbar_wait(bar + B_EMPTY + (c - 1) % kSets, (uint32_t)((c - 1) / kSets) & 1))
            issue_set(c + 1);
          else
            set_status(p.status, kDevTimeout);
        }
      }
      // ---- U^T = U'^T + D1[:, 64:128] -> fp16 A operands; tokens [32 hf, 32 hf + 32).  U' (image: [4 slices
      //      of 32 columns][64 m][32] fp16, row-major) and the decays are read while MMA 1 runs
      {
        float u[32], upv[32], dm[32];
        const __half *up = reinterpret_cast<const __half *>(sm + set + R_UP + (j >> 5) * 4096) + (j & 31);
#pragma unroll
        for (int e = 0; e < 32; ++e) upv[e] = transfer ? 0.0f : __half2float(up[(32 * hf + e) * 32]);
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 d4 = *reinterpret_cast<const float4 *>(sm + set + R_DEC + 4 * (32 * hf + e));
          dm[e] = d4.x; dm[e + 1] = d4.y; dm[e + 2] = d4.z; dm[e + 3] = d4.w;
        }
        ok = tc::mbar_wait(bar + B_M1, (uint32_t)c & 1) && ok;
        tc::fence_after_sync();
        tc::tmem_ld32(tmem + lane_off + COL_D + 64 + 32 * hf, u);
        float pk[16], pd[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float u0 = u[2 * e] + upv[2 * e], u1 = u[2 * e + 1] + upv[2 * e + 1];
          pk[e] = __uint_as_float(tc::pack_f16x2(u0, u1));
          pd[e] = __uint_as_float(tc::pack_f16x2(u0 * dm[2 * e], u1 * dm[2 * e + 1]));
        }
        tc::tmem_st16_nowait(tmem + lane_off + COL_AU + 16 * hf, pd);
        tc::tmem_st16_nowait(tmem + lane_off + COL_AU2 + 16 * hf, pk);
      }
      if (publish_chain()) { failed = true; break; }
      // ---- MMA 2: S += (U^T diag(d)) K (the chain's next step waits for it), then O2 = U^T (-A_Q)^T
      //      (K^T and -A_Q are adjacent in the set: the -A_Q descriptor is the K^T one + 16 KB)
      if (tid == 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc::mma16_ts(tmem + COL_S, tmem + COL_AU + 8 * k, (rs ? desc_kt1 : desc_kt0) + (uint64_t)(2 * k), kId128, 1u);
        tc::mma_commit(bar + B_M2);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc::mma16_ts(tmem + COL_O2, tmem + COL_AU2 + 8 * k,
                       (rs ? desc_kt1 : desc_kt0) + (uint64_t)((R_AQ - R_KT) / 16 + 2 * k), kId64, k > 0 ? 1u : 0u);
        tc::mma_commit(bar + B_ORDY);
        tc::mma_commit(bar + B_EMPTY + rs);
      }
      ok = tc::mbar_wait(bar + B_M2, (uint32_t)c & 1) && ok;
      tc::fence_after_sync();
    }
    if (!ok) failed = true;
    if (failed) {
      if (tid == 0) set_status(p.status, kDevTimeout);
    } else if (valid && final_base) {
      float v[32];
#pragma unroll 1
      for (int c32 = 0; c32 < 2; ++c32) {
        tc::tmem_ld32(tmem + lane_off + COL_S + 64 * hf + 32 * c32, v);
#pragma unroll
        for (int e = 0; e < 32; ++e) final_base[st_base + (size_t)(64 * hf + 32 * c32 + e) * kD] = v[e];
      }
    }
  } else {
    // ======================= RMSNormGated epilogue: thread = state column j, tokens [32 th, 32 th + 32)
    const int ew = warp - kChainWarps, q = ew & 3, th = ew >> 2, j = 32 * q + lane, et = tid - kChainThreads;
    const float scale = rsqrtf((float)kD);
    float *part = reinterpret_cast<float *>(sm + S_PART);
    float *inv = reinterpret_cast<float *>(sm + S_INV);
    int z_issued = 0, z_done = 0;
    auto issue_z = [&](int cc) {
      if (et == 0) {
        tc::mbar_arrive_expect_tx(bar + B_Z + (cc & 1), 64 * kD * 2);
        tc::tma_load_2d(sm + S_Z + (cc & 1) * 16384, &zmap, h * kD, s0 + kC * cc, bar + B_Z + (cc & 1));
      }
      z_issued = cc + 1;
    };
    auto wait_epi = [&](uint64_t *b, uint32_t parity) {
      const bool ok = tc::mbar_wait(b, parity);
      tc::fence_after_sync();
      return tc::named_barrier_or(kBarEpiTs, kEpiThreads, !ok);
    };
    if (!with_out) {  // a chain without outputs: only hand D1 and O2 back each chunk
      for (int c = 0; c < nch; ++c) {
        if (wait_epi(bar + B_ORDY, (uint32_t)c & 1)) { failed = true; break; }
        tc::fence_before_sync();
        tc::named_barrier(kBarEpiTs, kEpiThreads);
        if (et == 0) tc::mbar_arrive(bar + B_ODONE);
      }
      if (failed && et == 0) set_status(p.status, kDevTimeout);
    } else {
    if (nch > 0) issue_z(0);
    if (nch > 1) issue_z(1);
    for (int c = 0; c < nch; ++c) {
      const int b = c & 1;
      const uint32_t par = (c >> 1) & 1;
      const int t0 = s0 + kC * c, Lc = min(kC, s1 - t0);
      float gam[32];  // gamma of this thread's tokens, from the chunk's image (its ring slot may be refilled)
      {
        const float4 *gp = reinterpret_cast<const float4 *>(vslot(g0 + c) + kCGam) + 8 * th;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float4 g4 = gp[e];
          gam[4 * e] = g4.x; gam[4 * e + 1] = g4.y; gam[4 * e + 2] = g4.z; gam[4 * e + 3] = g4.w;
        }
      }
      if (wait_epi(bar + B_ORDY, (uint32_t)c & 1)) { failed = true; break; }
      float o[32];
      {
        uint32_t r1[32], r2[32];
        tc::tmem_ld32_issue(tmem + lane_off + COL_D + 32 * th, r1);
        tc::tmem_ld32_issue(tmem + lane_off + COL_O2 + 32 * th, r2);
        tc::tmem_ld_wait_regs(r1);
        tc::tmem_ld_wait_regs(r2);
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = fmaf(gam[e], __uint_as_float(r1[e]), __uint_as_float(r2[e]));
      }
      tc::fence_before_sync();
      tc::named_barrier(kBarEpiTs, kEpiThreads);
      if (et == 0) tc::mbar_arrive(bar + B_ODONE);  // D1 and O2 are read: the next chunk's products may write them
      {  // per token: the sum over j of o^2 (o = -scale (gamma D1 + O2)), across lanes and then lane quarters
        float sq[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) sq[e] = o[e] * o[e];
        part[q * 64 + 32 * th + lane] = reduce_scatter<32>(sq, lane);  // token 32 th + lane
      }
      tc::named_barrier(kBarEpiTs, kEpiThreads);
      if (et < kC) {
        const float tot = part[et] + part[64 + et] + part[128 + et] + part[192 + et];
        inv[et] = -scale * rsqrtf(tot * (scale * scale / kD) + kEpsRms);
      }
      if (wait_epi(bar + B_Z + b, par)) { failed = true; break; }  // also publishes inv[]
      z_done = c + 1;
      tc::bulk_wait_read();  // the previous chunk's y copies have left S_Y
      tc::named_barrier(kBarEpiTs, kEpiThreads);
      const __nv_bfloat16 *zt = reinterpret_cast<const __nv_bfloat16 *>(sm + S_Z + b * 16384) + 32 * th * kD + j;
      __nv_bfloat16 *yt = reinterpret_cast<__nv_bfloat16 *>(sm + S_Y) + 32 * th * kD + j;
      const float hw = 0.5f * sWn[j];
      {
        float z[32];  // every load before any store: the y tile and the z tile are not known apart
#pragma unroll
        for (int e = 0; e < 32; ++e) z[e] = __bfloat162float(zt[e * kD]);
#pragma unroll
        for (int e = 0; e < 32; e += 4) {  // o / rms(o) for four tokens
          const float4 iv = *reinterpret_cast<const float4 *>(inv + 32 * th + e);
          o[e] *= iv.x; o[e + 1] *= iv.y; o[e + 2] *= iv.z; o[e + 3] *= iv.w;
        }
#pragma unroll
        for (int e = 0; e < 32; e += 2) {  // token pairs: packed fp32 arithmetic
          // silu(z) w = (w / 2) z (1 + tanh(z / 2)), the hardware tanh (as the epilogue of the split pass)
          const float2 zz = make_float2(z[e], z[e + 1]);
          const float2 hz = tc::mul2(zz, tc::splat2(0.5f));
          const float2 g = tc::fma2(zz, make_float2(tc::tanh_approx(hz.x), tc::tanh_approx(hz.y)), zz);
          const float2 y = tc::mul2(make_float2(o[e], o[e + 1]), tc::mul2(g, tc::splat2(hw)));
          z[e] = y.x;
          z[e + 1] = y.y;
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) yt[e * kD] = __float2bfloat16_rn(z[e]);
      }
      tc::fence_before_sync();
      tc::fence_async_smem();
      tc::named_barrier(kBarEpiTs, kEpiThreads);
      if (c + 2 < nch) issue_z(c + 2);  // into the z buffer just consumed
      if (Lc == kC) {
        if (et == 0) {
          tc::tma_store_2d(&omap, h * kD, t0, sm + S_Y);
          tc::bulk_commit();
        }
      } else if (et < Lc) {  // a sequence's last, short chunk: only its own rows
        tc::bulk_s2g(out + ((size_t)(t0 + et) * h_v + h) * kD, sm + S_Y + et * kD * 2, kD * 2);
        tc::bulk_commit();
      }
    }
    tc::bulk_wait_all();
    if (failed) {
      if (et == 0) set_status(p.status, kDevTimeout);
      for (int cc = z_done; cc < z_issued; ++cc) tc::mbar_wait(bar + B_Z + (cc & 1), (cc >> 1) & 1);
    }
    }
  }
  if (tid == 0)  // copies in flight must land before the CTA's shared memory goes away
    for (int c = issued - kSets < 0 ? 0 : issued - kSets; c < issued; ++c)
      tc::mbar_wait(bar + B_FULL + c % kSets, (uint32_t)(c / kSets) & 1);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

// ================================================================ segment-parallel prefill
// For few long chains: every sequence is cut into segments of `seg` chunks.
// The state after segment s is affine in the state before it,
// H_out = M_s H_in + B_s, with B_s the state the segment leaves from a zero
// state and M_s the product of the chunks' maps H -> gamma_C H - K~^T W H (the
// segment run on the identity with U' taken as zero).  So one state pass runs,
// all at once, the first segment of each sequence for real (outputs and its
// end state), every later segment from a zero state (B_s), and every middle
// segment's M_s; a scan H_in(s + 1) = M_s H_in(s) + B_s gives each segment's
// true start state; a second state pass reruns the later segments from those
// states for their outputs and the sequence's final state.
struct SegTab {
  int max_seg;       // upper bound on the segments (host)
  int seg;           // chunks per segment
  int *seq_seg0;     // [N + 1]: first segment of each sequence; [N] = segments
  SegRun *runs1;     // [2 max_seg]: pass 1 (per segment: its run, then its transfer run)
  SegRun *runs3;     // [max_seg]: pass 2 (the reruns)
  float *bufB, *bufM, *bufH;  // [max_seg][h_v][d_k][d_v] each: B_s, M_s, H_in(s)
};

__global__ void __launch_bounds__(1024) seg_table_kernel(const PrefillParams p, const Ws ws, SegTab st) {
  __shared__ int scan[1024];
  const int N = p.N, tid = threadIdx.x;
  const int per = (N + 1023) / 1024;
  const int n0 = min(N, tid * per), n1 = min(N, n0 + per);
  auto nseg_of = [&](int n) {
    const int s0 = p.cu_seqlens[n], s1 = p.cu_seqlens[n + 1];
    const int nch = (s0 >= 0 && s1 >= s0 && s1 <= p.T) ? (s1 - s0 + kC - 1) / kC : 0;
    return max(1, (nch + st.seg - 1) / st.seg);  // an empty (or invalid) sequence: one empty segment
  };
  int cnt = 0;
  for (int n = n0; n < n1; ++n) cnt += nseg_of(n);
  scan[tid] = cnt;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {  // inclusive scan
    const int v = tid >= off ? scan[tid - off] : 0;
    __syncthreads();
    scan[tid] += v;
    __syncthreads();
  }
  const int total = scan[1023];
  const bool overflow = total > st.max_seg;  // only with invalid cu_seqlens (reported by the chunk table)
  int k = scan[tid] - cnt;
  const size_t state = (size_t)p.h_v * kD * kD;
  for (int n = n0; n < n1; ++n) {
    const int nseg = nseg_of(n);
    st.seq_seg0[n] = overflow ? 0 : k;
    const int s0 = p.cu_seqlens[n], s1 = p.cu_seqlens[n + 1];
    const bool ok = !overflow && s0 >= 0 && s1 >= s0 && s1 <= p.T &&
                    ws.chunk_base[n + 1] - ws.chunk_base[n] == (s1 - s0 + kC - 1) / kC;  // else reported
    for (int sg = 0; sg < nseg && !overflow; ++sg, ++k) {
      SegRun r, t, r3;
      r.s0 = ok ? min(s1, s0 + sg * st.seg * kC) : 0;
      r.s1 = ok ? min(s1, r.s0 + st.seg * kC) : 0;
      r.g0 = ok ? ws.chunk_base[n] + sg * st.seg : 0;
      t = r3 = r;
      // pass 1: the first segment for real; the others from a zero state
      r.flags = sg == 0 ? kRunOut : 0;
      r.init = (sg == 0 && p.init_state) ? p.init_state + (size_t)n * state : nullptr;
      r.final = (nseg == 1) ? (p.final_state ? p.final_state + (size_t)n * state : nullptr) : st.bufB + (size_t)k * state;
      // pass 1: the transfer of a middle segment (the scan needs M_s for 1 <= s <= nseg - 2)
      const bool middle = sg >= 1 && sg + 1 < nseg;
      t.flags = kRunTransfer;
      t.init = nullptr;
      t.final = middle ? st.bufM + (size_t)k * state : nullptr;
      if (!middle) t.s1 = t.s0;  // nothing to run
      // pass 2: the later segments from their true start states
      r3.flags = kRunOut;
      r3.init = st.bufH + (size_t)k * state;
      r3.final = (sg + 1 == nseg && p.final_state) ? p.final_state + (size_t)n * state : nullptr;
      if (sg == 0) { r3.s1 = r3.s0; r3.init = nullptr; r3.final = nullptr; }
      st.runs1[2 * k] = r;
      st.runs1[2 * k + 1] = t;
      st.runs3[k] = r3;
    }
  }
  if (tid == 1023) st.seq_seg0[N] = overflow ? 0 : total;
  // the runs past the last segment (all of them on an overflow) do nothing
  for (int r = (overflow ? 0 : total) + tid; r < st.max_seg; r += 1024) {
    SegRun z;
    z.s0 = z.s1 = z.g0 = 0;
    z.flags = 0;
    z.init = nullptr;
    z.final = nullptr;
    st.runs1[2 * r] = z;
    st.runs1[2 * r + 1] = z;
    st.runs3[r] = z;
  }
}

// The scan over a sequence's segments, per (sequence, value head, 16 state
// columns): H_in(1) = B_0 (segment 0's true end state), then
// H_in(s + 1) = M_s H_in(s) + B_s, in fp32.  Each step stages M_s in shared
// memory (rows padded to 132 floats); thread (ti, tj) keeps rows ti + 32 r
// (r < 4) x columns [2 tj, 2 tj + 2) of the product in registers.  A warp
// holds 4 consecutive ti and the 8 tj, so per 4 steps of m its reads of M
// (4 rows x 16 bytes per r) and of H (8 column pairs) are one wavefront each.
// The next step's M is loaded into registers while this step's product runs.
constexpr int kScanCols = 16, kScanThreads = 256, kScanPitch = kD + 4;
constexpr size_t kScanSmem = sizeof(float) * ((size_t)kD * kScanPitch + (size_t)kD * kScanCols);
__global__ void __launch_bounds__(kScanThreads) seg_scan_kernel(const PrefillParams p, SegTab st) {
  extern __shared__ __align__(16) float smem_scan[];
  float *sM = smem_scan;                   // [128 i][kScanPitch]: M_s
  float *sH = sM + kD * kScanPitch;        // [128 m][kScanCols]: the running H_in
  constexpr int kBlocks = kD / kScanCols;
  const int cb = blockIdx.x % kBlocks, h = (blockIdx.x / kBlocks) % p.h_v;
  const int n = blockIdx.x / (kBlocks * p.h_v);
  const int k0 = st.seq_seg0[n], nseg = st.seq_seg0[n + 1] - k0;
  if (nseg < 2) return;
  const size_t state = (size_t)p.h_v * kD * kD, head = (size_t)h * kD * kD;
  const int tid = threadIdx.x, j0 = kScanCols * cb, ti = tid >> 3, tj = tid & 7;
  for (int e = tid; e < kD * kScanCols; e += kScanThreads) {  // H = B_0
    const int i = e / kScanCols, jj = e % kScanCols;
    sH[e] = st.bufB[(size_t)k0 * state + head + (size_t)i * kD + j0 + jj];
  }
  constexpr int kMq = kD * kD / 4 / kScanThreads;  // float4 of M per thread
  float4 mreg[kMq];
  auto load_m = [&](int k) {  // M_k, row-major [i][m]: float4 q of this thread is float4 tid + 256 q
    const float4 *M = reinterpret_cast<const float4 *>(st.bufM + (size_t)k * state + head);
#pragma unroll
    for (int q = 0; q < kMq; ++q) mreg[q] = M[tid + kScanThreads * q];
  };
  if (nseg > 2) load_m(k0 + 1);
  __syncthreads();
  for (int sg = 1; sg < nseg; ++sg) {
    const int k = k0 + sg;
    for (int e = tid; e < kD * kScanCols; e += kScanThreads) {
      const int i = e / kScanCols, jj = e % kScanCols;
      st.bufH[(size_t)k * state + head + (size_t)i * kD + j0 + jj] = sH[e];
    }
    if (sg + 1 == nseg) break;
#pragma unroll
    for (int q = 0; q < kMq; ++q) {
      const int f = tid + kScanThreads * q;  // float4 f of M: row f / 32, columns 4 (f % 32) ...
      *reinterpret_cast<float4 *>(sM + (f >> 5) * kScanPitch + 4 * (f & 31)) = mreg[q];
    }
    __syncthreads();
    if (sg + 2 < nseg) load_m(k + 1);  // in flight during the product
    const float *B = st.bufB + (size_t)k * state + head + j0 + 2 * tj;
    float acc[4][2];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float2 b2 = *reinterpret_cast<const float2 *>(B + (size_t)(ti + 32 * r) * kD);
      acc[r][0] = b2.x;
      acc[r][1] = b2.y;
    }
#pragma unroll 2
    for (int m = 0; m < kD; m += 4) {
      float2 hr[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) hr[c] = *reinterpret_cast<const float2 *>(sH + (m + c) * kScanCols + 2 * tj);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float4 mr = *reinterpret_cast<const float4 *>(sM + (ti + 32 * r) * kScanPitch + m);
        acc[r][0] = fmaf(mr.x, hr[0].x, acc[r][0]); acc[r][1] = fmaf(mr.x, hr[0].y, acc[r][1]);
        acc[r][0] = fmaf(mr.y, hr[1].x, acc[r][0]); acc[r][1] = fmaf(mr.y, hr[1].y, acc[r][1]);
        acc[r][0] = fmaf(mr.z, hr[2].x, acc[r][0]); acc[r][1] = fmaf(mr.z, hr[2].y, acc[r][1]);
        acc[r][0] = fmaf(mr.w, hr[3].x, acc[r][0]); acc[r][1] = fmaf(mr.w, hr[3].y, acc[r][1]);
      }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 4; ++r)
      *reinterpret_cast<float2 *>(sH + (ti + 32 * r) * kScanCols + 2 * tj) = make_float2(acc[r][0], acc[r][1]);
    __syncthreads();
  }
}

// ================================================================ host side
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D map over a [rows][cols] bf16 tensor, boxes of box_cols columns x box_rows
// rows; out-of-range rows read as zero.
bool make_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_cols,
              uint32_t box_rows) {
  auto encode = tensor_map_encoder();
  if (!encode) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The U' images of the chunk prep as a 3-D fp16 tensor [slots][256 rows][32] (rows of 64 bytes; slot
// stride `slot_bytes`), boxes of one slot, 64-byte swizzle.
bool make_up_map(CUtensorMap *m, const void *base, uint64_t slots, uint64_t slot_bytes) {
  auto encode = tensor_map_encoder();
  if (!encode) return false;
  cuuint64_t dims[3] = {32, 256, slots};
  cuuint64_t strides[2] = {64, slot_bytes};
  cuuint32_t box[3] = {32, 256, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t prefill_tc_workspace_bytes(int T, int N, int h_qk, int h_v) { return WsLayout(T, N, h_qk, h_v).total; }

namespace {

// How the state pass runs.  It is bound by each chain's per-chunk latency, a
// good part of which is the copy of the chunk's operand set (~60 KB); 4 slices
// of 32 columns.  When every CTA fits on an SM of its own (few chains: the
// 4096-token workload has 32 chains, 128 CTAs), a ring of 3 operand sets lets
// the copies of the next chunks stream in while one is computed (0.114 against
// 0.127 ms with the next best, 8 slices at two CTAs per SM); with more chains
// one set per kind at two CTAs per SM keeps twice the chains in flight (the
// ring, at one CTA per SM, took 0.806 against 0.624 ms on the 32768-token
// varlen workload).  Measured and not taken: 2 slices of 64 columns and one
// 128-column CTA per chain (no faster with many chains, slower with few).
bool state_ring(const PrefillParams &p) {
  static int sms[64];
  static std::once_flag once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  dev = dev < 0 || dev >= 64 ? 0 : dev;
  std::call_once(once[dev], [dev] {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    sms[dev] = v > 0 ? v : 1;
  });
  return 4L * p.N * p.h_v <= (long)sms[dev];
}
constexpr int kStateSlices = 4;
static_assert(kD / kStateSlices == 32, "the prep writes U' in slices of 32 state columns");

template <int NS, int ST>
cudaError_t launch_state(const PrefillParams &p, const Ws &ws, cudaStream_t s) {
  using C = StateCfg<NS, ST>;
  CUtensorMap zmap, omap;
  std::memset(&zmap, 0, sizeof(zmap));
  std::memset(&omap, 0, sizeof(omap));
  if (p.T > 0 && !(make_map(&zmap, p.z, (uint64_t)p.T, (uint64_t)p.h_v * kD, C::kBV, kC) &&
                   make_map(&omap, p.out, (uint64_t)p.T, (uint64_t)p.h_v * kD, C::kBV, kC)))
    return cudaErrorInvalidValue;
  auto kern = state_kernel<NS, ST>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.N * (unsigned)p.h_v * NS);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = NS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // many chains: the prologue runs beside the prep's last CTAs.  Few chains (one
  // CTA per SM): clusters placed while the prep still holds SMs ran slower.
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = ST == 0 ? 2 : 1;
  trace_begin(s, GDN_K_STATE);
  e = cudaLaunchKernelEx(&cfg, kern, p, ws, zmap, omap);
  trace_end(s);
  return e;
}

cudaError_t launch_state_ts(const PrefillParams &p, const Ws &ws, cudaStream_t s, unsigned chains) {
  CUtensorMap zmap, omap;
  std::memset(&zmap, 0, sizeof(zmap));
  std::memset(&omap, 0, sizeof(omap));
  if (p.T > 0 && !(make_map(&zmap, p.z, (uint64_t)p.T, (uint64_t)p.h_v * kD, kD, kC) &&
                   make_map(&omap, p.out, (uint64_t)p.T, (uint64_t)p.h_v * kD, kD, kC)))
    return cudaErrorInvalidValue;
  cudaError_t e =
      cudaFuncSetAttribute(state_ts_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ts::kSmem);
  if (e != cudaSuccess) return e;
  if (chains == 0) return cudaSuccess;
  trace_begin(s, GDN_K_STATE);
  state_ts_kernel<<<chains * (unsigned)p.h_v, ts::kThreads, ts::kSmem, s>>>(p, ws, zmap, omap);
  trace_end(s);
  return cudaGetLastError();
}

}  // namespace

namespace {

Ws make_ws(const PrefillParams &p, const WsLayout &L, bool compact) {
  Ws ws;
  ws.chunk_base = reinterpret_cast<int *>(p.ws + L.base);
  ws.seq_order = reinterpret_cast<int *>(p.ws + L.order);
  ws.chunk_info = reinterpret_cast<int4 *>(p.ws + L.info);
  ws.vs = p.ws + L.vs;
  ws.max_chunks = L.max_chunks;
  ws.compact = compact ? 1 : 0;
  ws.qs = ws.vs + (size_t)L.max_chunks * p.h_v * kCSlot;
  ws.runs = nullptr;
  return ws;
}

// The chunk table and the chunk prep (all chunks in parallel).
cudaError_t launch_table_and_prep(const PrefillParams &p, const Ws &ws, cudaStream_t s) {
  trace_begin(s, GDN_K_CHUNK_TABLE);
  chunk_table_kernel<<<1, 1024, 0, s>>>(p, ws);
  trace_end(s);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.T > 0) {
    // the common two value heads per q/k head with its head counts fixed at compile time
    auto prep = p.h_v == 2 * p.h_qk ? chunk_prep_kernel<2> : chunk_prep_kernel<0>;
    e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPrepSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ws.max_chunks, (unsigned)(p.h_qk * ((p.h_v / p.h_qk + kMaxRep - 1) / kMaxRep)));
    cfg.blockDim = dim3(kPrepThreads);
    cfg.dynamicSmemBytes = kPrepSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // launched while the table runs
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    CUtensorMap upmap;
    std::memset(&upmap, 0, sizeof(upmap));
    if (!make_up_map(&upmap, ws.vs + (ws.compact ? kCUp : kVUp), (uint64_t)ws.max_chunks * p.h_v,
                     ws.compact ? kCSlot : kVSlot))
      return cudaErrorInvalidValue;
    trace_begin(s, GDN_K_CHUNK_PREP);
    e = cudaLaunchKernelEx(&cfg, prep, p, ws, upmap);
    trace_end(s);
  }
  return e;
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillParams &p, cudaStream_t s) {
  if (p.N <= 0) return cudaSuccess;
  const WsLayout L(p.T, p.N, p.h_qk, p.h_v);
  if (p.ws_bytes < L.total) return cudaErrorInvalidValue;
  // Few chains (every split-column cluster on SMs of its own): the split state
  // pass with a ring of operand sets has the shorter chain (1.6 against 2.0 us
  // per chunk on the 4096-token workload); otherwise one CTA per chain.
  const bool split_pass = state_ring(p);
  const Ws ws = make_ws(p, L, !split_pass);
  cudaError_t e = launch_table_and_prep(p, ws, s);
  if (e != cudaSuccess) return e;
  return split_pass ? launch_state<kStateSlices, 3>(p, ws, s) : launch_state_ts(p, ws, s, (unsigned)p.N);
}

size_t prefill_segmented_workspace_bytes(int T, int N, int h_qk, int h_v, int seg) {
  if (seg < 1) return 0;
  const WsLayout L(T, N, h_qk, h_v);
  const size_t max_seg = (size_t)(((T + kC - 1) / kC + N) / seg + N + 1);
  size_t off = (L.total + 255) / 256 * 256;
  off += (size_t)(N + 1) * sizeof(int);
  off = (off + 255) / 256 * 256 + 3 * max_seg * sizeof(SegRun);
  off = (off + 1023) / 1024 * 1024;
  return off + 3 * max_seg * (size_t)h_v * kD * kD * sizeof(float);
}

cudaError_t launch_prefill_segmented(const PrefillParams &p, int seg, cudaStream_t s) {
  if (p.N <= 0) return cudaSuccess;
  if (seg < 1 || p.ws_bytes < prefill_segmented_workspace_bytes(p.T, p.N, p.h_qk, p.h_v, seg))
    return cudaErrorInvalidValue;
  const WsLayout L(p.T, p.N, p.h_qk, p.h_v);
  Ws ws = make_ws(p, L, true);
  SegTab st;
  st.seg = seg;
  st.max_seg = (int)(((p.T + kC - 1) / kC + p.N) / seg + p.N + 1);
  size_t off = (L.total + 255) / 256 * 256;
  st.seq_seg0 = reinterpret_cast<int *>(p.ws + off);
  off += (size_t)(p.N + 1) * sizeof(int);
  off = (off + 255) / 256 * 256;
  st.runs1 = reinterpret_cast<SegRun *>(p.ws + off);
  st.runs3 = st.runs1 + 2 * (size_t)st.max_seg;
  off += 3 * (size_t)st.max_seg * sizeof(SegRun);
  off = (off + 1023) / 1024 * 1024;
  const size_t buf = (size_t)st.max_seg * p.h_v * kD * kD;
  st.bufB = reinterpret_cast<float *>(p.ws + off);
  st.bufM = st.bufB + buf;
  st.bufH = st.bufM + buf;

  cudaError_t e = launch_table_and_prep(p, ws, s);
  if (e != cudaSuccess) return e;
  trace_begin(s, GDN_K_SEG_SCAN);
  seg_table_kernel<<<1, 1024, 0, s>>>(p, ws, st);
  trace_end(s);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  ws.runs = st.runs1;
  if ((e = launch_state_ts(p, ws, s, 2u * (unsigned)st.max_seg)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(seg_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kScanSmem)) !=
      cudaSuccess)
    return e;
  trace_begin(s, GDN_K_SEG_SCAN);
  seg_scan_kernel<<<(unsigned)p.N * p.h_v * (kD / kScanCols), kScanThreads, kScanSmem, s>>>(p, st);
  trace_end(s);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  ws.runs = st.runs3;
  return launch_state_ts(p, ws, s, (unsigned)st.max_seg);
}

}  // namespace gdn
