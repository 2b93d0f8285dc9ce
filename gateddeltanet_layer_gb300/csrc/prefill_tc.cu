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
//                       U' = T diag(beta) V on the tensor cores; writes the
//                       state pass's MMA operands, already in their shared-
//                       memory image, to the workspace.
//   state_kernel        one CTA per (sequence, value head) chain: H lives in
//                       tensor memory (as S, lane j over d_v); per chunk three
//                       MMA groups  (P^T = S K^T, D2a = S Q^T),  U^T = U'^T -
//                       P^T (T diag(beta gamma))^T,  (D2b = U^T A_Q^T,
//                       S += U^T K~), and the RMSNormGated epilogue; the next
//                       chunk's operands stream in by TMA while it works.
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
// q, k, the SiLU-conv'd v of O(1) inputs, T diag(beta), P and the state).  The
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
constexpr int kPad = 65;  // fp32 64 x 64 matrices: padded rows

// ---------------------------------------------------------------- workspace
// Per (chunk, q/k head): the K and Q images ([64 rows][128 cols] fp16 SW128).
// Per (chunk, value head): A_Q [64][64], T diag(beta gamma) [64][64],
// U'^T [128][64], K~^T [128][64] (fp16 SW128 images) and gamma [64] fp32.
constexpr uint32_t kQkSlot = 32768;
constexpr uint32_t kQkK = 0, kQkQ = 16384;
constexpr uint32_t kVSlot = 50176;
constexpr uint32_t kVAq = 0, kVTbg = 8192, kVUp = 16384, kVKt = 32768, kVGam = 49152;

struct Ws {
  int *chunk_base;   // [N + 1]: first chunk of each sequence; [N] = number of chunks
  int2 *chunk_info;  // [max_chunks]: (sequence, first token)
  uint8_t *qk;       // [max_chunks][h_qk] x kQkSlot
  uint8_t *vs;       // [max_chunks][h_v] x kVSlot
  int max_chunks;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WsLayout {
  size_t base, info, qk, vs, total;
  int max_chunks;
  WsLayout(int T, int N, int h_qk, int h_v) {
    max_chunks = (T + kC - 1) / kC + N;
    base = 0;
    info = align_up(sizeof(int) * (size_t)(N + 1), 1024);
    qk = align_up(info + sizeof(int2) * (size_t)max_chunks, 1024);
    vs = qk + (size_t)max_chunks * h_qk * kQkSlot;
    total = vs + (size_t)max_chunks * h_v * kVSlot;
  }
};

// ---------------------------------------------------------------- helpers
__device__ __forceinline__ void mma_chain(uint32_t d, uint32_t a, int a_rows, int a_row0, uint32_t b, int b_rows,
                                          int b_row0, int ksteps, uint32_t idesc, bool acc) {
  for (int k = 0; k < ksteps; ++k)
    tc::mma16(d, tc::sdesc_kstep(a, a_rows, a_row0, k), tc::sdesc_kstep(b, b_rows, b_row0, k), idesc,
              (acc || k > 0) ? 1u : 0u);
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

// SiLU x sigmoid(x) with one special-function op: e^-x by the fast exponential,
// then 1 / (1 + e^-x) by two Newton-Raphson steps y <- y (2 - d y) from the
// classic bit-pattern reciprocal seed (relative error < 1e-5 after the two
// steps, far below the fp16 rounding of the result).
__device__ __forceinline__ float silu_fast(float x) {
  const float d = fminf(1.0f + __expf(-x), 1e30f);
  float y = __int_as_float(0x7EF311C7 - __float_as_int(d));
  y = y * (2.0f - d * y);
  y = y * (2.0f - d * y);
  return x * y;
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
__device__ __forceinline__ void st_chunk_f16_global(uint8_t *dst, const float *x) {
  uint4 u;
  u.x = tc::pack_f16x2(x[0], x[1]);
  u.y = tc::pack_f16x2(x[2], x[3]);
  u.z = tc::pack_f16x2(x[4], x[5]);
  u.w = tc::pack_f16x2(x[6], x[7]);
  *reinterpret_cast<uint4 *>(dst) = u;
}

// ================================================================ chunk table
__global__ void __launch_bounds__(1024) chunk_table_kernel(const PrefillParams p, Ws ws) {
  __shared__ int scan[1024];
  __shared__ int bad;
  const int N = p.N, tid = threadIdx.x;
  if (tid == 0) bad = 0;
  const int per = (N + 1023) / 1024;
  const int n0 = min(N, tid * per), n1 = min(N, n0 + per);
  int cnt = 0;
  for (int n = n0; n < n1; ++n) {
    const int s0 = p.cu_seqlens[n], s1 = p.cu_seqlens[n + 1];
    if (s0 >= 0 && s1 >= s0 && s1 <= p.T) cnt += (s1 - s0 + kC - 1) / kC;
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
    ws.chunk_info[g] = make_int2(lo, p.cu_seqlens[lo] + kC * (g - ws.chunk_base[lo]));
  }
}

// ================================================================ chunk prep
constexpr int kPrepThreads = 256;
// shared memory (from a 1024-aligned base)
constexpr uint32_t P_KQ = 0;                          // [K; Q] hi fp16 [128][128]
constexpr uint32_t P_KQL = 32768;                     // [K; Q] lo, later A and T fp32 [64][65]
constexpr uint32_t P_AF = P_KQL;
constexpr uint32_t P_TF = P_AF + 64 * kPad * 4;
constexpr uint32_t P_VT = 66560;                      // V^T fp16 [128 j][64 m]
constexpr uint32_t P_TB = P_VT + 16384;               // T diag(beta) fp16 [64 r][64 m]
constexpr uint32_t P_XF = P_TB + 8192;                // inverse block products 32 x 32 fp32
constexpr int kMaxRep = 8;                            // value heads per q/k head
constexpr uint32_t P_VEC = P_XF + 4096;               // per value head: G, gamma, beta, decay-to-end
constexpr uint32_t P_RED = P_VEC + kMaxRep * 1024;
constexpr uint32_t P_MISC = P_RED + 64;
constexpr size_t kPrepSmem = P_MISC + 64 + 1024;
static_assert(P_TF + 64 * kPad * 4 <= P_VT, "A and T fit over the lo tile");
static_assert(P_VT % 1024 == 0 && P_TB % 1024 == 0, "SW128 tiles 1024-aligned");
static_assert(2 * kPrepSmem <= 232448, "two prep CTAs per SM");

constexpr uint32_t kIdN64 = tc::idesc_f16(128, 64);
constexpr uint32_t kIdN128 = tc::idesc_f16(128, 128);

// conv(4) + SiLU of 8 rows x 4 channels of one head: rows r0 .. r0+7 of the
// chunk, channels c0 .. c0+3 (x points at channel c0 of token 0; bf16 row
// pitch `stride` elements; conv_w rows from `ch`).  Rows before the sequence
// start or past the chunk's end are 0.
__device__ __forceinline__ void conv_rows(const __nv_bfloat16 *x, size_t stride, const float *conv_w, int ch,
                                          int t0, int s0, int Lc, int r0, float (&y)[8][4]) {
  float4 w[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) w[c] = *reinterpret_cast<const float4 *>(conv_w + (size_t)(ch + c) * 4);
  uint2 xr[11];  // packed bf16 rows
#pragma unroll
  for (int rr = 0; rr < 11; ++rr) {
    const int row = r0 - 3 + rr;
    const int t = t0 + row;
    xr[rr] = (t >= s0 && row < Lc) ? *reinterpret_cast<const uint2 *>(x + (size_t)t * stride) : make_uint2(0u, 0u);
  }
  auto val = [&](int rr, int c) {
    const uint32_t w32 = (c < 2) ? xr[rr].x : xr[rr].y;
    return __uint_as_float((c & 1) ? (w32 & 0xFFFF0000u) : (w32 << 16));
  };
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const bool ok = r0 + r < Lc;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float a = w[c].x * val(r, c);
      a = fmaf(w[c].y, val(r + 1, c), a);
      a = fmaf(w[c].z, val(r + 2, c), a);
      a = fmaf(w[c].w, val(r + 3, c), a);
      y[r][c] = ok ? silu_fast(a) : 0.0f;
    }
  }
}

// L2-normalise the 8 rows held by a warp (each lane holds 4 of the 128 channels).
__device__ __forceinline__ void l2norm_rows(float (&y)[8][4], int lane) {
  float ss[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) ss[r] = y[r][0] * y[r][0] + y[r][1] * y[r][1] + y[r][2] * y[r][2] + y[r][3] * y[r][3];
  const float mine = reduce_scatter<8>(ss, lane);  // lane l: row l >> 2
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const float inv = rsqrtf(__shfl_sync(0xffffffffu, mine, 4 * r) + kEpsL2);
#pragma unroll
    for (int c = 0; c < 4; ++c) y[r][c] *= inv;
  }
}

__global__ void __launch_bounds__(kPrepThreads, 2) chunk_prep_kernel(const PrefillParams p, const Ws ws) {
  const int g = blockIdx.x, hq = blockIdx.y;
  const int total = ws.chunk_base[p.N];
  if (g >= total) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sbase = tc::smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int lr = tid & 127, gh = tid >> 7;
  const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
  const int h_v = p.h_v, h_qk = p.h_qk, rep = h_v / h_qk;

  const int2 info = ws.chunk_info[g];
  const int n = info.x, t0 = info.y;
  const int s0 = p.cu_seqlens[n], s1 = p.cu_seqlens[n + 1];
  const int Lc = min(kC, s1 - t0);

  float *AF = reinterpret_cast<float *>(sm + P_AF);
  float *TF = reinterpret_cast<float *>(sm + P_TF);
  float *XF = reinterpret_cast<float *>(sm + P_XF);
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
    tc::tmem_alloc(tmem_slot, 128);
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
  constexpr int COL_P1 = 0, COL_UP = 64;
  uint32_t phase = 0;
  bool failed = false;

  uint8_t *qk_slot = ws.qk + ((size_t)g * h_qk + hq) * kQkSlot;
  const int r0 = 8 * warp, c0 = 4 * lane;  // prologue: this thread's rows and channels
  auto v_slot_of = [&](int vv) { return ws.vs + ((size_t)g * h_v + hq * rep + vv) * kVSlot; };

  // ---------------- gates of every value head and their running sums inside the chunk
  for (int v0 = 0; v0 < rep; v0 += 4) {
    const int vv = v0 + (tid >> 6), r = tid & 63;
    float gsum = 0.0f;
    if (vv < rep) {
      const int h = hq * rep + vv;
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
    if (vv < rep) {
      if (r >= 32) gsum += carry[vv & 3];
      sG[vv * 256 + r] = gsum;
      const float gm = expf(gsum);
      sG[vv * 256 + 64 + r] = gm;
      *reinterpret_cast<float *>(v_slot_of(vv) + kVGam + 4 * r) = gm;
    }
    __syncthreads();
    if (vv < rep) sG[vv * 256 + 192 + r] = expf(sG[vv * 256 + 63] - sG[vv * 256 + r]);
    __syncthreads();
  }

  // ---------------- q and k: conv + SiLU + L2 norm -> [K; Q] hi / lo tiles, K and Q images,
  //                  and K~^T = (diag(e^(G_C - G)) K)^T images of every value head
  {
    float y[8][4], kreg[8][4];
    conv_rows(xq + hq * kD + c0, qk_stride, p.conv_w, hq * kD + c0, t0, s0, Lc, r0, y);
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
      *reinterpret_cast<uint2 *>(qk_slot + kQkQ + tc::sw128_offset(64, r0 + r, c0)) = hi;
    }
    conv_rows(xk + hq * kD + c0, qk_stride, p.conv_w, h_qk * kD + hq * kD + c0, t0, s0, Lc, r0, kreg);
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
      *reinterpret_cast<uint2 *>(qk_slot + kQkK + tc::sw128_offset(64, r0 + r, c0)) = hi;
    }
    for (int vv = 0; vv < rep; ++vv) {
      const float *dec = sG + vv * 256 + 192;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float kt[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) kt[r] = kreg[r][c] * dec[r0 + r];
        st_chunk_f16_global(v_slot_of(vv) + kVKt + tc::sw128_chunk(128, c0 + c, warp), kt);
      }
    }
  }
  publish_operands();

  // ---------------- P1 = [K; Q] K^T (hi.hi + hi.lo + lo.hi): rows 0..63 K K^T, 64..127 Q K^T
  if (tid == 0) {
    mma_chain(tmem + COL_P1, sbase + P_KQ, 128, 0, sbase + P_KQ, 128, 0, 8, kIdN64, false);
    mma_chain(tmem + COL_P1, sbase + P_KQ, 128, 0, sbase + P_KQL, 128, 0, 8, kIdN64, true);
    mma_chain(tmem + COL_P1, sbase + P_KQL, 128, 0, sbase + P_KQ, 128, 0, 8, kIdN64, true);
    tc::mma_commit(bar);
  }

  for (int vv = 0; vv < rep && !failed; ++vv) {
    const int h = hq * rep + vv;
    uint8_t *v_slot = v_slot_of(vv);

    const float *sG = sGall + vv * 256, *sGam = sG + 64, *sBeta = sG + 128;

    // ---------------- v: conv + SiLU -> V^T tile
    {
      float y[8][4];
      conv_rows(xv + h * kD + c0, v_stride, p.conv_w, 2 * h_qk * kD + h * kD + c0, t0, s0, Lc, r0, y);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float col[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) col[r] = y[r][c];
        tc::st_chunk_f16(sm + P_VT + tc::sw128_chunk(128, c0 + c, warp), col);
      }
    }
    if (vv == 0) {
      if (wait_all(bar, phase)) { failed = true; break; }
    }

    // ---------------- A (fp32, strictly lower) and A_Q (image)
    {
      float v[32];
      tc::tmem_ld32(tmem + lane_off + COL_P1 + 32 * gh, v);
      float Gs[32];  // shared-memory reads before the stores below
#pragma unroll
      for (int q = 0; q < 32; ++q) Gs[q] = sG[32 * gh + q];
      if (lr < 64) {
        const int r = lr;
        const float Gr = sG[r], br = sBeta[r];
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          const int s = 32 * gh + q;
          v[q] = (s < r) ? br * __expf(Gr - Gs[q]) * v[q] : 0.0f;
        }
#pragma unroll
        for (int q = 0; q < 32; ++q) AF[r * kPad + 32 * gh + q] = v[q];
      } else {
        const int r = lr - 64;
        const float Gr = sG[r];
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          const int s = 32 * gh + q;
          v[q] = (s <= r) ? __expf(Gr - Gs[q]) * v[q] : 0.0f;
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) st_chunk_f16_global(v_slot + kVAq + tc::sw128_chunk(64, r, 4 * gh + cc), v + 8 * cc);
      }
    }
    tc::fence_before_sync();
    __syncthreads();

    // ---------------- T = (I + A)^-1 by recursive doubling on the unit lower-triangular L = I + A
    // (a) the four diagonal 16x16 blocks by forward substitution, one column per thread
    if (tid < 64) {
      const int bb = tid >> 4, s = tid & 15;
      float x[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        const float *arow = AF + (16 * bb + r) * kPad + 16 * bb;
        float acc0 = (r == s) ? 1.0f : 0.0f, acc1 = 0.0f;
#pragma unroll
        for (int m = 0; m + 1 < r; m += 2) {
          acc0 = fmaf(-arow[m], x[m], acc0);
          acc1 = fmaf(-arow[m + 1], x[m + 1], acc1);
        }
        if (r & 1) acc0 = fmaf(-arow[r - 1], x[r - 1], acc0);
        x[r] = acc0 + acc1;
      }
#pragma unroll
      for (int r = 0; r < 16; ++r) TF[(16 * bb + r) * kPad + 16 * bb + s] = x[r];
    }
    __syncthreads();
    // (b) T_10 = -T_11 (A_10 T_00) and T_32 = -T_33 (A_32 T_22): two elements per thread
    {
      float xv2[2];
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int e = tid + kPrepThreads * it;
        const int blk = e >> 8, r = (e >> 4) & 15, s = e & 15, o = 32 * blk;
        const float *arow = AF + (o + 16 + r) * kPad + o;
        float acc0 = 0.0f, acc1 = 0.0f;
#pragma unroll
        for (int k = 0; k < 16; k += 2) {  // T_00 is lower triangular
          const float ta = (k >= s) ? TF[(o + k) * kPad + o + s] : 0.0f;
          const float tb = (k + 1 >= s) ? TF[(o + k + 1) * kPad + o + s] : 0.0f;
          acc0 = fmaf(arow[k], ta, acc0);
          acc1 = fmaf(arow[k + 1], tb, acc1);
        }
        xv2[it] = acc0 + acc1;
      }
#pragma unroll
      for (int it = 0; it < 2; ++it) XF[tid + kPrepThreads * it] = xv2[it];
      __syncthreads();
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int e = tid + kPrepThreads * it;
        const int blk = e >> 8, r = (e >> 4) & 15, s = e & 15, o = 32 * blk;
        const float *trow = TF + (o + 16 + r) * kPad + o + 16;
        float acc0 = 0.0f, acc1 = 0.0f;
#pragma unroll
        for (int k = 0; k < 16; k += 2) {  // T_11 is lower triangular
          acc0 = fmaf((k <= r) ? trow[k] : 0.0f, XF[blk * 256 + k * 16 + s], acc0);
          acc1 = fmaf((k + 1 <= r) ? trow[k + 1] : 0.0f, XF[blk * 256 + (k + 1) * 16 + s], acc1);
        }
        TF[(o + 16 + r) * kPad + o + s] = -(acc0 + acc1);
      }
    }
    __syncthreads();
    // (c) the lower-left 32x32 block T_21 = -T_2 (A_21 T_1): four rows per thread
    {
      const int rb = tid >> 5, s = tid & 31;  // rows rb, rb+8, rb+16, rb+24
      float y[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int k = 0; k < 32; ++k) {  // T_1 is lower triangular
        const float t = (k >= s) ? TF[k * kPad + s] : 0.0f;
#pragma unroll
        for (int q = 0; q < 4; ++q) y[q] = fmaf(AF[(32 + rb + 8 * q) * kPad + k], t, y[q]);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) XF[(rb + 8 * q) * 32 + s] = y[q];
      __syncthreads();
      float z[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int k = 0; k < 32; ++k) {  // T_2 is lower triangular
        const float yk = XF[k * 32 + s];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int r = rb + 8 * q;
          z[q] = fmaf((k <= r) ? TF[(32 + r) * kPad + 32 + k] : 0.0f, yk, z[q]);
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) TF[(32 + rb + 8 * q) * kPad + s] = -z[q];
    }
    __syncthreads();
    // T diag(beta) (shared-memory operand) and T diag(beta gamma) (image)
    {
      const int r = tid & 63, oq = tid >> 6;  // columns [16 oq, 16 oq + 16)
      float a16[16], b16[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {  // shared-memory reads before the stores below
        const int m = 16 * oq + e;
        const float t = (m <= r) ? TF[r * kPad + m] : 0.0f;
        b16[e] = t * sBeta[m];
        a16[e] = b16[e] * sGam[m];
      }
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        tc::st_chunk_f16(sm + P_TB + tc::sw128_chunk(64, r, 2 * oq + hh), b16 + 8 * hh);
        st_chunk_f16_global(v_slot + kVTbg + tc::sw128_chunk(64, r, 2 * oq + hh), a16 + 8 * hh);
      }
    }
    publish_operands();

    // ---------------- U'^T = V^T (T diag(beta))^T -> image
    if (tid == 0) {
      mma_chain(tmem + COL_UP, sbase + P_VT, 128, 0, sbase + P_TB, 64, 0, 4, kIdN64, false);
      tc::mma_commit(bar);
    }
    if (wait_all(bar, phase)) { failed = true; break; }
    {
      float u[32];
      tc::tmem_ld32(tmem + lane_off + COL_UP + 32 * gh, u);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) st_chunk_f16_global(v_slot + kVUp + tc::sw128_chunk(128, lr, 4 * gh + cc), u + 8 * cc);
    }
    tc::fence_before_sync();
    __syncthreads();  // V^T, T, A are reused by the next value head
  }
  if (failed && tid == 0) set_status(p.status, kDevTimeout);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 128);
}

// ================================================================ state pass
// Warps 0-7 (256 threads) run the state chain; warps 8-11 (128 threads) run
// the RMSNormGated epilogue of the previous chunk at the same time, handed
// over through two mbarriers (o-ready: main -> epilogue; o-done: back).
constexpr int kMainThreads = 256;
constexpr int kOutThreads = 128;
constexpr int kStateThreads = kMainThreads + kOutThreads;
constexpr int kBarMain = 1, kBarOut = 2;  // named barriers of the two groups
constexpr uint32_t S_SB = 0;          // S fp16 [128 j][128 i]
constexpr uint32_t S_KH = 32768;      // K image [64][128]    } one bulk set (with gamma)
constexpr uint32_t S_QH = 49152;      // Q image [64][128]    }
constexpr uint32_t S_AQ = 65536;      // A_Q image            } one bulk set
constexpr uint32_t S_KTT = 73728;     // K~^T image           }
constexpr uint32_t S_TBG = 90112;     // T diag(beta gamma)   } one bulk set
constexpr uint32_t S_UP = 98304;      // U'^T image           }
constexpr uint32_t S_Z = 114688;      // z rows [64][256 B] (TMA tensor copy)
constexpr uint32_t S_PT = 131072;     // -P^T fp16 [128 j][64 m]
constexpr uint32_t S_US = 147456;     // U^T fp16 [128 j][64 r]
constexpr uint32_t S_OUT = 163840;    // y rows [64][256 B] bf16, stored by TMA
constexpr uint32_t S_GAM = 180224;    // gamma [64] (bulk, with K and Q)
constexpr uint32_t S_GAML = S_GAM + 256;  // gamma of the last two chunks [2][64]
constexpr uint32_t S_RED = S_GAML + 512;
constexpr uint32_t S_INV = S_RED + 2048;
constexpr uint32_t S_MISC = S_INV + 256;
constexpr size_t kStateSmem = S_MISC + 128 + 1024;
static_assert(S_US % 1024 == 0 && S_KTT % 1024 == 0 && S_TBG % 1024 == 0, "SW128 tiles 1024-aligned");
static_assert(S_OUT % 128 == 0 && S_Z % 128 == 0, "TMA boxes 128-byte aligned");
static_assert(kStateSmem <= 232448, "shared memory budget");

// tensor memory: S, P^T, D2a (two buffers: chunk c's epilogue reads one while
// chunk c+1's first MMA group writes the other), D2b, X
constexpr int COL_S = 0, COL_PM = 128, COL_D2A = 192, COL_D2B = 320, COL_X = 384;

__global__ void __launch_bounds__(kStateThreads, 1) state_kernel(const PrefillParams p, const Ws ws,
                                                                 const __grid_constant__ CUtensorMap zmap,
                                                                 const __grid_constant__ CUtensorMap omap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sbase = tc::smem_u32(sm);
  const int h_v = p.h_v, h_qk = p.h_qk;
  const int n = blockIdx.x / h_v, h = blockIdx.x % h_v;
  const int hq = h / (h_v / h_qk);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int lr = tid & 127;
  const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
  const bool is_main = tid < kMainThreads;

  const int s0 = p.cu_seqlens[n], s1 = p.cu_seqlens[n + 1];
  if (s0 < 0 || s1 < s0 || s1 > p.T) return;  // reported by the chunk table
  const int g0 = ws.chunk_base[n], g1 = ws.chunk_base[n + 1];
  if (g1 - g0 != (s1 - s0 + kC - 1) / kC) return;  // table overflow (invalid cu_seqlens), reported

  const float *sGamIn = reinterpret_cast<const float *>(sm + S_GAM);
  float *sGamL = reinterpret_cast<float *>(sm + S_GAML);
  float *red = reinterpret_cast<float *>(sm + S_RED);
  float *sInv = reinterpret_cast<float *>(sm + S_INV);
  uint64_t *bar = reinterpret_cast<uint64_t *>(sm + S_MISC);
  uint64_t *bar_kq = bar + 1, *bar_aq = bar + 2, *bar_tu = bar + 3, *bar_z = bar + 4;
  uint64_t *bar_oready = bar + 5, *bar_odone = bar + 6;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + S_MISC + 64);
  __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out);

  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, 512);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < 7; ++i) tc::mbar_init(bar + i, 1);
    tc::fence_mbar_init();
    tc::prefetch_tmap(&zmap);
    tc::prefetch_tmap(&omap);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  bool failed = false;

  if (is_main) {
    // ======================= state chain (warps 0-7)
    const int gh = tid >> 7;
    uint32_t ph = 0, ph_kq = 0, ph_aq = 0, ph_tu = 0, ph_odone = 0;
    int pend_kq = 0, pend_aq = 0, pend_tu = 0;
    auto qk_slot = [&](int gg) { return ws.qk + ((size_t)gg * h_qk + hq) * kQkSlot; };
    auto v_slot = [&](int gg) { return ws.vs + ((size_t)gg * h_v + h) * kVSlot; };
    auto issue_kq = [&](int gg) {
      if (tid == 0) {
        tc::mbar_arrive_expect_tx(bar_kq, 2 * 16384 + 256);
        tc::bulk_g2s(sm + S_KH, qk_slot(gg) + kQkK, 16384, bar_kq);
        tc::bulk_g2s(sm + S_QH, qk_slot(gg) + kQkQ, 16384, bar_kq);
        tc::bulk_g2s(sm + S_GAM, v_slot(gg) + kVGam, 256, bar_kq);
      }
    };
    auto issue_aq = [&](int gg) {
      if (tid == 0) {
        tc::mbar_arrive_expect_tx(bar_aq, 8192 + 16384);
        tc::bulk_g2s(sm + S_AQ, v_slot(gg) + kVAq, 8192, bar_aq);
        tc::bulk_g2s(sm + S_KTT, v_slot(gg) + kVKt, 16384, bar_aq);
      }
    };
    auto issue_tu = [&](int gg) {
      if (tid == 0) {
        tc::mbar_arrive_expect_tx(bar_tu, 8192 + 16384);
        tc::bulk_g2s(sm + S_TBG, v_slot(gg) + kVTbg, 8192, bar_tu);
        tc::bulk_g2s(sm + S_UP, v_slot(gg) + kVUp, 16384, bar_tu);
      }
    };
    // wait (all 256 main threads) for a phase; true if it ran out
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
    // S (fp32, tensor memory) -> its fp16 copy, then S <- gamma_C S for the
    // coming chunk's update (gamma_C from the freshly loaded gamma vector).
    auto copy_and_scale_state = [&]() {
      const float gC = sGamIn[63];
      float v[32];
      for (int c0 = 0; c0 < 64; c0 += 32) {
        tc::tmem_ld32(tmem + lane_off + COL_S + 64 * gh + c0, v);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
          tc::st_chunk_f16(sm + S_SB + tc::sw128_chunk(128, lr, 8 * gh + (c0 >> 3) + cc), v + 8 * cc);
#pragma unroll
        for (int q = 0; q < 32; ++q) v[q] *= gC;
        tc::tmem_st32(tmem + lane_off + COL_S + 64 * gh + c0, v);
      }
    };

    // ---------------- initial state -> TMEM S (fp32)
    const size_t st_off = ((size_t)n * h_v + h) * kD * kD;
    {
      float v[32];
      for (int c0 = 0; c0 < 64; c0 += 32) {
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          const int i = 64 * gh + c0 + q;
          v[q] = p.init_state ? p.init_state[st_off + (size_t)i * kD + lr] : 0.0f;
        }
        tc::tmem_st32(tmem + lane_off + COL_S + 64 * gh + c0, v);
      }
    }
    tc::fence_before_sync();
    tc::named_barrier(kBarMain, kMainThreads);
    tc::fence_after_sync();
    if (g1 > g0) {
      issue_kq(g0);
      issue_tu(g0);
      issue_aq(g0);
      pend_kq = pend_tu = pend_aq = 1;
      if (wait_main(bar_kq, ph_kq)) failed = true;
      if (!failed) {
        pend_kq = 0;
        if (tid < 64) sGamL[tid] = sGamIn[tid];
        copy_and_scale_state();
      }
    }
    publish_main();

    for (int g = g0; g < g1 && !failed; ++g) {
      const int buf = (g - g0) & 1;
      const bool more = g + 1 < g1;

      // ---------------- group 1: P^T = S K^T, D2a = S Q^T (S entering the chunk, fp16 copy)
      if (tid == 0) {
        mma_chain(tmem + COL_PM, sbase + S_SB, 128, 0, sbase + S_KH, 64, 0, 8, kIdN64, false);
        mma_chain(tmem + COL_D2A + 64 * buf, sbase + S_SB, 128, 0, sbase + S_QH, 64, 0, 8, kIdN64, false);
        tc::mma_commit(bar);
      }
      if (wait_main(bar, ph)) { failed = true; break; }
      if (more) {
        tc::fence_async_smem();
        issue_kq(g + 1);
        pend_kq = 1;
      }
      {  // -P^T -> fp16 operand
        float v[32];
        tc::tmem_ld32(tmem + lane_off + COL_PM + 32 * gh, v);
#pragma unroll
        for (int q = 0; q < 32; ++q) v[q] = -v[q];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tc::st_chunk_f16(sm + S_PT + tc::sw128_chunk(128, lr, 4 * gh + cc), v + 8 * cc);
      }
      publish_main();

      // ---------------- group 2: X = -P^T (T diag(beta gamma))^T;  U^T = U'^T + X
      if (wait_main(bar_tu, ph_tu)) { failed = true; break; }
      pend_tu = 0;
      if (tid == 0) {
        mma_chain(tmem + COL_X, sbase + S_PT, 128, 0, sbase + S_TBG, 64, 0, 4, kIdN64, false);
        tc::mma_commit(bar);
      }
      if (wait_main(bar, ph)) { failed = true; break; }
      {
        float u[32];
        tc::tmem_ld32(tmem + lane_off + COL_X + 32 * gh, u);
        uint4 raw[4];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
          raw[cc] = *reinterpret_cast<const uint4 *>(sm + S_UP + tc::sw128_chunk(128, lr, 4 * gh + cc));
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const __half2 *hp = reinterpret_cast<const __half2 *>(&raw[cc]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __half22float2(hp[e]);
            u[8 * cc + 2 * e] += f.x;
            u[8 * cc + 2 * e + 1] += f.y;
          }
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tc::st_chunk_f16(sm + S_US + tc::sw128_chunk(128, lr, 4 * gh + cc), u + 8 * cc);
      }
      publish_main();
      if (more) {
        tc::fence_async_smem();
        issue_tu(g + 1);
        pend_tu = 1;
      }

      // ---------------- group 3: D2b = U^T A_Q^T;  S += U^T K~   (S already scaled by gamma_C)
      if (g > g0) {  // the epilogue has read the previous chunk's D2b
        if (wait_main(bar_odone, ph_odone)) { failed = true; break; }
      }
      if (wait_main(bar_aq, ph_aq)) { failed = true; break; }
      pend_aq = 0;
      if (tid == 0) {
        mma_chain(tmem + COL_D2B, sbase + S_US, 128, 0, sbase + S_AQ, 64, 0, 4, kIdN64, false);
        mma_chain(tmem + COL_S, sbase + S_US, 128, 0, sbase + S_KTT, 128, 0, 4, kIdN128, true);
        tc::mma_commit(bar);
      }
      if (wait_main(bar, ph)) { failed = true; break; }
      if (tid == 0) {  // this chunk's D2a, D2b and gamma are ready for the epilogue
        tc::fence_before_sync();
        tc::mbar_arrive(bar_oready);
      }
      if (more) {
        tc::fence_async_smem();
        issue_aq(g + 1);
        pend_aq = 1;
      }

      // ---------------- next chunk's fp16 state copy (and gamma_C scaling of S)
      if (more) {
        if (wait_main(bar_kq, ph_kq)) { failed = true; break; }
        pend_kq = 0;
        if (tid < 64) sGamL[64 * (buf ^ 1) + tid] = sGamIn[tid];
        copy_and_scale_state();
      }
      publish_main();
    }

    if (failed) {
      if (tid == 0) set_status(p.status, kDevTimeout);
      // copies still in flight must land before the CTA's shared memory goes away
      if (pend_kq) tc::mbar_wait(bar_kq, ph_kq & 1);
      if (pend_aq) tc::mbar_wait(bar_aq, ph_aq & 1);
      if (pend_tu) tc::mbar_wait(bar_tu, ph_tu & 1);
    } else if (p.final_state) {
      float v[32];
      for (int c0 = 0; c0 < 64; c0 += 32) {
        tc::tmem_ld32(tmem + lane_off + COL_S + 64 * gh + c0, v);
#pragma unroll
        for (int q = 0; q < 32; ++q) p.final_state[st_off + (size_t)(64 * gh + c0 + q) * kD + lr] = v[q];
      }
    }
  } else {
    // ======================= RMSNormGated epilogue (warps 8-11), one chunk behind
    const int otid = tid - kMainThreads, ow = warp - 8;  // lane j = otid
    uint32_t ph_oready = 0, ph_z = 0;
    int pend_z = 0;
    const float scale = rsqrtf((float)kD);
    const float wj = p.norm_w[lr];
    auto issue_z = [&](int t0_) {
      if (otid == 0) {
        tc::mbar_arrive_expect_tx(bar_z, kC * 256);
        tc::tma_load_2d(sm + S_Z, &zmap, h * kD, t0_, bar_z);
      }
    };
    auto wait_out = [&](uint64_t *b, uint32_t &phase) {
      const bool ok = tc::mbar_wait(b, phase & 1);
      ++phase;
      tc::fence_after_sync();
      return tc::named_barrier_or(kBarOut, kOutThreads, !ok);
    };
    if (g1 > g0) {
      issue_z(s0);
      pend_z = 1;
    }
    for (int g = g0; g < g1; ++g) {
      const int t0 = s0 + kC * (g - g0);
      const int Lc = min(kC, s1 - t0);
      const int buf = (g - g0) & 1;
      if (wait_out(bar_oready, ph_oready)) { failed = true; break; }
      // o = scale (gamma_r D2a + D2b) for this lane j and the chunk's 64 tokens
      float o[64];
      {
        float d[32];
        const float *gam = sGamL + 64 * buf;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float a32[32];
          tc::tmem_ld32(tmem + lane_off + COL_D2A + 64 * buf + 32 * hh, a32);
          tc::tmem_ld32(tmem + lane_off + COL_D2B + 32 * hh, d);
#pragma unroll
          for (int q = 0; q < 32; ++q) o[32 * hh + q] = scale * fmaf(gam[32 * hh + q], a32[q], d[q]);
        }
      }
      // D2a, D2b and gamma are read: the state chain may overwrite them
      tc::fence_before_sync();
      tc::named_barrier(kBarOut, kOutThreads);
      if (otid == 0) tc::mbar_arrive(bar_odone);
      // per-token sum of squares over j (the 128 lanes of the four epilogue warps)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float sq[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) sq[q] = o[32 * hh + q] * o[32 * hh + q];
        red[(hh * 4 + ow) * 32 + lane] = reduce_scatter<32>(sq, lane);
      }
      if (otid < 64) tc::bulk_wait_read();  // the previous chunk's y rows have left S_OUT
      tc::named_barrier(kBarOut, kOutThreads);
      if (otid < 64) {
        const int hh = otid >> 5, q = otid & 31;
        const float ssum = red[(hh * 4) * 32 + q] + red[(hh * 4 + 1) * 32 + q] + red[(hh * 4 + 2) * 32 + q] +
                           red[(hh * 4 + 3) * 32 + q];
        sInv[otid] = rsqrtf(ssum * (1.0f / kD) + kEpsRms);
      }
      if (wait_out(bar_z, ph_z)) { failed = true; break; }
      pend_z = 0;
      const __nv_bfloat16 *zst = reinterpret_cast<const __nv_bfloat16 *>(sm + S_Z);
      __nv_bfloat16 *yst = reinterpret_cast<__nv_bfloat16 *>(sm + S_OUT);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float zz[32], iv[32];  // shared-memory reads before the stores
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          zz[q] = __bfloat162float(zst[(32 * hh + q) * kD + lr]);
          iv[q] = sInv[32 * hh + q];
        }
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          // silu(z) = z (1 + tanh(z / 2)) / 2 with the hardware tanh: its ~2^-11
          // error scales one output element, well inside the output rounding
          const float th = tc::tanh_approx(0.5f * zz[q]);
          o[32 * hh + q] = o[32 * hh + q] * iv[q] * wj * (0.5f * zz[q]) * (1.0f + th);
        }
#pragma unroll
        for (int q = 0; q < 32; ++q) yst[(32 * hh + q) * kD + lr] = __float2bfloat16_rn(o[32 * hh + q]);
      }
      tc::fence_async_smem();
      tc::named_barrier(kBarOut, kOutThreads);
      if (Lc == kC) {
        if (otid == 0) {
          tc::tma_store_2d(&omap, h * kD, t0, sm + S_OUT);
          tc::bulk_commit();
        }
      } else if (otid < Lc) {  // a sequence's last, short chunk: only its own rows
        tc::bulk_s2g(out + ((size_t)(t0 + otid) * h_v + h) * kD, sm + S_OUT + otid * 256, 256);
        tc::bulk_commit();
      }
      if (g + 1 < g1) {  // the z rows of the next chunk, over the ones just used
        tc::fence_async_smem();
        issue_z(t0 + kC);
        pend_z = 1;
      }
    }
    if (otid < 64) tc::bulk_wait_all();
    if (failed) {
      if (otid == 0) set_status(p.status, kDevTimeout);
      if (pend_z) tc::mbar_wait(bar_z, ph_z & 1);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
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

// 2-D map over a [rows][cols] bf16 tensor, boxes of 128 columns x box_rows rows;
// out-of-range rows read as zero.
bool make_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto encode = tensor_map_encoder();
  if (!encode) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t prefill_tc_workspace_bytes(int T, int N, int h_qk, int h_v) { return WsLayout(T, N, h_qk, h_v).total; }

cudaError_t launch_prefill_tc(const PrefillParams &p, cudaStream_t s) {
  if (p.N <= 0) return cudaSuccess;
  const WsLayout L(p.T, p.N, p.h_qk, p.h_v);
  if (p.ws_bytes < L.total) return cudaErrorInvalidValue;
  Ws ws;
  ws.chunk_base = reinterpret_cast<int *>(p.ws + L.base);
  ws.chunk_info = reinterpret_cast<int2 *>(p.ws + L.info);
  ws.qk = p.ws + L.qk;
  ws.vs = p.ws + L.vs;
  ws.max_chunks = L.max_chunks;
  CUtensorMap zmap, omap;
  std::memset(&zmap, 0, sizeof(zmap));
  std::memset(&omap, 0, sizeof(omap));
  if (p.T > 0 && !(make_map(&zmap, p.z, (uint64_t)p.T, (uint64_t)p.h_v * kD, kC) &&
                   make_map(&omap, p.out, (uint64_t)p.T, (uint64_t)p.h_v * kD, kC)))
    return cudaErrorInvalidValue;

  trace_begin(s, GDN_K_CHUNK_TABLE);
  chunk_table_kernel<<<1, 1024, 0, s>>>(p, ws);
  trace_end(s);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.T > 0) {
    e = cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPrepSmem);
    if (e != cudaSuccess) return e;
    trace_begin(s, GDN_K_CHUNK_PREP);
    chunk_prep_kernel<<<dim3((unsigned)L.max_chunks, (unsigned)p.h_qk), kPrepThreads, kPrepSmem, s>>>(p, ws);
    trace_end(s);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  e = cudaFuncSetAttribute(state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStateSmem);
  if (e != cudaSuccess) return e;
  trace_begin(s, GDN_K_STATE);
  state_kernel<<<(unsigned)p.N * (unsigned)p.h_v, kStateThreads, kStateSmem, s>>>(p, ws, zmap, omap);
  trace_end(s);
  return cudaGetLastError();
}

}  // namespace gdn
