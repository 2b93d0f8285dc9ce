// Chunked prefill on the 5th-generation tensor cores (bf16 streams, d_k = d_v = 128).
//
// One CTA per (sequence, value head) chain walks the sequence in chunks of
// C = 64 tokens.  The state H = S^T (d_k x d_v, fp32) stays in tensor memory
// for the whole sequence as S (lane j over d_v, column i over d_k); an fp16
// copy of it in shared memory is the MMA operand.  Per chunk, with G_r the
// running sum of the gates g inside the chunk and gamma_r = exp(G_r)
// (the chunked WY/UT form of the gated delta rule: Yang et al., "Gated Delta
// Networks", ICLR 2025; "Parallelizing Linear Transformers with the Delta
// Rule over Sequence Length", NeurIPS 2024):
//
//   prologue  q, k, v <- silu(conv4(x)); q, k L2-normalised; g, beta per token
//   group 1   P1  = [K; Q] K^T      -> A   = beta_r e^(G_r-G_s) (k_r.k_s)   (s < r)
//                                      A_Q = e^(G_r-G_s) (q_r.k_s)          (s <= r)
//             P^T = S K^T           (P = K H: the entering state seen by each key)
//             D2a = S Q^T
//   inverse   T = (I + A)^-1        (fp32: 16 x 16 diagonal blocks, then 32 x 32 halves)
//   group 2   U^T = V^T (T diag(beta))^T - P^T (T diag(beta gamma))^T
//             (= U' - W H with W = T diag(beta gamma) K: the per-token u_r of the rule)
//   group 3   D2b = U^T A_Q^T;   S <- gamma_C S + U^T K~,   K~ = diag(e^(G_C - G)) K
//   output    o_r = d_k^-1/2 (gamma_r D2a + D2b)[:, r];  y = RMSNorm(o) w silu(z)
//
// Every dense contraction is a tcgen05.mma chain with M = 128 (the transposed
// forms above keep M at d_k or d_v), fp16 operands in 128-byte-swizzled
// K-major shared memory and fp32 accumulators in tensor memory; one thread
// issues, tcgen05.commit signals an mbarrier, and every wait is bounded.  Raw
// stream rows reach shared memory by TMA tensor copies one chunk ahead.
// Decays between two tokens are always exp(G_r - G_s) with r >= s.
//
// Operand precision.  The streams arrive in bf16, but every value the kernel
// computes (conv outputs, T, P, U, the state copy) is rounded to fp16 for the
// tensor cores: 3 more mantissa bits than bf16 at the same MMA rate and
// operand size.  The layer's output is normalised per token (RMSNorm), which
// magnifies the rounding error of rows whose o is small; with bf16 operands
// single outputs drifted by up to 6 % of max(1, |y|), with fp16 by under 1 %.
// Every operand is bounded well inside the fp16 range (|x| <= ~4 for unit-
// normalised q, k, the SiLU-conv'd v of O(1) inputs, T diag(beta), P and the
// state).  The q.k and k.k products of P1 additionally use a hi + lo split
// (q = q_hi + q_lo, both fp16; P1 = hi.hi + hi.lo + lo.hi), which recovers
// ~22 bits for the entries of A and A_Q.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

constexpr int kC = 64;
constexpr int kD = 128;
constexpr int kThreads = 512;
constexpr int kPad = 65;  // fp32 64x64 matrices are stored with a padded row
constexpr int kStageRows = kC + 3;

// Shared-memory map (bytes from a 1024-aligned base).  Operand tiles are fp16,
// 128-byte-swizzled K-major, each on a 1024-byte boundary.
constexpr uint32_t OFF_SB = 0;                   // S            [128 j][128 i]
constexpr uint32_t OFF_KQ = OFF_SB + 32768;      // [K; Q] hi    [128 rows][128 i]; later z rows
constexpr uint32_t OFF_VT = OFF_KQ + 32768;      // V^T          [128 j][64 m]
constexpr uint32_t OFF_KTT = OFF_VT + 16384;     // K~^T         [128 i][64 r]
constexpr uint32_t OFF_AQ = OFF_KTT + 16384;     // A_Q          [64 r][64 s]
constexpr uint32_t OFF_TBG = OFF_AQ + 8192;      // T diag(beta gamma) [64 r][64 m]
constexpr uint32_t OFF_TB = OFF_TBG + 8192;      // T diag(beta)       [64 r][64 m]
constexpr uint32_t OFF_US = OFF_TB + 8192;       // U^T          [128 j][64 r]
constexpr uint32_t OFF_PT = OFF_US + 16384;      // -P^T         [128 j][64 m]
constexpr uint32_t OFF_KQL = OFF_PT + 16384;     // [K; Q] lo    (P1 only) ...
constexpr uint32_t OFF_AF = OFF_KQL;             // ... then A fp32 [64][65]
constexpr uint32_t OFF_TF = OFF_AF + 64 * kPad * 4;  // and T fp32 [64][65]
constexpr uint32_t OFF_XF = OFF_TF + 64 * kPad * 4;  // block products of the inverse, 32 x 32 fp32
constexpr uint32_t OFF_VEC = OFF_XF + 1024 * 4;      // G, gamma, beta, decay-to-end: 4 x 64 fp32
constexpr uint32_t OFF_RED = OFF_VEC + 4 * 64 * 4;   // reductions: 16 x 32 fp32
constexpr uint32_t OFF_INV = OFF_RED + 8 * 64 * 4;   // per-row inverse norms: 64 fp32
constexpr uint32_t OFF_MISC = OFF_INV + 64 * 4;      // mbarriers, TMEM base, scan carry
constexpr uint32_t SMEM_USED = OFF_MISC + 64;
constexpr size_t kSmemBytes = SMEM_USED + 1024;      // + alignment slack
// Raw stream rows, staged by TMA in tiles idle at the time:
//   x rows [3][67][256 B] (q, k, v of rows t0-3 .. t0+63) over A_Q .. -P^T,
//   loaded once the previous chunk's group 3 is done;
//   z rows [64][256 B] over [K; Q], loaded once group 1 is done.
constexpr uint32_t OFF_XST = OFF_AQ;
constexpr uint32_t OFF_ZST = OFF_KQ;
constexpr uint32_t kXTileBytes = kStageRows * 256;

static_assert(OFF_PT % 1024 == 0 && OFF_KQL % 1024 == 0 && OFF_US % 1024 == 0, "SW128 tiles must be 1024-aligned");
static_assert(OFF_KQL + 32768 <= OFF_XF, "the low-part tile fits in the A/T scratch");
static_assert(OFF_XST + 3 * kXTileBytes <= OFF_KQL, "x staging fits in A_Q .. -P^T");
static_assert(kXTileBytes % 128 == 0 && OFF_XST % 128 == 0, "TMA destinations 128-byte aligned");
static_assert(kSmemBytes <= 232448, "shared memory budget");

// Tensor-memory columns (512 allocated).
constexpr int COL_S = 0, COL_D2A = 128, COL_D2B = 192, COL_P1 = 256, COL_PM = 320, COL_X = 384;
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kIdN64 = tc::idesc_f16(128, 64);
constexpr uint32_t kIdN128 = tc::idesc_f16(128, 128);

struct TcMaps {
  CUtensorMap xq, xk, xv, z;  // [T][heads * 128] bf16, boxes of 128 columns x 67 (x) / 64 (z) rows
};

// K-steps of one MMA chain: D (+)= A[rows a_row0..] * B[rows b_row0..]^T over k16 in [0, ksteps).
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
// steps, far below the fp16 rounding of the result).  The reciprocal runs on
// the FMA pipe, which has 8x the throughput of the special-function unit.
__device__ __forceinline__ float silu_fast(float x) {
  const float d = fminf(1.0f + __expf(-x), 1e30f);
  float y = __int_as_float(0x7EF311C7 - __float_as_int(d));
  y = y * (2.0f - d * y);
  y = y * (2.0f - d * y);
  return x * y;
}

// All threads: wait for an MMA commit (or a TMA transaction) phase; true if it
// ran out (every thread then takes the exit path).
__device__ __forceinline__ bool wait_all(uint64_t *bar, uint32_t &phase) {
  const bool ok = tc::mbar_wait(bar, phase & 1);
  ++phase;
  tc::fence_after_sync();
  return __syncthreads_or(!ok) != 0;
}

// Make this thread's shared-memory operand writes and tensor-memory accesses
// visible to the next MMA, then synchronise the CTA.
__device__ __forceinline__ void publish_operands() {
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
}

__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const PrefillParams p,
                                                                  const __grid_constant__ TcMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sbase = tc::smem_u32(sm);

  const int h_v = p.h_v, h_qk = p.h_qk;
  const int n = blockIdx.x / h_v;
  const int h = blockIdx.x % h_v;
  const int hq = h / (h_v / h_qk);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int lr = tid & 127;    // tensor-memory lane of this thread
  const int gq = tid >> 7;     // which quarter of the columns this thread takes
  const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;

  const int s0 = p.cu_seqlens[n], s1 = p.cu_seqlens[n + 1];
  if (s0 < 0 || s1 < s0 || s1 > p.T) {
    if (tid == 0) set_status(p.status, kDevBadSeqlens);
    return;
  }

  float *AF = reinterpret_cast<float *>(sm + OFF_AF);
  float *TF = reinterpret_cast<float *>(sm + OFF_TF);
  float *XF = reinterpret_cast<float *>(sm + OFF_XF);
  float *sG = reinterpret_cast<float *>(sm + OFF_VEC);
  float *sGam = sG + 64;
  float *sBeta = sG + 128;
  float *sDec = sG + 192;
  float *red = reinterpret_cast<float *>(sm + OFF_RED);
  float *sInv = reinterpret_cast<float *>(sm + OFF_INV);
  uint64_t *bar = reinterpret_cast<uint64_t *>(sm + OFF_MISC);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_MISC + 8);
  float *carry = reinterpret_cast<float *>(sm + OFF_MISC + 16);
  uint64_t *bar_x = reinterpret_cast<uint64_t *>(sm + OFF_MISC + 24);
  uint64_t *bar_z = reinterpret_cast<uint64_t *>(sm + OFF_MISC + 32);

  const __nv_bfloat16 *xa = static_cast<const __nv_bfloat16 *>(p.a);
  const __nv_bfloat16 *xb = static_cast<const __nv_bfloat16 *>(p.b);
  __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out);

  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(bar, 1);
    tc::mbar_init(bar_x, 1);
    tc::mbar_init(bar_z, 1);
    tc::fence_mbar_init();
    tc::prefetch_tmap(&maps.xq);
    tc::prefetch_tmap(&maps.xk);
    tc::prefetch_tmap(&maps.xv);
    tc::prefetch_tmap(&maps.z);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  uint32_t phase = 0, phase_x = 0, phase_z = 0;
  bool failed = false, x_pending = false, z_pending = false;

  // q, k, v rows t_next-3 .. t_next+63 -> x staging (rows outside the tensor
  // read as zero; rows of neighbouring sequences are masked where used).
  auto issue_x = [&](int t_next) {
    if (tid == 0) {
      tc::mbar_arrive_expect_tx(bar_x, 3 * kXTileBytes);
      tc::tma_load_2d(sm + OFF_XST, &maps.xq, hq * kD, t_next - 3, bar_x);
      tc::tma_load_2d(sm + OFF_XST + kXTileBytes, &maps.xk, hq * kD, t_next - 3, bar_x);
      tc::tma_load_2d(sm + OFF_XST + 2 * kXTileBytes, &maps.xv, h * kD, t_next - 3, bar_x);
    }
  };
  auto issue_z = [&](int t0_) {
    if (tid == 0) {
      tc::mbar_arrive_expect_tx(bar_z, kC * 256);
      tc::tma_load_2d(sm + OFF_ZST, &maps.z, h * kD, t0_, bar_z);
    }
  };

  // ---------------- initial state -> TMEM S (fp32) and its fp16 copy
  const size_t st_off = ((size_t)n * h_v + h) * kD * kD;
  {
    const int j = lr;
    float v[32];
#pragma unroll
    for (int q = 0; q < 32; ++q) {
      const int i = 32 * gq + q;
      v[q] = p.init_state ? p.init_state[st_off + (size_t)i * kD + j] : 0.0f;
    }
    tc::tmem_st32(tmem + lane_off + COL_S + 32 * gq, v);
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) tc::st_chunk_f16(sm + OFF_SB + tc::sw128_chunk(128, j, 4 * gq + cc), v + 8 * cc);
  }
  publish_operands();

  const float A_exp = expf(p.A_log[h]);
  const float dtb = p.dt_bias[h];
  const float scale = rsqrtf((float)kD);

  // the first chunk's raw rows and gate inputs
  float a_in = 0.0f, b_in = 0.0f;
  if (s1 > s0) {
    issue_x(s0);
    x_pending = true;
    if (tid < 64 && s0 + tid < s1) {
      a_in = __bfloat162float(xa[(size_t)(s0 + tid) * h_v + h]);
      b_in = __bfloat162float(xb[(size_t)(s0 + tid) * h_v + h]);
    }
  }

  for (int t0 = s0; t0 < s1 && !failed; t0 += kC) {
    const int Lc = min(kC, s1 - t0);

    // ---------------- gates and their running sum inside the chunk
    {
      float gsum = 0.0f;
      if (tid < 64) {
        const int r = tid;
        float g = 0.0f, be = 0.0f;
        if (r < Lc) {
          g = gate_g(a_in, A_exp, dtb);
          be = sigmoid_f(b_in);
        }
        gsum = g;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, gsum, off);
          if (lane >= off) gsum += y;
        }
        if (tid == 31) carry[0] = gsum;
        sBeta[r] = be;
      }
      __syncthreads();
      if (tid < 64) {
        if (tid >= 32) gsum += carry[0];
        sG[tid] = gsum;
        sGam[tid] = expf(gsum);
      }
      __syncthreads();
      if (tid < 64) sDec[tid] = expf(sG[63] - sG[tid]);
    }
    if (wait_all(bar_x, phase_x)) { failed = true; break; }
    x_pending = false;

    // ---------------- prologue: conv(4) + SiLU (+ L2 norm) of q, k, v
    // thread -> channels (2cp, 2cp+1), rows [8 rb, 8 rb + 8)
    {
      const int cp = tid & 63, rb = tid >> 6;
      for (int mat = 0; mat < 3; ++mat) {
        const int ch = mat == 0 ? hq * kD + 2 * cp
                       : mat == 1 ? h_qk * kD + hq * kD + 2 * cp
                                  : 2 * h_qk * kD + h * kD + 2 * cp;
        const uint8_t *stage = sm + OFF_XST + (uint32_t)mat * kXTileBytes + 4 * cp;
        const float4 w0 = *reinterpret_cast<const float4 *>(p.conv_w + (size_t)ch * 4);
        const float4 w1 = *reinterpret_cast<const float4 *>(p.conv_w + (size_t)(ch + 1) * 4);
        float x0[11], x1[11];
#pragma unroll
        for (int rr = 0; rr < 11; ++rr) {
          const int row = 8 * rb - 3 + rr;
          if (t0 + row >= s0 && row < Lc) {
            const float2 f =
                __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(stage + (row + 3) * 256));
            x0[rr] = f.x;
            x1[rr] = f.y;
          } else {
            x0[rr] = 0.0f;
            x1[rr] = 0.0f;
          }
        }
        float y0[8], y1[8], ss[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const bool ok = 8 * rb + r < Lc;
          float a0 = w0.x * x0[r];
          a0 = fmaf(w0.y, x0[r + 1], a0);
          a0 = fmaf(w0.z, x0[r + 2], a0);
          a0 = fmaf(w0.w, x0[r + 3], a0);
          float a1 = w1.x * x1[r];
          a1 = fmaf(w1.y, x1[r + 1], a1);
          a1 = fmaf(w1.z, x1[r + 2], a1);
          a1 = fmaf(w1.w, x1[r + 3], a1);
          y0[r] = ok ? silu_fast(a0) : 0.0f;
          y1[r] = ok ? silu_fast(a1) : 0.0f;
          ss[r] = y0[r] * y0[r] + y1[r] * y1[r];
        }
        if (mat < 2) {  // L2 norm over the 128 channels of each row: 64 threads, 2 warps
          const float part = reduce_scatter<8>(ss, lane);
          if ((lane & 3) == 0) red[warp * 8 + (lane >> 2)] = part;
          __syncthreads();
          if (tid < 64) {
            const int rbb = tid >> 3, rr = tid & 7;
            sInv[tid] = rsqrtf(red[(2 * rbb) * 8 + rr] + red[(2 * rbb + 1) * 8 + rr] + kEpsL2);
          }
          __syncthreads();
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            const float inv = sInv[8 * rb + r];
            y0[r] *= inv;
            y1[r] *= inv;
          }
          // [K; Q] rows (K: 0..63, Q: 64..127), high and low fp16 parts
          const int row0 = mat == 0 ? 64 : 0;
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            const __half2 hi = __floats2half2_rn(y0[r], y1[r]);
            const __half2 lo = __floats2half2_rn(y0[r] - __low2float(hi), y1[r] - __high2float(hi));
            const uint32_t off = tc::sw128_offset(128, row0 + 8 * rb + r, 2 * cp);
            *reinterpret_cast<__half2 *>(sm + OFF_KQ + off) = hi;
            *reinterpret_cast<__half2 *>(sm + OFF_KQL + off) = lo;
          }
        }
        if (mat == 1) {  // K~^T = (diag(e^(G_C - G)) K)^T
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            const float dcy = sDec[8 * rb + r];
            y0[r] *= dcy;
            y1[r] *= dcy;
          }
          tc::st_chunk_f16(sm + OFF_KTT + tc::sw128_chunk(128, 2 * cp, rb), y0);
          tc::st_chunk_f16(sm + OFF_KTT + tc::sw128_chunk(128, 2 * cp + 1, rb), y1);
        }
        if (mat == 2) {  // V^T
          tc::st_chunk_f16(sm + OFF_VT + tc::sw128_chunk(128, 2 * cp, rb), y0);
          tc::st_chunk_f16(sm + OFF_VT + tc::sw128_chunk(128, 2 * cp + 1, rb), y1);
        }
      }
    }
    publish_operands();

    // ---------------- group 1: P1 = [K; Q] K^T (hi.hi + hi.lo + lo.hi), P^T = S K^T, D2a = S Q^T
    if (tid == 0) {
      mma_chain(tmem + COL_P1, sbase + OFF_KQ, 128, 0, sbase + OFF_KQ, 128, 0, 8, kIdN64, false);
      mma_chain(tmem + COL_P1, sbase + OFF_KQ, 128, 0, sbase + OFF_KQL, 128, 0, 8, kIdN64, true);
      mma_chain(tmem + COL_P1, sbase + OFF_KQL, 128, 0, sbase + OFF_KQ, 128, 0, 8, kIdN64, true);
      mma_chain(tmem + COL_PM, sbase + OFF_SB, 128, 0, sbase + OFF_KQ, 128, 0, 8, kIdN64, false);
      mma_chain(tmem + COL_D2A, sbase + OFF_SB, 128, 0, sbase + OFF_KQ, 128, 64, 8, kIdN64, false);
      tc::mma_commit(bar);
    }
    // meanwhile: S <- gamma_C S in tensor memory (the MMAs above read the fp16 copy)
    {
      const float gC = sGam[63];
      float v[32];
      tc::tmem_ld32(tmem + lane_off + COL_S + 32 * gq, v);
#pragma unroll
      for (int q = 0; q < 32; ++q) v[q] *= gC;
      tc::tmem_st32(tmem + lane_off + COL_S + 32 * gq, v);
    }
    if (wait_all(bar, phase)) { failed = true; break; }
    // [K; Q] is consumed: stage this chunk's z rows over it
    tc::fence_async_smem();
    issue_z(t0);
    z_pending = true;

    // ---------------- A (fp32, strictly lower), A_Q and -P^T (fp16 operands)
    {
      float v[16];
      tc::tmem_ld16(tmem + lane_off + COL_P1 + 16 * gq, v);
      if (lr < 64) {
        const int r = lr;
        const float Gr = sG[r], br = sBeta[r];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const int s = 16 * gq + q;
          AF[r * kPad + s] = (s < r) ? br * __expf(Gr - sG[s]) * v[q] : 0.0f;
        }
      } else {
        const int r = lr - 64;
        const float Gr = sG[r];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const int s = 16 * gq + q;
          v[q] = (s <= r) ? __expf(Gr - sG[s]) * v[q] : 0.0f;
        }
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) tc::st_chunk_f16(sm + OFF_AQ + tc::sw128_chunk(64, r, 2 * gq + cc), v + 8 * cc);
      }
      tc::tmem_ld16(tmem + lane_off + COL_PM + 16 * gq, v);
#pragma unroll
      for (int q = 0; q < 16; ++q) v[q] = -v[q];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) tc::st_chunk_f16(sm + OFF_PT + tc::sw128_chunk(128, lr, 2 * gq + cc), v + 8 * cc);
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
    // (b) the 32x32 halves: T_10 = -T_11 (A_10 T_00) and T_32 = -T_33 (A_32 T_22)
    {
      const int blk = tid >> 8, r = (tid >> 4) & 15, s = tid & 15;
      const int o = 32 * blk;
      const float *arow = AF + (o + 16 + r) * kPad + o;
      float acc0 = 0.0f, acc1 = 0.0f;
#pragma unroll
      for (int k = 0; k < 16; k += 2) {  // T_00 is lower triangular: rows k < s do not contribute
        const float t0 = (k >= s) ? TF[(o + k) * kPad + o + s] : 0.0f;
        const float t1 = (k + 1 >= s) ? TF[(o + k + 1) * kPad + o + s] : 0.0f;
        acc0 = fmaf(arow[k], t0, acc0);
        acc1 = fmaf(arow[k + 1], t1, acc1);
      }
      XF[blk * 256 + r * 16 + s] = acc0 + acc1;
      __syncthreads();
      const float *trow = TF + (o + 16 + r) * kPad + o + 16;
      acc0 = 0.0f;
      acc1 = 0.0f;
#pragma unroll
      for (int k = 0; k < 16; k += 2) {  // T_11 is lower triangular: columns k > r do not contribute
        const float t0 = (k <= r) ? trow[k] : 0.0f;
        const float t1 = (k + 1 <= r) ? trow[k + 1] : 0.0f;
        acc0 = fmaf(t0, XF[blk * 256 + k * 16 + s], acc0);
        acc1 = fmaf(t1, XF[blk * 256 + (k + 1) * 16 + s], acc1);
      }
      TF[(o + 16 + r) * kPad + o + s] = -(acc0 + acc1);
    }
    __syncthreads();
    // (c) the lower-left 32x32 block: T_21 = -T_2 (A_21 T_1), two rows per thread
    {
      const int r = tid >> 5, s = tid & 31;
      const float *a0 = AF + (32 + r) * kPad, *a1 = AF + (48 + r) * kPad;
      float y0 = 0.0f, y1 = 0.0f, y2 = 0.0f, y3 = 0.0f;
#pragma unroll
      for (int k = 0; k < 32; k += 2) {  // T_1 is lower triangular: rows k < s do not contribute
        const float t0 = (k >= s) ? TF[k * kPad + s] : 0.0f;
        const float t1 = (k + 1 >= s) ? TF[(k + 1) * kPad + s] : 0.0f;
        y0 = fmaf(a0[k], t0, y0);
        y1 = fmaf(a1[k], t0, y1);
        y2 = fmaf(a0[k + 1], t1, y2);
        y3 = fmaf(a1[k + 1], t1, y3);
      }
      XF[r * 32 + s] = y0 + y2;
      XF[(r + 16) * 32 + s] = y1 + y3;
      __syncthreads();
      const float *t0r = TF + (32 + r) * kPad + 32, *t1r = TF + (48 + r) * kPad + 32;
      float z0 = 0.0f, z1 = 0.0f, z2 = 0.0f, z3 = 0.0f;
#pragma unroll
      for (int k = 0; k < 32; k += 2) {  // T_2 is lower triangular: columns k > row do not contribute
        const float yk0 = XF[k * 32 + s], yk1 = XF[(k + 1) * 32 + s];
        z0 = fmaf((k <= r) ? t0r[k] : 0.0f, yk0, z0);
        z2 = fmaf((k + 1 <= r) ? t0r[k + 1] : 0.0f, yk1, z2);
        z1 = fmaf((k <= r + 16) ? t1r[k] : 0.0f, yk0, z1);
        z3 = fmaf((k + 1 <= r + 16) ? t1r[k + 1] : 0.0f, yk1, z3);
      }
      TF[(32 + r) * kPad + s] = -(z0 + z2);
      TF[(48 + r) * kPad + s] = -(z1 + z3);
    }
    __syncthreads();
    // T diag(beta gamma) and T diag(beta) as fp16 operands (rows r, columns m)
    {
      const int r = tid & 63, oq = tid >> 6;
      float a8[8], b8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int m = 8 * oq + e;
        const float t = (m <= r) ? TF[r * kPad + m] : 0.0f;
        b8[e] = t * sBeta[m];
        a8[e] = b8[e] * sGam[m];
      }
      tc::st_chunk_f16(sm + OFF_TBG + tc::sw128_chunk(64, r, oq), a8);
      tc::st_chunk_f16(sm + OFF_TB + tc::sw128_chunk(64, r, oq), b8);
    }
    publish_operands();

    // ---------------- group 2: U^T = V^T (T diag(beta))^T + (-P^T) (T diag(beta gamma))^T
    if (tid == 0) {
      mma_chain(tmem + COL_X, sbase + OFF_VT, 128, 0, sbase + OFF_TB, 64, 0, 4, kIdN64, false);
      mma_chain(tmem + COL_X, sbase + OFF_PT, 128, 0, sbase + OFF_TBG, 64, 0, 4, kIdN64, true);
      tc::mma_commit(bar);
    }
    if (wait_all(bar, phase)) { failed = true; break; }
    // U^T (lane j) -> fp16 operand rows j, columns r
    {
      float u[16];
      tc::tmem_ld16(tmem + lane_off + COL_X + 16 * gq, u);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) tc::st_chunk_f16(sm + OFF_US + tc::sw128_chunk(128, lr, 2 * gq + cc), u + 8 * cc);
    }
    publish_operands();

    // ---------------- group 3: D2b = U^T A_Q^T;  S += U^T K~
    if (tid == 0) {
      mma_chain(tmem + COL_D2B, sbase + OFF_US, 128, 0, sbase + OFF_AQ, 64, 0, 4, kIdN64, false);
      mma_chain(tmem + COL_S, sbase + OFF_US, 128, 0, sbase + OFF_KTT, 128, 0, 4, kIdN128, true);
      tc::mma_commit(bar);
    }
    if (wait_all(bar, phase)) { failed = true; break; }
    // A_Q .. -P^T are consumed: stage the next chunk's raw rows there
    if (t0 + kC < s1) {
      tc::fence_async_smem();
      issue_x(t0 + kC);
      x_pending = true;
      if (tid < 64 && t0 + kC + tid < s1) {
        a_in = __bfloat162float(xa[(size_t)(t0 + kC + tid) * h_v + h]);
        b_in = __bfloat162float(xb[(size_t)(t0 + kC + tid) * h_v + h]);
      }
    }

    // ---------------- output: o = scale (gamma_r D2a + D2b), RMSNormGated, store
    {
      const int j = lr;
      float o[16], d2b[16];
      tc::tmem_ld16(tmem + lane_off + COL_D2A + 16 * gq, o);
      tc::tmem_ld16(tmem + lane_off + COL_D2B + 16 * gq, d2b);
      float sq[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        o[q] = scale * fmaf(sGam[16 * gq + q], o[q], d2b[q]);
        sq[q] = o[q] * o[q];
      }
      const float part = reduce_scatter<16>(sq, lane);
      // warp w (quarter gq = w / 4) covers j in [32 (w & 3), +32) and tokens [16 gq, +16)
      if ((lane & 1) == 0) red[warp * 16 + (lane >> 1)] = part;
      __syncthreads();
      if (tid < 64) {
        const int qq = tid >> 4, q = tid & 15;
        const float ssum = red[(4 * qq) * 16 + q] + red[(4 * qq + 1) * 16 + q] + red[(4 * qq + 2) * 16 + q] +
                           red[(4 * qq + 3) * 16 + q];
        sInv[tid] = rsqrtf(ssum * (1.0f / kD) + kEpsRms);
      }
      const bool zok = tc::mbar_wait(bar_z, phase_z & 1);
      ++phase_z;
      if (__syncthreads_or(!zok)) { failed = true; break; }
      z_pending = false;
      const float wj = p.norm_w[j];
      const __nv_bfloat16 *zst = reinterpret_cast<const __nv_bfloat16 *>(sm + OFF_ZST);
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int r = 16 * gq + q;
        if (r < Lc) {
          const float zz = __bfloat162float(zst[r * kD + j]);
          out[((size_t)(t0 + r) * h_v + h) * kD + j] = __float2bfloat16_rn(o[q] * sInv[r] * wj * silu_fast(zz));
        }
      }
    }
    // next chunk's fp16 copy of S
    {
      float v[32];
      tc::tmem_ld32(tmem + lane_off + COL_S + 32 * gq, v);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tc::st_chunk_f16(sm + OFF_SB + tc::sw128_chunk(128, lr, 4 * gq + cc), v + 8 * cc);
    }
    publish_operands();
  }

  if (failed) {
    if (tid == 0) set_status(p.status, kDevTimeout);
    // copies still in flight must land before the CTA's shared memory goes away
    if (x_pending) tc::mbar_wait(bar_x, phase_x & 1);
    if (z_pending) tc::mbar_wait(bar_z, phase_z & 1);
  } else if (p.final_state) {
    const int j = lr;
    float v[32];
    tc::tmem_ld32(tmem + lane_off + COL_S + 32 * gq, v);
#pragma unroll
    for (int q = 0; q < 32; ++q) p.final_state[st_off + (size_t)(32 * gq + q) * kD + j] = v[q];
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ host side
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

size_t prefill_fused_workspace_bytes() { return 0; }

cudaError_t launch_prefill_fused(const PrefillParams &p, cudaStream_t s) {
  const unsigned grid = (unsigned)p.N * (unsigned)p.h_v;
  if (grid == 0) return cudaSuccess;
  TcMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  if (p.T > 0) {  // with no tokens every chain is empty and no copy is issued
    const bool ok = make_map(&maps.xq, p.q, (uint64_t)p.T, (uint64_t)p.h_qk * kD, kStageRows) &&
                    make_map(&maps.xk, p.k, (uint64_t)p.T, (uint64_t)p.h_qk * kD, kStageRows) &&
                    make_map(&maps.xv, p.v, (uint64_t)p.T, (uint64_t)p.h_v * kD, kStageRows) &&
                    make_map(&maps.z, p.z, (uint64_t)p.T, (uint64_t)p.h_v * kD, kC);
    if (!ok) return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  prefill_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(p, maps);
  return cudaGetLastError();
}

}  // namespace gdn
