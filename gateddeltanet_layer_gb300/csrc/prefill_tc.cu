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
//   P1        [K; Q] K^T                      -> A = beta_r e^(G_r-G_s) (k_r.k_s)  (s < r)
//                                              A_Q = e^(G_r-G_s) (q_r.k_s)         (s <= r)
//   inverse   T = (I + A)^-1                  (fp32, blocked 16x16 forward substitution)
//   P2        W^T  = K^T (T diag(beta gamma))^T,   U'^T = V^T (T diag(beta))^T
//   state     D1   = S W^T,  D2a = S Q^T                  (S entering the chunk, fp16 copy)
//             U^T  = U'^T - D1                             (= the per-token u_r of the rule)
//             D2b  = U^T A_Q^T
//             S   <- gamma_C S + U^T K~,   K~ = diag(e^(G_C - G)) K
//   output    o_r  = d_k^-1/2 (gamma_r D2a + D2b)[:, r];  y = RMSNorm(o) w silu(z)
//
// Every dense contraction (P1, P2, D1, D2a, D2b and the state update) is one
// tcgen05.mma chain with M = 128 (the transposed forms above keep M at d_k or
// d_v), fp16 operands in 128-byte-swizzled K-major shared memory and fp32
// accumulators in tensor memory; one thread issues, tcgen05.commit signals an
// mbarrier, and every wait is bounded.  Decays between two tokens are always
// exp(G_r - G_s) with r >= s.
//
// Operand precision.  The streams arrive in bf16, but every value the kernel
// computes (conv outputs, T, W, U, the state copy) is rounded to fp16 for the
// tensor cores: 3 more mantissa bits than bf16 at the same MMA rate and
// operand size.  The layer's output is normalised per token (RMSNorm), which
// magnifies the rounding error of rows whose o is small; with bf16 operands
// single outputs drifted by up to 6 % of max(1, |y|), with fp16 by under 1 %.
// Every operand is bounded well inside the fp16 range (|x| <= ~4 for unit-
// normalised q, k, the SiLU-conv'd v of O(1) inputs, T diag(beta) and the
// state).  The q.k and k.k products of P1 additionally use a hi + lo split
// (q = q_hi + q_lo, both fp16; P1 = hi.hi + hi.lo + lo.hi), which recovers
// ~22 bits for the entries of A and A_Q.
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

constexpr int kC = 64;
constexpr int kD = 128;
constexpr int kThreads = 256;
constexpr int kPad = 65;  // fp32 64x64 matrices are stored with a padded row

// Shared-memory map (bytes from a 1024-aligned base).  The SW128 operand tiles
// come first, each at a multiple of 1024.
constexpr uint32_t OFF_SB = 0;                  // S fp16        [128 j][128 i]
constexpr uint32_t OFF_KQ = OFF_SB + 32768;     // [K; Q] fp16   [128 rows][128 i]
constexpr uint32_t OFF_KT = OFF_KQ + 32768;     // K^T fp16      [128 i][64 r]
constexpr uint32_t OFF_VT = OFF_KT + 16384;     // V^T fp16      [128 j][64 r]
constexpr uint32_t OFF_KTT = OFF_VT + 16384;    // K~^T fp16     [128 i][64 r]
constexpr uint32_t OFF_WS = OFF_KTT + 16384;    // W fp16        [64 r][128 i]
constexpr uint32_t OFF_AQ = OFF_WS + 16384;     // A_Q fp16      [64 r][64 s]
constexpr uint32_t OFF_TBG = OFF_AQ + 8192;     // T diag(beta gamma) fp16 [64 r][64 m]
constexpr uint32_t OFF_TB = OFF_TBG + 8192;     // T diag(beta) fp16       [64 r][64 m]
constexpr uint32_t OFF_US = OFF_TB + 8192;      // U^T fp16      [128 j][64 r]
constexpr uint32_t OFF_AF = OFF_US + 16384;     // A fp32 [64][65]
constexpr uint32_t OFF_KQL = OFF_AF;            // [K; Q] low parts, fp16 (P1 only; overlays A and T)
constexpr uint32_t OFF_TF = OFF_AF + 64 * kPad * 4;  // T fp32 [64][65]
constexpr uint32_t OFF_XF = OFF_TF + 64 * kPad * 4;  // block products, 3 x 16 x 16 fp32
constexpr uint32_t OFF_VEC = OFF_XF + 3 * 256 * 4;   // G, gamma, beta, dec: 4 x 64 fp32
constexpr uint32_t OFF_RED = OFF_VEC + 4 * 64 * 4;   // reductions: 8 x 64 fp32
constexpr uint32_t OFF_INV = OFF_RED + 8 * 64 * 4;   // per-row inverse norms: 64 fp32
constexpr uint32_t OFF_MISC = OFF_INV + 64 * 4;      // mbarrier, TMEM base, scan carry
constexpr uint32_t SMEM_USED = OFF_MISC + 64;
constexpr size_t kSmemBytes = SMEM_USED + 1024;      // + alignment slack

static_assert(OFF_US % 1024 == 0 && OFF_TB % 1024 == 0 && OFF_KQL % 1024 == 0, "SW128 tiles must be 1024-aligned");
static_assert(OFF_KQL + 32768 <= OFF_XF, "the low-part tile fits in the A/T scratch");
static_assert(kSmemBytes <= 232448, "shared memory budget");

// Tensor-memory columns (512 allocated).
constexpr int COL_S = 0, COL_D1 = 128, COL_D2A = 192, COL_D2B = 256, COL_P1 = 320, COL_UP = 384;
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kIdN64 = tc::idesc_f16(128, 64);
constexpr uint32_t kIdN128 = tc::idesc_f16(128, 128);

// K-steps of one MMA chain: D (+)= A[rows a_row0..] * B[rows b_row0..]^T over k16 in [0, ksteps).
__device__ __forceinline__ void mma_chain(uint32_t d, uint32_t a, int a_rows, int a_row0, uint32_t b, int b_rows,
                                          int b_row0, int ksteps, uint32_t idesc, bool acc) {
  for (int k = 0; k < ksteps; ++k)
    tc::mma16(d, tc::sdesc_kstep(a, a_rows, a_row0, k), tc::sdesc_kstep(b, b_rows, b_row0, k), idesc,
                 (acc || k > 0) ? 1u : 0u);
}

// Sum of v[i] over the 32 lanes of the warp for each i; lane l returns the sum for i = l.
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float send = upper ? v[i] : v[i + off];
      const float keep = upper ? v[i + off] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  return v[0];
}

// Same for 16 values: lane l returns the warp sum for i = l >> 1.
__device__ __forceinline__ float reduce_scatter16(float (&v)[16], int lane) {
#pragma unroll
  for (int off = 16; off >= 2; off >>= 1) {
    const int half = off >> 1;
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

__device__ __forceinline__ float2 ld_bf16x2(const __nv_bfloat16 *p) {
  const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(p);
  return __bfloat1622float2(v);
}

__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sbase = tc::smem_u32(sm);

  const int h_v = p.h_v, h_qk = p.h_qk;
  const int n = blockIdx.x / h_v;
  const int h = blockIdx.x % h_v;
  const int hq = h / (h_v / h_qk);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int lr = tid & 127;    // tensor-memory lane of this thread
  const int gh = tid >> 7;     // which half of the columns this thread takes
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

  const __nv_bfloat16 *xq = static_cast<const __nv_bfloat16 *>(p.q);
  const __nv_bfloat16 *xk = static_cast<const __nv_bfloat16 *>(p.k);
  const __nv_bfloat16 *xv = static_cast<const __nv_bfloat16 *>(p.v);
  const __nv_bfloat16 *xa = static_cast<const __nv_bfloat16 *>(p.a);
  const __nv_bfloat16 *xb = static_cast<const __nv_bfloat16 *>(p.b);
  const __nv_bfloat16 *xz = static_cast<const __nv_bfloat16 *>(p.z);
  __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out);
  const size_t qk_stride = (size_t)h_qk * kD, v_stride = (size_t)h_v * kD;

  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
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

  // ---------------- initial state -> TMEM S (fp32) and its fp16 copy
  const size_t st_off = ((size_t)n * h_v + h) * kD * kD;
  {
    const int j = lr;
    for (int c0 = 0; c0 < 64; c0 += 32) {
      float v[32];
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const int i = 64 * gh + c0 + q;
        v[q] = p.init_state ? p.init_state[st_off + (size_t)i * kD + j] : 0.0f;
      }
      tc::tmem_st32(tmem + lane_off + COL_S + 64 * gh + c0, v);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc)
        tc::st_chunk_f16(sm + OFF_SB + tc::sw128_chunk(128, j, 8 * gh + (c0 >> 3) + cc), v + 8 * cc);
    }
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  const float A_exp = expf(p.A_log[h]);
  const float dtb = p.dt_bias[h];
  const float scale = rsqrtf((float)kD);

  for (int t0 = s0; t0 < s1 && !failed; t0 += kC) {
    const int Lc = min(kC, s1 - t0);

    // ---------------- L2 prefetch of the next chunk's streams
    {
      const int row = tid & 63, mat = tid >> 6;
      const int tn = t0 + kC + row;
      if (tn < s1) {
        const void *src = mat == 0   ? (const void *)(xq + (size_t)tn * qk_stride + hq * kD)
                          : mat == 1 ? (const void *)(xk + (size_t)tn * qk_stride + hq * kD)
                          : mat == 2 ? (const void *)(xv + (size_t)tn * v_stride + h * kD)
                                     : (const void *)(xz + (size_t)tn * v_stride + h * kD);
        prefetch_l2(src, 256);
      }
    }

    // ---------------- gates and their running sum inside the chunk
    {
      float gsum = 0.0f;
      if (tid < 64) {
        const int r = tid;
        float g = 0.0f, be = 0.0f;
        if (r < Lc) {
          const size_t gi = (size_t)(t0 + r) * h_v + h;
          g = gate_g(__bfloat162float(xa[gi]), A_exp, dtb);
          be = sigmoid_f(__bfloat162float(xb[gi]));
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

    // ---------------- prologue: conv(4) + SiLU (+ L2 norm) of q, k, v
    // thread -> channels (2cp, 2cp+1), rows [16 rb, 16 rb + 16)
    {
      const int cp = tid & 63, rb = tid >> 6;
      for (int mat = 0; mat < 3; ++mat) {
        const __nv_bfloat16 *src;
        size_t stride;
        int ch;
        if (mat == 0) {
          src = xq + hq * kD + 2 * cp; stride = qk_stride; ch = hq * kD + 2 * cp;
        } else if (mat == 1) {
          src = xk + hq * kD + 2 * cp; stride = qk_stride; ch = h_qk * kD + hq * kD + 2 * cp;
        } else {
          src = xv + h * kD + 2 * cp; stride = v_stride; ch = 2 * h_qk * kD + h * kD + 2 * cp;
        }
        const float4 w0 = *reinterpret_cast<const float4 *>(p.conv_w + (size_t)ch * 4);
        const float4 w1 = *reinterpret_cast<const float4 *>(p.conv_w + (size_t)(ch + 1) * 4);
        float x0[19], x1[19];
#pragma unroll
        for (int rr = 0; rr < 19; ++rr) {
          const int row = 16 * rb - 3 + rr;
          const int t = t0 + row;
          if (t >= s0 && row < Lc) {
            const float2 f = ld_bf16x2(src + (size_t)t * stride);
            x0[rr] = f.x;
            x1[rr] = f.y;
          } else {
            x0[rr] = 0.0f;
            x1[rr] = 0.0f;
          }
        }
        float y0[16], y1[16], ss[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          const bool ok = 16 * rb + r < Lc;
          float a0 = w0.x * x0[r];
          a0 = fmaf(w0.y, x0[r + 1], a0);
          a0 = fmaf(w0.z, x0[r + 2], a0);
          a0 = fmaf(w0.w, x0[r + 3], a0);
          float a1 = w1.x * x1[r];
          a1 = fmaf(w1.y, x1[r + 1], a1);
          a1 = fmaf(w1.z, x1[r + 2], a1);
          a1 = fmaf(w1.w, x1[r + 3], a1);
          y0[r] = ok ? silu_f(a0) : 0.0f;
          y1[r] = ok ? silu_f(a1) : 0.0f;
          ss[r] = y0[r] * y0[r] + y1[r] * y1[r];
        }
        if (mat < 2) {  // L2 norm over the 128 channels of each row: 64 threads, 2 warps
          const float part = reduce_scatter16(ss, lane);
          if ((lane & 1) == 0) red[warp * 16 + (lane >> 1)] = part;
          __syncthreads();
          if (tid < 64) {
            const int rbb = tid >> 4, rr = tid & 15;
            sInv[tid] = rsqrtf(red[(2 * rbb) * 16 + rr] + red[(2 * rbb + 1) * 16 + rr] + kEpsL2);
          }
          __syncthreads();
#pragma unroll
          for (int r = 0; r < 16; ++r) {
            const float inv = sInv[16 * rb + r];
            y0[r] *= inv;
            y1[r] *= inv;
          }
        }
        if (mat < 2) {  // [K; Q] rows (K: 0..63, Q: 64..127), high and low fp16 parts
          const int row0 = mat == 0 ? 64 : 0;
#pragma unroll
          for (int r = 0; r < 16; ++r) {
            const __half2 hi = __floats2half2_rn(y0[r], y1[r]);
            const __half2 lo = __floats2half2_rn(y0[r] - __low2float(hi), y1[r] - __high2float(hi));
            const uint32_t off = tc::sw128_offset(128, row0 + 16 * rb + r, 2 * cp);
            *reinterpret_cast<__half2 *>(sm + OFF_KQ + off) = hi;
            *reinterpret_cast<__half2 *>(sm + OFF_KQL + off) = lo;
          }
        }
        if (mat == 1) {  // K^T and K~^T
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            tc::st_chunk_f16(sm + OFF_KT + tc::sw128_chunk(128, 2 * cp, 2 * rb + hh), y0 + 8 * hh);
            tc::st_chunk_f16(sm + OFF_KT + tc::sw128_chunk(128, 2 * cp + 1, 2 * rb + hh), y1 + 8 * hh);
          }
          float d0[16], d1[16];
#pragma unroll
          for (int r = 0; r < 16; ++r) {
            const float dcy = sDec[16 * rb + r];
            d0[r] = y0[r] * dcy;
            d1[r] = y1[r] * dcy;
          }
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            tc::st_chunk_f16(sm + OFF_KTT + tc::sw128_chunk(128, 2 * cp, 2 * rb + hh), d0 + 8 * hh);
            tc::st_chunk_f16(sm + OFF_KTT + tc::sw128_chunk(128, 2 * cp + 1, 2 * rb + hh), d1 + 8 * hh);
          }
        }
        if (mat == 2) {  // V^T
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            tc::st_chunk_f16(sm + OFF_VT + tc::sw128_chunk(128, 2 * cp, 2 * rb + hh), y0 + 8 * hh);
            tc::st_chunk_f16(sm + OFF_VT + tc::sw128_chunk(128, 2 * cp + 1, 2 * rb + hh), y1 + 8 * hh);
          }
        }
      }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // ---------------- P1 = [K; Q] K^T (hi.hi + hi.lo + lo.hi) and D2a = S Q^T (one commit)
    if (tid == 0) {
      mma_chain(tmem + COL_P1, sbase + OFF_KQ, 128, 0, sbase + OFF_KQ, 128, 0, 8, kIdN64, false);
      mma_chain(tmem + COL_P1, sbase + OFF_KQ, 128, 0, sbase + OFF_KQL, 128, 0, 8, kIdN64, true);
      mma_chain(tmem + COL_P1, sbase + OFF_KQL, 128, 0, sbase + OFF_KQ, 128, 0, 8, kIdN64, true);
      mma_chain(tmem + COL_D2A, sbase + OFF_SB, 128, 0, sbase + OFF_KQ, 128, 64, 8, kIdN64, false);
      tc::mma_commit(bar);
    }
    // meanwhile: S <- gamma_C S in tensor memory (the MMAs above read the fp16 copy)
    {
      const float gC = sGam[63];
      for (int c0 = 0; c0 < 64; c0 += 32) {
        float v[32];
        tc::tmem_ld32(tmem + lane_off + COL_S + 64 * gh + c0, v);
#pragma unroll
        for (int q = 0; q < 32; ++q) v[q] *= gC;
        tc::tmem_st32(tmem + lane_off + COL_S + 64 * gh + c0, v);
      }
    }
    {
      const bool ok = tc::mbar_wait(bar, phase & 1);
      ++phase;
      tc::fence_after_sync();
      if (__syncthreads_or(!ok)) { failed = true; break; }
    }

    // ---------------- A (fp32, strictly lower) and A_Q (fp16, lower with diagonal)
    {
      float v[32];
      tc::tmem_ld32(tmem + lane_off + COL_P1 + 32 * gh, v);
      if (lr < 64) {
        const int r = lr;
        const float Gr = sG[r], br = sBeta[r];
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          const int s = 32 * gh + q;
          AF[r * kPad + s] = (s < r) ? br * expf(Gr - sG[s]) * v[q] : 0.0f;
        }
      } else {
        const int r = lr - 64;
        const float Gr = sG[r];
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          const int s = 32 * gh + q;
          v[q] = (s <= r) ? expf(Gr - sG[s]) * v[q] : 0.0f;
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tc::st_chunk_f16(sm + OFF_AQ + tc::sw128_chunk(64, r, 4 * gh + cc), v + 8 * cc);
      }
    }
    tc::fence_before_sync();
    __syncthreads();

    // ---------------- T = (I + A)^-1: diagonal 16x16 blocks by forward substitution
    if (tid < 64) {
      const int bb = tid >> 4, s = tid & 15;
      float x[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        float acc = (r == s) ? 1.0f : 0.0f;
        const float *arow = AF + (16 * bb + r) * kPad + 16 * bb;
#pragma unroll
        for (int m = 0; m < r; ++m) acc = fmaf(-arow[m], x[m], acc);
        x[r] = acc;
      }
#pragma unroll
      for (int r = 0; r < 16; ++r) TF[(16 * bb + r) * kPad + 16 * bb + s] = x[r];
    }
    __syncthreads();
    // off-diagonal blocks, one block row at a time: T_ij = -T_ii sum_{m=j}^{i-1} A_im T_mj
    for (int i = 1; i < 4; ++i) {
      for (int e = tid; e < 256 * i; e += kThreads) {
        const int j = e >> 8, r = (e >> 4) & 15, s = e & 15;
        float acc = 0.0f;
        for (int m = j; m < i; ++m) {
          const float *arow = AF + (16 * i + r) * kPad + 16 * m;
          const float *tcol = TF + (16 * m) * kPad + 16 * j + s;
#pragma unroll
          for (int kk = 0; kk < 16; ++kk) acc = fmaf(arow[kk], tcol[kk * kPad], acc);
        }
        XF[j * 256 + r * 16 + s] = acc;
      }
      __syncthreads();
      for (int e = tid; e < 256 * i; e += kThreads) {
        const int j = e >> 8, r = (e >> 4) & 15, s = e & 15;
        const float *trow = TF + (16 * i + r) * kPad + 16 * i;
        float acc = 0.0f;
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) acc = fmaf(trow[kk], XF[j * 256 + kk * 16 + s], acc);
        TF[(16 * i + r) * kPad + 16 * j + s] = -acc;
      }
      __syncthreads();
    }
    // T diag(beta gamma) and T diag(beta) as fp16 operands (rows r, columns m)
    {
      const int r = tid >> 2, qq = tid & 3;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float a8[8], b8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int m = 16 * qq + 8 * hh + e;
          const float t = (m <= r) ? TF[r * kPad + m] : 0.0f;
          b8[e] = t * sBeta[m];
          a8[e] = b8[e] * sGam[m];
        }
        tc::st_chunk_f16(sm + OFF_TBG + tc::sw128_chunk(64, r, 2 * qq + hh), a8);
        tc::st_chunk_f16(sm + OFF_TB + tc::sw128_chunk(64, r, 2 * qq + hh), b8);
      }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // ---------------- P2: W^T = K^T (T diag(beta gamma))^T, U'^T = V^T (T diag(beta))^T
    if (tid == 0) {
      mma_chain(tmem + COL_P1, sbase + OFF_KT, 128, 0, sbase + OFF_TBG, 64, 0, 4, kIdN64, false);
      mma_chain(tmem + COL_UP, sbase + OFF_VT, 128, 0, sbase + OFF_TB, 64, 0, 4, kIdN64, false);
      tc::mma_commit(bar);
    }
    {
      const bool ok = tc::mbar_wait(bar, phase & 1);
      ++phase;
      tc::fence_after_sync();
      if (__syncthreads_or(!ok)) { failed = true; break; }
    }
    // W (rows r, columns i) from W^T in tensor memory (lane i)
    {
      const int i = lr;
      float v[32];
      tc::tmem_ld32(tmem + lane_off + COL_P1 + 32 * gh, v);
#pragma unroll
      for (int q = 0; q < 32; ++q)
        *reinterpret_cast<__half *>(sm + OFF_WS + tc::sw128_offset(64, 32 * gh + q, i)) = __float2half_rn(v[q]);
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // ---------------- D1 = S W^T
    if (tid == 0) {
      mma_chain(tmem + COL_D1, sbase + OFF_SB, 128, 0, sbase + OFF_WS, 64, 0, 8, kIdN64, false);
      tc::mma_commit(bar);
    }
    {
      const bool ok = tc::mbar_wait(bar, phase & 1);
      ++phase;
      tc::fence_after_sync();
      if (__syncthreads_or(!ok)) { failed = true; break; }
    }
    // U^T = U'^T - D1 (lane j), fp16 operand rows j, columns r
    {
      const int j = lr;
      float d1[32], up[32];
      tc::tmem_ld32(tmem + lane_off + COL_D1 + 32 * gh, d1);
      tc::tmem_ld32(tmem + lane_off + COL_UP + 32 * gh, up);
#pragma unroll
      for (int q = 0; q < 32; ++q) up[q] -= d1[q];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tc::st_chunk_f16(sm + OFF_US + tc::sw128_chunk(128, j, 4 * gh + cc), up + 8 * cc);
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // ---------------- D2b = U^T A_Q^T;  S += U^T K~
    if (tid == 0) {
      mma_chain(tmem + COL_D2B, sbase + OFF_US, 128, 0, sbase + OFF_AQ, 64, 0, 4, kIdN64, false);
      mma_chain(tmem + COL_S, sbase + OFF_US, 128, 0, sbase + OFF_KTT, 128, 0, 4, kIdN128, true);
      tc::mma_commit(bar);
    }
    {
      const bool ok = tc::mbar_wait(bar, phase & 1);
      ++phase;
      tc::fence_after_sync();
      if (__syncthreads_or(!ok)) { failed = true; break; }
    }

    // ---------------- output: o = scale (gamma_r D2a + D2b), RMSNormGated, store
    {
      const int j = lr;
      float o[32], d2b[32];
      tc::tmem_ld32(tmem + lane_off + COL_D2A + 32 * gh, o);
      tc::tmem_ld32(tmem + lane_off + COL_D2B + 32 * gh, d2b);
      float sq[32];
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        o[q] = scale * fmaf(sGam[32 * gh + q], o[q], d2b[q]);
        sq[q] = o[q] * o[q];
      }
      const float part = reduce_scatter32(sq, lane);
      red[warp * 32 + lane] = part;  // warp w of half gh covers j in [32 (w&3), +32)
      __syncthreads();
      const float wj = p.norm_w[j];
#pragma unroll 4
      for (int q = 0; q < 32; ++q) {
        const int r = 32 * gh + q;
        if (r < Lc) {
          const float ssum = red[(4 * gh) * 32 + q] + red[(4 * gh + 1) * 32 + q] + red[(4 * gh + 2) * 32 + q] +
                             red[(4 * gh + 3) * 32 + q];
          const float inv = rsqrtf(ssum * (1.0f / kD) + kEpsRms);
          const size_t oi = ((size_t)(t0 + r) * h_v + h) * kD + j;
          const float zz = __bfloat162float(xz[oi]);
          out[oi] = __float2bfloat16_rn(o[q] * inv * wj * silu_f(zz));
        }
      }
    }
    // next chunk's fp16 copy of S
    {
      const int j = lr;
      for (int c0 = 0; c0 < 64; c0 += 32) {
        float v[32];
        tc::tmem_ld32(tmem + lane_off + COL_S + 64 * gh + c0, v);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
          tc::st_chunk_f16(sm + OFF_SB + tc::sw128_chunk(128, j, 8 * gh + (c0 >> 3) + cc), v + 8 * cc);
      }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
  }

  if (failed) {
    if (tid == 0) set_status(p.status, kDevTimeout);
  } else if (p.final_state) {
    const int j = lr;
    for (int c0 = 0; c0 < 64; c0 += 32) {
      float v[32];
      tc::tmem_ld32(tmem + lane_off + COL_S + 64 * gh + c0, v);
#pragma unroll
      for (int q = 0; q < 32; ++q) p.final_state[st_off + (size_t)(64 * gh + c0 + q) * kD + j] = v[q];
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

size_t prefill_tc_workspace_bytes(int, int) { return 0; }

cudaError_t launch_prefill_tc(const PrefillParams &p, cudaStream_t s) {
  const unsigned grid = (unsigned)p.N * (unsigned)p.h_v;
  if (grid == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  prefill_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
