// Self-test of the tensor-core path (see include/gdn_selftest.h): one CTA of
// 128 threads stages A and B into the SW128 K-major layout, one thread issues
// the MMAs, and every thread reads its accumulator lane back.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdn_selftest.h"
#include "gdn_common.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

__global__ void __launch_bounds__(128) umma_selftest_kernel(const uint16_t *__restrict__ A,
                                                            const uint16_t *__restrict__ B,
                                                            float *__restrict__ D, int *flag, int N, int K,
                                                            int b_row0, int fp16) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base_s;
  uint8_t *smem = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  const int BR = b_row0 + N;
  uint8_t *sA = smem;                    // 128 rows x K
  uint8_t *sB = smem + 128 * K * 2;      // BR rows x K (1024-aligned: 128*K*2 is)
  const int tid = threadIdx.x, warp = tid >> 5;

  // stage A (row tid) and B (rows < BR), 16 bytes at a time
  for (int c = 0; c < K / 8; ++c) {
    *reinterpret_cast<uint4 *>(sA + tc::sw128_chunk(128, tid, c)) =
        *reinterpret_cast<const uint4 *>(A + (size_t)tid * K + 8 * c);
    for (int row = tid; row < BR; row += 128)
      *reinterpret_cast<uint4 *>(sB + tc::sw128_chunk(BR, row, c)) =
          *reinterpret_cast<const uint4 *>(B + (size_t)row * K + 8 * c);
  }
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base_s, 256);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base_s;

  if (tid == 0) {
    const uint32_t a0 = tc::smem_u32(sA), b0 = tc::smem_u32(sB);
    const uint32_t id = fp16 ? tc::idesc_f16(128, N) : tc::idesc_bf16(128, N);
    for (int k16 = 0; k16 < K / 16; ++k16)
      tc::mma16(tmem, tc::sdesc_kstep(a0, 128, 0, k16), tc::sdesc_kstep(b0, BR, b_row0, k16), id,
                   k16 > 0 ? 1u : 0u);
    tc::mma_commit(&bar);
  }
  const bool ok = tc::mbar_wait(&bar, 0);
  if (!ok && tid == 0) atomicExch(flag, kDevTimeout);
  tc::fence_after_sync();
  if (__syncthreads_and(ok)) {
    const uint32_t lane_base = tc::tmem_addr(tmem, warp * 32, 0);
    for (int c = 0; c < N; c += 32) {
      float v[32];
      tc::tmem_ld32(lane_base + c, v);
      for (int i = 0; i < 32; ++i) {
        D[(size_t)tid * N + c + i] = v[i];
        v[i] *= 2.0f;
      }
      tc::tmem_st32(lane_base + c, v);
    }
    for (int c = 0; c < N; c += 32) {
      float v[32];
      tc::tmem_ld32(lane_base + c, v);
      for (int i = 0; i < 32; ++i) D[(size_t)128 * N + (size_t)tid * N + c + i] = v[i];
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

// The same product with A read from tensor memory: every thread packs its row
// of A (row tid) into 16-bit pairs and stores them to the columns at A_COL by
// tcgen05.st; B is staged in shared memory as above.
__global__ void __launch_bounds__(128) umma_ts_selftest_kernel(const uint16_t *__restrict__ A,
                                                               const uint16_t *__restrict__ B,
                                                               float *__restrict__ D, int *flag, int N, int K,
                                                               int fp16) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base_s;
  uint8_t *smem = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t *sB = smem;  // N rows x K
  const int tid = threadIdx.x, warp = tid >> 5;
  constexpr int A_COL = 256;
  for (int c = 0; c < K / 8; ++c)
    for (int row = tid; row < N; row += 128)
      *reinterpret_cast<uint4 *>(sB + tc::sw128_chunk(N, row, c)) =
          *reinterpret_cast<const uint4 *>(B + (size_t)row * K + 8 * c);
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base_s, 512);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base_s;
  const uint32_t lane_base = tc::tmem_addr(tmem, warp * 32, 0);
  for (int c0 = 0; c0 < K / 2; c0 += 16) {  // 16 packed columns (32 elements) at a time
    float v[16];
    for (int i = 0; i < 16; ++i) {
      const uint32_t lo = A[(size_t)tid * K + 2 * (c0 + i)], hi = A[(size_t)tid * K + 2 * (c0 + i) + 1];
      v[i] = __uint_as_float(lo | (hi << 16));
    }
    tc::tmem_st16(lane_base + A_COL + c0, v);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (tid == 0) {
    const uint32_t b0 = tc::smem_u32(sB);
    const uint32_t id = fp16 ? tc::idesc_f16(128, N) : tc::idesc_bf16(128, N);
    for (int k16 = 0; k16 < K / 16; ++k16)
      tc::mma16_ts(tmem, tmem + A_COL + 8 * k16, tc::sdesc_kstep(b0, N, 0, k16), id, k16 > 0 ? 1u : 0u);
    tc::mma_commit(&bar);
  }
  const bool ok = tc::mbar_wait(&bar, 0);
  if (!ok && tid == 0) atomicExch(flag, kDevTimeout);
  tc::fence_after_sync();
  if (__syncthreads_and(ok)) {
    for (int c = 0; c < N; c += 32) {
      float v[32];
      tc::tmem_ld32(lane_base + c, v);
      for (int i = 0; i < 32; ++i) D[(size_t)tid * N + c + i] = v[i];
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

// A wait that runs out: the mbarrier expects one arrival that never comes.
__global__ void __launch_bounds__(32) wait_timeout_kernel(int *flag, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0 && !tc::mbar_wait(&bar, 0, limit_ns)) atomicExch(flag, kDevTimeout);
}

}  // namespace
}  // namespace gdn

extern "C" int gdn_selftest_wait_timeout(int *flag, int limit_us, void *stream) {
  if (!flag || limit_us < 1 || limit_us > 1000000) return GDN_ERR_INVALID_ARG;
  gdn::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(flag, (uint64_t)limit_us * 1000ull);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" int gdn_selftest_umma(const void *A, const void *B, float *D, int *flag, int N, int K, int b_row0,
                                 int fp16, void *stream) {
  if (!A || !B || !D || !flag) return GDN_ERR_INVALID_ARG;
  if ((N != 32 && N != 64 && N != 128 && N != 256) || (K != 64 && K != 128) || (b_row0 != 0 && b_row0 != 64) ||
      b_row0 + N > 256)
    return GDN_ERR_INVALID_ARG;
  const size_t smem = 1024 + (size_t)128 * K * 2 + (size_t)(b_row0 + N) * K * 2;
  auto kern = gdn::umma_selftest_kernel;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return GDN_ERR_CUDA;
  kern<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(static_cast<const uint16_t *>(A),
                                                             static_cast<const uint16_t *>(B), D, flag, N, K,
                                                             b_row0, fp16);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" int gdn_selftest_umma_ts(const void *A, const void *B, float *D, int *flag, int N, int K, int fp16,
                                    void *stream) {
  if (!A || !B || !D || !flag) return GDN_ERR_INVALID_ARG;
  if ((N != 64 && N != 128 && N != 256) || (K != 32 && K != 64 && K != 128)) return GDN_ERR_INVALID_ARG;
  const size_t smem = 1024 + (size_t)N * (K < 64 ? 64 : K) * 2;
  auto kern = gdn::umma_ts_selftest_kernel;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return GDN_ERR_CUDA;
  kern<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(static_cast<const uint16_t *>(A),
                                                             static_cast<const uint16_t *>(B), D, flag, N, K, fp16);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
