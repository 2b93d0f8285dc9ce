/*
 * gdn_selftest.h -- self-test entry point of libgdn.so for the tensor-core
 * building blocks the prefill kernel uses (tcgen05.mma with bf16 operands in
 * the 128-byte-swizzled K-major shared-memory layout, fp32 accumulators in
 * tensor memory, commit to an mbarrier, tcgen05.ld / tcgen05.st).  It is test
 * infrastructure: the layer never calls it.
 */
#ifndef GDN_SELFTEST_H_
#define GDN_SELFTEST_H_

#include <stdint.h>

#include "gdn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * One CTA computes D = A * B[b_row0 : b_row0 + N]^T with the prefill's MMA path.
 * A     [128, K] row-major (device), bf16 or (fp16 != 0) fp16
 * B     [b_row0 + N, K] row-major (device), same type; the MMA reads rows from b_row0
 * D     fp32 [2, 128, N] (device): D[0] = the product read back from tensor
 *       memory; D[1] = the same after a tensor-memory round trip that doubles
 *       it (tcgen05.ld, x2, tcgen05.st, tcgen05.ld)
 * flag  int32 (device): set to GDN_ERR_TIMEOUT if the MMA completion wait ran out
 * Supported: N in {32, 64, 128, 256}, K in {64, 128}, b_row0 in {0, 64}, b_row0 + N <= 256.
 * Returns GDN_OK, GDN_ERR_INVALID_ARG or GDN_ERR_CUDA.
 */
GDN_API int gdn_selftest_umma(const void *A, const void *B, float *D, int *flag, int N, int K, int b_row0,
                              int fp16, void *stream);

/*
 * The same product with the A operand read from tensor memory instead of shared
 * memory (tcgen05.mma with A in TMEM: row m in lane m, 16-bit elements packed
 * two per 32-bit column), as the transposed state pass uses it.
 * A [128, K], B [N, K] row-major (device), bf16 or (fp16 != 0) fp16;
 * D fp32 [128, N].  Supported: N in {64, 128, 256}, K in {32, 64, 128}.
 */
GDN_API int gdn_selftest_umma_ts(const void *A, const void *B, float *D, int *flag, int N, int K, int fp16,
                                 void *stream);

/*
 * Failure detection without a fault: one CTA waits, with the bounded wait every
 * kernel of the library uses, on an mbarrier that nothing ever signals.  After
 * limit_us microseconds (1 .. 1,000,000) of %globaltimer the wait gives up, the
 * kernel writes GDN_ERR_TIMEOUT to *flag (device int32) and returns: no trap,
 * no hang, and the CUDA context stays usable.  Returns GDN_OK, GDN_ERR_INVALID_ARG
 * or GDN_ERR_CUDA (launch).
 */
GDN_API int gdn_selftest_wait_timeout(int *flag, int limit_us, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_SELFTEST_H_ */
