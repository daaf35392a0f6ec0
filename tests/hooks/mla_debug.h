/*
 * mla_debug.h -- test hooks (not part of the MLA operation, not in libmla.so).
 *
 * They live in a test-only library, tests/hooks/libmla_debug.so, linked from
 * the same compiled kernels as libmla.so plus mla_debug_hooks.cu, so that the
 * product library ships no test entry points.  They let the test-suite
 * exercise single kernels of the library in isolation: the tcgen05 GEMM used by every projection, the
 * bounded device-side wait that turns a missing arrival into an error status
 * instead of a hang, and a layout check of the tensor-memory accumulator.
 * Same conventions as mla.h: device pointers, asynchronous on `stream`,
 * status codes from mla.h.
 */
#ifndef MLA_DEBUG_H_
#define MLA_DEBUG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* C[M, N] (bf16, row stride ldc) = A[M, K] . B^T with A bf16 [M, K] (row
 * stride lda) and B either bf16 [N, K] (b_mn_major = 0, row stride ldb) or
 * bf16 [K, N] (b_mn_major = 1, row stride ldb).  K % 64 == 0; N % 128 == 0
 * (or % 192).  Float32 accumulation in tensor memory. */
int mla_debug_gemm(const void* A, int lda, const void* B, int ldb, int b_mn_major, void* C, int ldc, int M, int N,
                   int K, void* stream);

/* Launches one CTA that waits on an mbarrier nobody arrives at, with a wait
 * limit of limit_ns nanoseconds.  The wait gives up, ORs the timeout bit into
 * *status_word (device uint32) and the kernel returns. */
int mla_debug_wait_timeout(void* status_word, uint64_t limit_ns, void* stream);

/* One kind::f16 MMA with M = m (64 or 128), N = 64, K = 16 from operands
 * A[r][0] = r + 1, A[r][1] = 128, B[n][0] = 1, B[n][1] = n (others 0), so that
 * D[r][n] = r + 1 + 128 n; writes all 128 TMEM lanes x 64 columns of the
 * accumulator to out (float32 [128, 64], lane-major).  Shows where each
 * accumulator row lives in tensor memory. */
int mla_debug_umma_probe(float* out, int m, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DEBUG_H_ */
