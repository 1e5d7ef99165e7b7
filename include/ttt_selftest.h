/*
 * ttt_selftest.h - self-test entry point of the library's GEMM building block.
 *
 * The pages have no counterpart for this call: it exists so that the tests can
 * check the tensor-core tile machinery (TMA boxes, shared-memory descriptors
 * for K-major and M/N-major operands, TMEM accumulators) in isolation, against
 * a plain matrix product, before the layer kernels built on it are compared
 * with the oracle.  It follows the conventions of ttt.h (device pointers,
 * asynchronous on `stream`, status codes of ttt_status).
 */
#ifndef TTT_GB300_TTT_SELFTEST_H
#define TTT_GB300_TTT_SELFTEST_H

#include "ttt.h"

#ifdef __cplusplus
extern "C" {
#endif

/* D[z] = A[z] * B[z] for z in 0..Z-1, fp32 output [Z, M, N].
 *   A: a_mn_major = 0 -> [Z, M, K] (K contiguous); 1 -> [Z, K, M].
 *   B: b_mn_major = 0 -> [Z, N, K] (K contiguous); 1 -> [Z, K, N].
 *   dtype TTT_BF16 runs the tensor-core kernel (M, N, K multiples of 64,
 *   tile_n in {64, 128, 192, 256}); TTT_F32 runs the fp32 SIMT kernel (any
 *   sizes; tile_n ignored). */
int ttt_selftest_gemm(const void* A, const void* B, float* D, int Z, int M, int N, int K,
                      int a_mn_major, int b_mn_major, int dtype, int tile_n,
                      ttt_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TTT_GB300_TTT_SELFTEST_H */
