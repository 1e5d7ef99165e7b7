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

/* Test hook for the bounded waits of the one-launch linear-attention kernel
 * (linattn_chunked_forward on the shapes it handles: bf16, d_v = 128,
 * d_k in {64, 128}).  From the next call on, the partial-state items of
 * batch-head index `bh` (b * H + h) never report that they are done, so the
 * items that wait for them (that batch-head's prefix and output items) run
 * into their wait limit, record TTT_ERR_TIMEOUT in the device status word
 * and give up without storing anything; the other batch-heads are computed
 * as usual.  The waits that run out are taken before the waiting item issues
 * any copy, so nothing is in flight when it gives up.  bh < 0 turns the hook
 * off.  Process-wide; not for production use. */
void ttt_selftest_withhold_release(int bh);

#ifdef __cplusplus
}
#endif

#endif /* TTT_GB300_TTT_SELFTEST_H */
