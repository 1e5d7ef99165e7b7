// Muon as separate GEMM launches per Newton-Schulz product ("5.2.1 LaCT and
// TTT-E2E", eq (6); the quintic of the Muon write-up): for any batch of
// equally shaped matrices, bf16 on the tensor cores or fp32 on the SIMT
// kernel.  Used where no fused cluster kernel applies (non-square fast
// weights) and for the many small matrices of the parallel linear-attention
// form (one per update of every sequence).
#pragma once

#include <cuda_runtime.h>

#include "builder.h"

namespace ttt {

// One group of Z matrices of R x C elements (dense, row-major, Z-major).
struct NsGroup {
  void* X[2];           // iterates [Z][R*C] (bf16 or fp32); X[0] holds M on entry
  void* G;              // Gram products [Z][s*s], s = min(R, C)
  void* Bm;             // polynomial products [Z][s*s]
  float* U;             // fp32 result Muon(M) [Z][R*C]
  const float* normsq;  // squared Frobenius norm of each M [Z]
  int Z, R, C;
};

// Enqueues `steps` Newton-Schulz steps for every matrix of the groups (at most
// two; their products share each launch): per step G = X X^T (scaled by
// 1/(|M|_F + eps)^2 on the first step; X^T X for tall matrices),
// Bm = b G + c G G, X' = a X + Bm X (X' = X (a I + Bm) for tall ones; scaled
// by 1/(|M|_F + eps) on the first step), the last step writing U in fp32.
// Returns 0, or a negative ttt_status code.
int enqueue_ns_products(LaunchBuilder& LB, const NsGroup* groups, int ngroups, int steps,
                        const float ns[3], cudaStream_t st);

}  // namespace ttt
