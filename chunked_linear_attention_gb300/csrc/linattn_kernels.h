// Launchers of the chunked linear-attention helper kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ttt {

constexpr int kMaxFlagChunks = 2048;

// Per-chunk update flags passed by value (strided mask); all = 1 means every
// chunk updates.
struct UpdateFlags {
  int all;
  uint32_t bits[kMaxFlagChunks / 32];
};

// vt = eta (per row) * v, in bf16 or fp32.
cudaError_t launch_scale_rows(const void* v, const float* eta, void* vt, long long rows, int cols,
                              bool bf16, cudaStream_t stream);

// Sums per-split partial states into the state each chunk reads
// (s_read [BH][nc][dv*dk], bf16 or fp32) and the final state (fp32).
cudaError_t launch_linattn_prefix(const float* partials, const float* S0, void* s_read,
                                  float* s_final, int BH, int nc, int splits, int dvdk,
                                  int apply_first, const UpdateFlags& flags, bool bf16,
                                  cudaStream_t stream);

}  // namespace ttt
