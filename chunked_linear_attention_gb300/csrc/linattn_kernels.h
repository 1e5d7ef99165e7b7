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

// Momentum and per-chunk learning rate of the state update ("Test-Time
// Training with KV Binding Is Secretly Linear Attention", Thm 5.3, App. H):
// per updating chunk c, M <- alpha_c M + G_c and S <- S + lr_c M (or, with
// mom = 0, S <- S + lr_c G_c).  alpha / lr are [BH][nc] (NULL: alpha = 0,
// lr = 1, or the constants below); M0 / M_final are [BH][dv*dk] fp32 (NULL:
// zeros / not written).
struct LinRule {
  const float* alpha = nullptr;
  const float* lr = nullptr;
  const float* M0 = nullptr;
  float* M_final = nullptr;
  int mom = 0;
  float alpha_const = 0.f;   // alpha of every chunk when alpha is NULL
  float lr_const = 1.f;      // learning rate of every chunk when lr is NULL
  float inc_scale = 1.f;     // factor of every increment (the sign of a negated Muon output)
};

// vt = eta (per row) * v, in bf16 or fp32.
cudaError_t launch_scale_rows(const void* v, const float* eta, void* vt, long long rows, int cols,
                              bool bf16, cudaStream_t stream);

// Sums per-split partial states into the state each chunk reads
// (s_read [BH][nc][dv*dk], bf16 or fp32) and the final state (fp32), through
// the rule's momentum and learning rates.  `compact`: the partials hold one
// increment per UPDATING chunk ([BH][n_upd][dv*dk], splits = 1) instead of
// one per chunk and split.
cudaError_t launch_linattn_prefix(const float* partials, const float* S0, void* s_read,
                                  float* s_final, int BH, int nc, int splits, int dvdk,
                                  int apply_first, const UpdateFlags& flags, const LinRule& rule,
                                  int compact, int n_upd, bool bf16, cudaStream_t stream);

// The momentum of every update, for Muon: per (batch-head, updating chunk u)
// M_u = alpha_c M_{u-1} + sum of the chunk's split partials, written to
// x [BH][n_upd][dv*dk] (bf16 or fp32) with its squared Frobenius norm as
// per-block partial sums norm_part [BH][n_upd][nslot] (nslot = blocks per
// batch-head, 256 elements each; summed in a fixed order later), and the last
// M to rule.M_final.
cudaError_t launch_linattn_momentum(const float* partials, int splits, const LinRule& rule,
                                    void* x, float* norm_part, int BH, int nc, int n_upd,
                                    int dvdk, const UpdateFlags& flags, bool bf16,
                                    cudaStream_t stream);
int linattn_momentum_slots(int dvdk);

// out[z] = sum of part[z][0 .. nslot) (fixed order), z < Z.
cudaError_t launch_normsq_sum(const float* part, int nslot, float* out, int Z,
                              cudaStream_t stream);

}  // namespace ttt
