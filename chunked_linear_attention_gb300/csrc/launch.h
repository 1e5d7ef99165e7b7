// Host-side launchers of the library's kernels (one definition per .cu file).
#pragma once

#include <cuda_runtime.h>

#include "gemm_desc.h"

namespace ttt {

// Dynamic shared memory of the tensor-core GEMM: the whole 227 KB, so one CTA
// owns an SM and its TMEM (no allocation contention).
constexpr int kUmmaSmemBytes = 227 * 1024;
constexpr int kSimtTile = 64;

// SMs of the current device (0 if unknown).
int device_sm_count();

// Grid of a tensor-core GEMM launch (the persistent kernel: at most one CTA
// per SM, capped at `max_ctas` when > 0).
int umma_gemm_grid(const GemmLaunch& L, int max_ctas);

// `priority`: launch priority (0: the stream's own; lower values run first).
// `max_ctas` > 0 caps the persistent grid below one CTA per SM.
cudaError_t launch_umma_gemm(const GemmLaunch& L, cudaStream_t stream, int priority = 0,
                             int max_ctas = 0);
// One-time per-device kernel attributes (call before any stream capture).
cudaError_t prepare_umma_gemm();
cudaError_t launch_simt_gemm(const GemmLaunch& L, cudaStream_t stream);

// ---- elementwise / reduction kernels (aux_kernels.cu)

// One fast-weight matrix family (W1, W2 or W3) for the update steps.
struct MatSet {
  const float* init;      // initial weights [H or B*H][rows*cols]
  int init_per_batch;     // 1: init indexed by b*H+h, 0: by h
  float* master;          // fp32 state [B*H][rows*cols] (the caller's W_final)
  void* work;             // operand copy [B*H][rows*cols] (bf16) or NULL
  const float* update;    // U [B*H][rows*cols] subtracted by normalize
  int rows, cols;
};

// For up to three sets in one launch: master = init (broadcast over the batch
// unless per batch), work = bf16(master); also clears n0 floats at zero0 and
// n1 at zero1 (either may be NULL).
cudaError_t launch_init_layer(const MatSet* sets, int nsets, int B, int H, float* zero0,
                              long long n0, float* zero1, long long n1, cudaStream_t stream);

// master = RowNorm(master - update) (or master - update), work = bf16(master).
cudaError_t launch_update_normalize(const MatSet* sets, int nsets, int BH, int l2norm,
                                    cudaStream_t stream);

// out[s * BH + h] = sum of the nslot partial sums at part + (s * BH + h) * nslot,
// in a fixed order, for s = 0..2 and h in [h0, h0 + nh).
cudaError_t launch_normsq_reduce(const float* part, int nslot, float* out, int BH, int h0,
                                 int nh, cudaStream_t stream);

// dst[i] = src[i] (float), for i < n; src NULL -> zeros.
cudaError_t launch_copy_f32(float* dst, const float* src, long long n, cudaStream_t stream);

}  // namespace ttt
