// Internal interface between the C ABI (capi.cu) and the host orchestration
// of the TTT layer (layer.cu) and chunked linear attention (linattn.cu).
// Arguments reaching these functions have been validated.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

namespace ttt {

struct LayerDims {
  int B, H, N, d, m, chunk;
  bool bf16;
  int mode;
  int l2norm;
  int muon_steps;
  float beta;
  float ns[3];
  int last_only = 0;     // only W2 updates (W1, W3 static: a static feature map)
  int inner_steps = 1;   // update steps per updating chunk
  int parallel = 0;      // the parallel form (last_only, no normalisation, one inner step)
};

// Page-locked host tensors of a host-buffer call: the layer copies each
// chunk's q, k, v, eta into the device tensors of LayerArgs on a copy stream
// just ahead of the launches that read it, copies each chunk's output back as
// soon as it is written, and the weights in before and out after the scan.
struct HostIO {
  const void* q;
  const void* k;       // may equal q (then LayerArgs::k equals LayerArgs::q)
  const void* v;
  const float* eta;
  const float* W[3];   // W1, W2, W3
  void* out;
  float* Wf[3];        // W1_final, W2_final, W3_final
  float* momentum;     // or NULL
};

struct LayerArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* eta;
  const float* W[3];   // W1, W2, W3
  int w_per_batch;
  const unsigned char* update_chunks;  // host
  void* out;
  float* Wf[3];        // W1_final, W2_final, W3_final
  float* momentum;     // [3][B*H][d*m] (M1, M2, M3) or NULL
  void* workspace;
  cudaStream_t stream;
  const HostIO* host = nullptr;   // set: the device tensors above are staging copies
};

size_t layer_workspace_bytes(const LayerDims& D);
// Returns a ttt_status code.
int layer_forward(const LayerArgs& a, const LayerDims& D, int* status, unsigned long long wait_ns);

struct LinDims {
  int B, H, N, dk, dv, chunk;
  bool bf16;
  int mode;
  int mom = 0;              // a momentum accumulator is carried (alpha, M0 or M_final given)
  int muon_steps = 0;       // Newton-Schulz steps of Muon(M) per update (0: none)
  float ns[3] = {0.f, 0.f, 0.f};
};

struct LinArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* eta;
  const float* S0;
  const unsigned char* update_chunks;  // host
  void* out;
  float* S_final;
  void* workspace;
  cudaStream_t stream;
  const float* alpha = nullptr;   // [B*H][nc] momentum factor per chunk, or NULL (0)
  const float* lr = nullptr;      // [B*H][nc] learning rate per chunk, or NULL (1)
  const float* M0 = nullptr;      // [B*H][dv*dk] initial momentum, or NULL (zeros)
  float* M_final = nullptr;       // [B*H][dv*dk] final momentum, or NULL
  float alpha_const = 0.f;        // alpha of every chunk when alpha is NULL
  float lr_const = 1.f;           // learning rate of every chunk when lr is NULL
};

size_t linattn_workspace_bytes(const LinDims& D);
int linattn_forward(const LinArgs& a, const LinDims& D, int* status, unsigned long long wait_ns);

// Self-test GEMM (capi.cu) uses the builder directly.
int selftest_gemm(const void* A, const void* Bp, float* Dp, int Z, int M, int N, int K, int a_mn,
                  int b_mn, bool bf16, int tile_n, cudaStream_t stream, int* status,
                  unsigned long long wait_ns);

}  // namespace ttt
