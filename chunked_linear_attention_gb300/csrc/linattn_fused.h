// Host entry of the one-launch chunked linear attention (linattn_fused.cu).
#pragma once

#include <cuda_runtime.h>

#include "builder.h"
#include "layer.h"
#include "linattn_kernels.h"

namespace ttt {

// Work split of one call: token splits of each chunk's state sum, state
// elements per prefix item (dv * dk / pparts), output rows per item.
struct LinFusedPlan {
  int splits, pparts, rb;
};

struct LinFusedArgs {
  const LinDims* D;
  const void* q;
  const void* k;
  const void* v;
  const float* eta;
  const float* S0;              // or NULL
  const UpdateFlags* flags;
  LinRule rule;                 // momentum / per-chunk learning rates (no Muon here)
  void* out;
  float* S_final;               // or NULL
  void* scratch;                // linattn_fused_scratch() bytes, 256-byte aligned
};

// Test hook: from the next launch on, batch-head `bh`'s state items never
// report completion (-1 turns this off), so that the items waiting for them
// run into their bounded waits.
void linattn_fused_withhold_release(int bh);

// True for the shapes the kernel handles: bf16, d_v = 128, d_k = 64 or 128,
// chunk a multiple of 128.
bool linattn_fused_applicable(const LinDims& D);
LinFusedPlan linattn_fused_plan(const LinDims& D);
// Scratch bytes: fp32 partial states, bf16 per-chunk states, counters.
size_t linattn_fused_scratch(const LinDims& D, const LinFusedPlan& p);
// One-time per-device setup (before any stream capture); false if the device
// cannot run the cooperative kernel.
bool prepare_linattn_fused();
// Enqueues the whole call.  Returns 0 on success, 1 if this shape/device/output
// alignment is not handled (the caller uses the multi-launch path), or a
// negative status.
int launch_linattn_fused(MapCache& cache, const LinFusedArgs& a, int* status,
                         unsigned long long wait_ns, cudaStream_t stream);

}  // namespace ttt
