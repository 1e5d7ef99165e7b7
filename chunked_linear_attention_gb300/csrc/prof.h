// Launch accounting: a process-wide launch counter and, while a profile
// records, CUDA events around each launch with its algorithmic work.
#pragma once

#include <cuda_runtime.h>

namespace ttt {

enum ProfTag : int {
  PT_INIT = 0,
  PT_PROJ,
  PT_GRAD,
  PT_NS_GRAM,
  PT_NS_POLY,
  PT_NS_STEP,
  PT_NORM,
  PT_LIN_SCALE,
  PT_LIN_PARTIAL,
  PT_LIN_PREFIX,
  PT_LIN_OUT,
  PT_SELFTEST,
  PT_MUON,
  PT_MUON_HALF,
  PT_LIN_FUSED,
  PT_APPLY_PROJ,
  PT_APPLY_OUT,
  PT_FEATURIZE,
  PT_COUNT
};

// True while a profile is recording (launch sequences are then not cached as
// graphs, so every launch gets its events).
bool prof_recording();
// Adds launches that ran without a ProfScope (graph replays).
void prof_count_launches(size_t n);

// Records (when profiling) an event before the launch; the destructor
// records the one after and counts the launch.
class ProfScope {
 public:
  // `sm_share`: fraction of the device's SMs the launch's grid holds (<= 1).
  ProfScope(int tag, cudaStream_t s, double flops, double bytes, double sm_share = 1.0);
  ~ProfScope();

 private:
  int idx_;
  cudaStream_t s_;
};

}  // namespace ttt
