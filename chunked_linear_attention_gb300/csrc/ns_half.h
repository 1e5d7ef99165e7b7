// Host entry of the half-panel Newton-Schulz + normalise kernel (ns_half.cu):
// square d x d fast weights with d a multiple of 128, d <= 512.
#pragma once

#include <cuda_runtime.h>

#include "builder.h"
#include "ns_cluster.h"

namespace ttt {

// True if the half-panel kernel handles d x d matrices (shared-memory fit).
bool ns_half_applicable(int d);

// One-time per-device setup (call before any stream capture); false if the
// kernel cannot run d x d matrices on this device (cluster of 2 d / 128).
bool prepare_ns_half(int d);

// Enqueues the whole Muon + update + normalisation of the (batch, head) range
// of `a` for all three matrix slots.  Uses a.X[0] (holding M on entry),
// a.X[1], a.G, a.normsq, a.W, a.Wb; a.Bm and a.U are not touched.
// Returns 0 on success, 1 if the kernel does not apply, or a negative status.
int launch_ns_half(MapCache& cache, const NsArgs& a, int* status, unsigned long long wait_ns,
                   cudaStream_t stream);

}  // namespace ttt
