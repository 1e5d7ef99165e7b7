// Host entry of the cluster Newton-Schulz + normalise kernel (ns_cluster.cu).
#pragma once

#include <cuda_runtime.h>

#include "builder.h"

namespace ttt {

struct NsArgs {
  void* X[2];        // bf16 iterates [3*B*H][d*d]; X[0] holds M on entry
  void* G;           // bf16 Gram products [3*B*H][d*d]
  void* Bm;          // bf16 polynomial products [3*B*H][d*d]
  float* U;          // fp32 Muon output [3*B*H][d*d]
  float* normsq;     // squared Frobenius norms of M [3*B*H] (per-product paths)
  const float* normsq_part;  // their partial sums [3*B*H][nslot] (fused kernels)
  int nslot;
  float* W[3];       // fp32 state per slot (W1, W3, W2)
  void* Wb[3];       // bf16 operand copies per slot
  int BH, d, steps, l2norm;
  int h0, nh;        // (batch, head) range handled by this launch: [h0, h0 + nh)
  int slot0 = 0;     // matrix slots handled: [slot0, slot0 + nslots) of (W1, W3, W2)
  int nslots = 3;
  int zcount = 0;    // matrices in X / G (tensor-map extents); 0 = 3 * BH
  float ns[3];
  int priority = 0;  // launch priority (0: the stream's own)
};

// True if the cluster kernel handles d x d matrices; gives cluster size and N tile.
bool ns_cluster_applicable(int d, int* cs, int* bn);

// One-time per-device setup for d x d matrices (call before any stream
// capture); false if the cluster kernel cannot run them on this device.
bool prepare_ns_cluster(int d);

// Enqueues the whole Muon + update + normalisation for all matrices.
// Returns 0 on success, 1 if this device/shape cannot use the cluster kernel
// (the caller then uses the per-product launches), or a negative status.
int launch_ns_cluster(MapCache& cache, const NsArgs& a, int* status, unsigned long long wait_ns,
                      cudaStream_t stream);

}  // namespace ttt
