// Descriptors of one grouped-GEMM launch, shared by the host orchestration,
// the tcgen05 tensor-core kernel (bf16 operands) and the fp32 SIMT kernel.
//
// A launch holds up to kMaxProblems independent batched GEMM problems.  Each
// problem computes, for every batch index z and every 128 x bn output tile,
// up to three accumulators D_j = A_j * B_j (shared M, N, K) and hands the
// tile to one fused epilogue (gating, momentum, Newton-Schulz combination,
// output store).  Operands are 2-D row-major views: a K-major operand keeps
// K contiguous ("rows" are M or N), an MN-major operand keeps M or N
// contiguous ("rows" are K).
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace ttt {

constexpr int kMaxProblems = 4;
constexpr int kMaxMaps = 14;
constexpr int kMaxAcc = 3;

enum EpiKind : int {
  EPI_STORE_F32 = 0,   // out0 (fp32) = acc0
  EPI_PROJ_Q = 1,      // out0 (work) = SiLU(acc0) * acc1 (A_q); x (-eta) or x a if set
  EPI_PROJ_K = 2,      // dH1, dH3, P from H1 = acc0, H3 = acc1, VW2 = acc2
  EPI_GRAD = 3,        // M = beta M + acc; U or bf16 X (+ |M|_F^2) from M
  EPI_OUT = 4,         // out0 (io) = acc0
  EPI_NS_GRAM = 5,     // out0 (work) = acc0 * s^2          (A = X X^T)
  EPI_NS_POLY = 6,     // out0 (work) = b * in0 + c * acc0  (B = bA + cAA)
  EPI_NS_STEP = 7,     // out0 (work) or out0 (fp32) = s * (a * in0 + acc0)
};

// One operand of one accumulator.
struct OpDesc {
  // tensor-core path: a 2-D TMA map over the backing tensor
  short map;          // slot in GemmLaunch::maps
  short map3;         // MN-major tiles of 128+ columns: a 3-D map whose one box is the
                      // whole stage tile (64-column blocks), or -1 (one box per block)
  int mn_major;       // 0: K contiguous; 1: M/N contiguous
  int outer_base;     // outer (row) coordinate of batch 0's origin
  int inner_base;     // inner (column) coordinate of batch 0's origin
  int z_outer;        // outer-coordinate step per batch index
  int z_div;          // batch index used for this operand is z / z_div
  // SIMT path: element addressing (ptr already at batch 0's origin)
  const void* ptr;
  long long ld;       // elements between consecutive rows
  long long z_stride; // elements between consecutive batch indices (of z / z_div)
};

struct EpiDesc {
  int kind;
  int in_tmem;             // EPI_NS_POLY: G comes from the other TMEM accumulator buffer
  void* out[3];
  long long out_ld;       // elements between output rows
  long long out_z;        // elements between output batches
  long long out_row0;     // first output row of the problem's M range
  const void* in0;        // extra input tile (same indexing as out)
  const float* eta;       // per-row (token) learning rate
  long long eta_z;        // elements between batches of eta
  long long eta_row0;     // eta index of the problem's first row
  const float* normsq;    // per-batch sum of squares (Newton-Schulz scale)
  float* normsq_out;      // EPI_GRAD: per-batch partial sums of squares, one slot per
                          // (tile, warp): slot (tm * tiles_n + tn) * warps + warp of
                          // batch zz at normsq_out + zz * nslot (plain stores)
  int nslot;              // partial slots per batch
  float* mom;             // momentum, fp32, same indexing as out
  int z_div;              // batch index of eta / out is z / z_div (0/1 = z)
  int first;              // Newton-Schulz: first step (apply 1/|M|_F)
  int rows32;             // every output / input row is 32-byte aligned (set by the builder)
  float a, b, c;          // coefficients (NS a, b, c; momentum beta in a)
  float eps;
};

struct Problem {
  int M, N, K, Z;
  int bn;             // N tile (tensor-core path: 64..256, multiple of 16)
  int nacc;           // accumulators 1..3
  int a_shared;       // bit j: accumulator j reuses accumulator j-1's A tile
  int tiles_m, tiles_n;
  int tile_start;     // first linear tile index of this problem
  int kd;             // 64-deep K steps per pipeline stage: 0 or 1, or 2 (MN-major
                      // operand boxes then span 128 K rows, K-major tiles two boxes)
  OpDesc a[kMaxAcc];
  OpDesc b[kMaxAcc];
  EpiDesc epi;
};

struct GemmLaunch {
  CUtensorMap maps[kMaxMaps];
  Problem prob[kMaxProblems];
  int nprob;
  int total_tiles;
  int* status;                       // device status word
  unsigned long long wait_limit_ns;  // bounded-wait limit
};

}  // namespace ttt
