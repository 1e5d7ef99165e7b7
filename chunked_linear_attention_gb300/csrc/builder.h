// Host-side construction of grouped-GEMM launches: tensor views, TMA maps
// (encoded once per call and reused), tile counts, and the launch itself on
// the tensor-core kernel (bf16) or the fp32 SIMT kernel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <vector>

#include "gemm_desc.h"
#include "launch.h"

namespace ttt {

// A dense row-major 2-D view: `rows` rows of `inner` elements.
struct TensorRef {
  const void* ptr;
  int bf16;        // element type: 1 = bf16, 0 = fp32
  long long rows;
  int inner;
};

// TMA descriptors encoded during one call, keyed by view and box height.
// Boxes are one 128-byte swizzle row wide (64 bf16 or 32 fp32 elements).
class MapCache {
 public:
  bool get(const TensorRef& t, int box_rows, CUtensorMap* out);
  // bf16 view read as 64-column blocks: coordinates {column in block, row,
  // block}; one box is `nblk` consecutive blocks of box_rows rows, landing in
  // shared memory block after block (MN-major operand atoms of 64 columns).
  bool get_blocked(const TensorRef& t, int box_rows, int nblk, CUtensorMap* out);

 private:
  struct Entry {
    const void* ptr;
    int bf16;
    long long rows;
    int inner;
    int box_rows;
    int nblk;   // 0: plain 2-D map
    CUtensorMap map;
  };
  std::vector<Entry> entries_;
};

class LaunchBuilder {
 public:
  LaunchBuilder(bool tensor_cores, MapCache* cache, int* status, unsigned long long wait_ns);

  void reset();
  // Operand view: K-major (mn_major = 0) or MN-major; the tile origin of batch
  // z is row outer_base + z * z_outer of `t`.
  // MN-major operands load boxes of 64 M/N columns by mn_krows K rows (64, or
  // 128 for problems with two K steps per stage).
  OpDesc op(const TensorRef& t, int mn_major, int outer_base, int z_outer, int box_rows,
            int mn_krows = 64);
  // Tile N size for a problem with `nacc` accumulators and N columns.
  int choose_bn(int N, int nacc) const;
  // Fills tiles and appends.  Returns false when the launch is full.
  bool add(Problem p);
  // Launches with launch accounting under profile tag `tag` (tensor-core
  // launches at `priority`, 0 = the stream's own).
  cudaError_t launch(cudaStream_t stream, int tag, int priority = 0, int max_ctas = 0);
  bool ok() const { return ok_; }
  bool tensor_cores() const { return tc_; }
  int bm() const { return tc_ ? 128 : kSimtTile; }

 private:
  GemmLaunch L_;
  bool tc_;
  MapCache* cache_;
  int nmaps_;
  const void* keys_ptr_[kMaxMaps];
  long long keys_rows_[kMaxMaps];
  int keys_inner_[kMaxMaps];
  int keys_box_[kMaxMaps];
  int keys_nblk_[kMaxMaps];   // 0: 2-D map; else a 3-D blocked map of nblk 64-column blocks
  // Slot of the 3-D blocked map for an MN-major operand whose tile spans
  // `cols` columns (>= 128), or -1 when the 2-D boxes must serve.
  int blocked_slot(int map2d, int cols);
  bool ok_;
  int* status_;
  unsigned long long wait_ns_;
};

}  // namespace ttt
