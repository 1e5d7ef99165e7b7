// Persistent grouped batched GEMM on the 5th-generation tensor cores (tcgen05
// + TMEM), operands staged by TMA into 128-byte-swizzled shared memory, fused
// epilogues from epilogue.cuh.
//
// One CTA per SM (the whole 227 KB of shared memory, all 512 TMEM columns)
// walks the launch's tiles with a static stride of gridDim.x.  Warp roles:
// lane 0 of warps 0 and 2 issue TMA loads into a ring of stages (alternate
// entries), warp 1 issues tcgen05.mma (the whole warp runs the loop, one
// elected lane issues), warps 3.. drain TMEM
// (tcgen05.ld) and run the epilogue.  When a tile needs at most 256 TMEM columns the accumulator is
// double-buffered, so the epilogue of one tile overlaps the MMAs of the next;
// the producer always runs ahead into the next tile.  Every wait is bounded
// and reports TTT_ERR_TIMEOUT into the device status word.
#include "exec.h"
#include "launch.h"
#include "tc_epilogue.cuh"
#include "umma_core.cuh"

namespace ttt {

static_assert(sizeof(GemmLaunch) <= 4096, "kernel parameter block too large");

// warp 0 and warp 2: TMA producers; warp 1: MMA issuer; warps 3..: epilogue
constexpr int kGemmKernelThreads = 96 + 32 * kEpiWarps;

// V8: every problem's epilogue rows are 32-byte aligned (lane-per-row 32-byte
// accesses); the other instantiation stages rows through shared memory.
template <bool V8>
__global__ void __launch_bounds__(kGemmKernelThreads, 1)
    umma_gemm_kernel(const __grid_constant__ GemmLaunch L) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxStages;
  uint64_t* accf = empty + kMaxStages;   // [2] accumulator ready (MMA -> epilogue)
  uint64_t* acce = accf + 2;             // [2] accumulator free (epilogue -> MMA)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce + 2);
  float* staging = reinterpret_cast<float*>(smem + kCtrlBytes);
  uint8_t* tiles = smem + kCtrlBytes + kStagingBytes;
  // The problem descriptors are read in every loop of every role: keep a copy
  // in shared memory (parameter space behind a generic pointer is slow).
  Problem* probs = reinterpret_cast<Problem*>(smem + kProbOffset);
  static_assert(kProbOffset + kMaxProblems * sizeof(Problem) <= kCtrlBytes, "control region");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  {
    const uint32_t* sw = reinterpret_cast<const uint32_t*>(L.prob);
    uint32_t* dw = reinterpret_cast<uint32_t*>(probs);
    const int words = (int)(L.nprob * sizeof(Problem) / 4);
    for (int i = threadIdx.x; i < words; i += blockDim.x) dw[i] = sw[i];
  }
  const int nprob = L.nprob, total_tiles = L.total_tiles;
  // each problem's stage plan, computed once (the roles look it up per tile)
  SmemPlan* plans = reinterpret_cast<SmemPlan*>(smem + kPlanOffset);
  static_assert(kProbOffset + kMaxProblems * sizeof(Problem) <= kPlanOffset, "control region");
  static_assert(kPlanOffset + kMaxProblems * sizeof(SmemPlan) <= kCtrlBytes - 64, "control region");
  __syncthreads();
  if (threadIdx.x < nprob) plan_problem(probs[threadIdx.x], plans[threadIdx.x]);
  __syncthreads();

  // one stage layout for the whole launch: the largest problem's
  uint32_t stage_bytes = 0;
  int max_cols = 0;
  for (int p = 0; p < nprob; ++p) {
    stage_bytes = max(stage_bytes, plans[p].max_bytes);
    max_cols = max(max_cols, probs[p].nacc * probs[p].bn);
  }
  int nstages = (kUmmaSmemBytes - 1024 - kCtrlBytes - kStagingBytes) / (int)stage_bytes;
  if (nstages > kMaxStages) nstages = kMaxStages;
  const int nbuf = max_cols <= 256 ? 2 : 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nstages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], kEpiWarps);
    }
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int p = 0; p < nprob; ++p)
      for (int j = 0; j < probs[p].nacc; ++j) {
        tma_prefetch_map(&L.maps[probs[p].a[j].map]);
        tma_prefetch_map(&L.maps[probs[p].b[j].map]);
      }
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const unsigned long long lim = L.wait_limit_ns;
  // everything above is this launch's own setup; from here on it reads and
  // writes what earlier launches in the stream produced or still read
  pdl_wait();

  if (warp == 0 || warp == 2) {
    // Two producer threads in different warps share the ring entries round
    // robin: each thread keeps only a few TMA boxes in flight.
    if (lane == 0) {
      const int plane = warp == 0 ? 0 : 1;
      int s = 0, filled = 0, e = 0;
      uint32_t ph = 0;
      for (int t = blockIdx.x; t < total_tiles; t += gridDim.x) {
        const TileCoord tc = decode_tile(probs, nprob, t);
        const Problem& P = probs[tc.prob];
        const SmemPlan& sp = plans[tc.prob];
        filled += sp.ngroups * (P.K / (kBK * sp.kd));
        if (!produce_tile(L.maps, P, sp, tc, tiles, stage_bytes, nstages, full, empty, s, ph,
                          plane, kProdLanes, e, L.status, lim))
          break;
      }
      if (plane == 0) drain_producer(full, nstages, s, ph, filled, L.status, lim);
    }
  } else if (warp == 1) {
    {   // the whole warp walks the loop; one elected lane issues
      int s = 0, it = 0;
      uint32_t ph = 0;
      const uint32_t tiles_saddr = smem_u32(tiles);
      for (int t = blockIdx.x; t < total_tiles; t += gridDim.x, ++it) {
        const TileCoord tc = decode_tile(probs, nprob, t);
        const Problem& P = probs[tc.prob];
        const SmemPlan& sp = plans[tc.prob];
        const int buf = it % nbuf;
        const uint32_t bph = (it / nbuf) & 1;
        if (!mbar_wait_w(&acce[buf], bph ^ 1, L.status, lim)) break;
        tc_fence_after();
        const bool ok = mma_tile(P, sp, tiles_saddr, stage_bytes, nstages, full, empty,
                                 tmem + buf * 256, s, ph, L.status, lim);
        umma_commit_w(&accf[buf]);
        if (!ok) break;
      }
      // the main loops are done: the next launch may start its setup while the
      // epilogues finish
      pdl_launch_dependents();
    }
  } else {
    int it = 0;
    const int ew = warp - 3;
    float* stage = staging + ew * kStageFloats;
    for (int t = blockIdx.x; t < total_tiles; t += gridDim.x, ++it) {
      const TileCoord tc = decode_tile(probs, nprob, t);
      const Problem& P = probs[tc.prob];
      const int buf = it % nbuf;
      const uint32_t bph = (it / nbuf) & 1;
      bool ok = false;
      const float sumsq = tc_epilogue_tile<V8>(P, tc.z, tc.tm, tc.tn, tmem + buf * 256, &accf[buf], bph,
                                           L.status, lim, &ok, stage, warp, ew, lane);
      if (P.epi.kind == EPI_GRAD && P.epi.normsq_out) {
        float ss = sumsq;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        if (lane == 0) {
          const int zz = P.epi.z_div > 1 ? tc.z / P.epi.z_div : tc.z;
          const int slot = (tc.tm * P.tiles_n + tc.tn) * kEpiWarps + ew;
          P.epi.normsq_out[(long long)zz * P.epi.nslot + slot] = ss;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce[buf]);
      if (!ok) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

static int g_attr_done[64] = {0};
static int g_sm_count[64] = {0};

cudaError_t prepare_umma_gemm() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(setup_mutex());
  if (!g_attr_done[dev]) {
    e = cudaFuncSetAttribute(umma_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kUmmaSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(umma_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kUmmaSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&g_sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_attr_done[dev] = 1;
  }
  return cudaSuccess;
}

int device_sm_count() {
  if (prepare_umma_gemm() != cudaSuccess) return 0;
  int dev = 0;
  cudaGetDevice(&dev);
  return g_sm_count[dev];
}

int umma_gemm_grid(const GemmLaunch& L, int max_ctas) {
  const int sms = device_sm_count();
  int grid = L.total_tiles < sms ? L.total_tiles : sms;
  if (max_ctas > 0 && grid > max_ctas) grid = max_ctas;
  return grid;
}

cudaError_t launch_umma_gemm(const GemmLaunch& L, cudaStream_t stream, int priority,
                             int max_ctas) {
  cudaError_t e = prepare_umma_gemm();
  if (e != cudaSuccess) return e;
  if (L.total_tiles <= 0) return cudaSuccess;
  const int grid = umma_gemm_grid(L, max_ctas);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributePriority;
  attr[1].val.priority = priority;
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kGemmKernelThreads, 1, 1);
  cfg.dynamicSmemBytes = kUmmaSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = priority != 0 ? 2 : 1;
  bool rows32 = true;
  for (int p = 0; p < L.nprob; ++p) rows32 = rows32 && L.prob[p].epi.rows32;
  if (rows32)
    return cudaLaunchKernelEx(&cfg, umma_gemm_kernel<true>, L);
  return cudaLaunchKernelEx(&cfg, umma_gemm_kernel<false>, L);
}

}  // namespace ttt
