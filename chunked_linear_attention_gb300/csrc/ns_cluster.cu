// Muon for square fast-weight matrices in one launch per update: every
// Newton-Schulz step (eq 6 of the LaCT notes; the quintic of the Muon
// write-up) and the final W <- L2-Normalize(W - U) (eq 5), for all matrices.
//
// One thread-block cluster per matrix; each CTA of the cluster owns one
// 128 x bn output tile of every product (e.g. 6 CTAs for 384 x 384 with
// bn = 192).  Per step the cluster runs
//     G  = X X^T          (first step: scaled by 1/(|M|_F + eps)^2)
//     Bm = b G + c G G
//     X' = a X + Bm X     (first step: scaled by 1/(|M|_F + eps))
// with the same TMA -> tcgen05 -> TMEM machinery as the grouped GEMM.  Each
// product's tiles go to global memory (they stay in L2); a cluster barrier
// (release/acquire) separates dependent products, so there is no kernel
// boundary between the 3 x steps products.  The last product writes U in
// fp32; after one more barrier the cluster's CTAs split the rows of the
// matrix for the update and row normalisation, refresh the bf16 operand copy
// and clear the matrix's Frobenius accumulator.
#include <cstring>

#include "builder.h"
#include "exec.h"
#include "launch.h"
#include "ns_cluster.h"
#include "prof.h"
#include "tc_epilogue.cuh"
#include "umma_core.cuh"

namespace ttt {

enum NsMap : int {
  NM_X0_A = 0, NM_X0_B, NM_X0_MN, NM_X1_A, NM_X1_B, NM_X1_MN, NM_G_A, NM_G_B, NM_BM_A, NM_COUNT
};

struct NsLaunch {
  CUtensorMap maps[kMaxMaps];
  Problem gram, poly, step;   // templates for even steps (X0 -> X1)
  const void* X[2];
  float* U;
  float* W[3];                // fp32 state per slot (W1, W3, W2), [B*H][d*d]
  void* Wb[3];                // bf16 operand copies per slot
  int BH, d, steps, cs, l2norm;
  int h0, nh;                 // (batch, head) range of this launch
  int slot0;                  // first matrix slot of this launch
  int* status;
  unsigned long long wait_limit_ns;
};

static_assert(sizeof(NsLaunch) <= 4096, "kernel parameter block too large");

// Rewrites the step-dependent fields of one product for step t.
__device__ __forceinline__ void ns_patch(const NsLaunch& L, Problem& P, int which, int t) {
  const int in = t & 1;
  const bool last = t == L.steps - 1;
  if (which == 0) {          // G = X X^T
    P.a[0].map = in ? NM_X1_A : NM_X0_A;
    P.b[0].map = in ? NM_X1_B : NM_X0_B;
    P.epi.first = t == 0;
  } else if (which == 1) {   // Bm = b G + c G G, G from the other TMEM buffer
    P.epi.first = t == 0;
  } else if (which == 2) {   // X' = a X + Bm X
    P.b[0].map = in ? NM_X1_MN : NM_X0_MN;
    P.epi.in0 = L.X[in];
    P.epi.first = t == 0;
    if (last) {
      P.epi.out[0] = nullptr;
      P.epi.out[1] = L.U;
    } else {
      P.epi.out[0] = const_cast<void*>(L.X[in ^ 1]);
      P.epi.out[1] = nullptr;
    }
  }
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    ns_cluster_kernel(const __grid_constant__ NsLaunch L) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxStages;
  uint64_t* accf = empty + kMaxStages;
  uint64_t* acce = accf + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce + 2);
  Problem* cur = reinterpret_cast<Problem*>(smem + 256);
  static_assert(256 + sizeof(Problem) <= kCtrlBytes, "control region too small");
  float* staging = reinterpret_cast<float*>(smem + kCtrlBytes);
  uint8_t* tiles = smem + kCtrlBytes + kStagingBytes;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)cluster_ctarank();
  // matrix index (slot-major over B*H) of this cluster
  const int zl = blockIdx.x / L.cs;
  const int z = (L.slot0 + zl / L.nh) * L.BH + L.h0 + (zl % L.nh);

  uint32_t stage_bytes = 0;
  {
    SmemPlan sp;
    plan_problem(L.gram, sp);
    stage_bytes = max(stage_bytes, sp.max_bytes);
    plan_problem(L.poly, sp);
    stage_bytes = max(stage_bytes, sp.max_bytes);
    plan_problem(L.step, sp);
    stage_bytes = max(stage_bytes, sp.max_bytes);
  }
  int nstages = (kUmmaSmemBytes - 1024 - kCtrlBytes - kStagingBytes) / (int)stage_bytes;
  if (nstages > kMaxStages) nstages = kMaxStages;

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
  if (warp == 0 && lane == 0)
    for (int i = 0; i < NM_COUNT; ++i) tma_prefetch_map(&L.maps[i]);
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const unsigned long long lim = L.wait_limit_ns;
  const uint32_t tiles_saddr = smem_u32(tiles);

  int s_prod = 0, s_mma = 0, filled = 0, it_mma = 0, it_epi = 0, e_prod = 0;
  uint32_t ph_prod = 0, ph_mma = 0;
  bool ok = true;
  for (int t = 0; t < L.steps; ++t) {
    for (int which = 0; which < 3; ++which) {
      {  // copy the product's template into shared memory (all threads), then patch it
        const Problem& src = which == 0 ? L.gram : (which == 1 ? L.poly : L.step);
        const uint32_t* sw = reinterpret_cast<const uint32_t*>(&src);
        uint32_t* dw = reinterpret_cast<uint32_t*>(cur);
        for (int i = threadIdx.x; i < (int)(sizeof(Problem) / 4); i += blockDim.x) dw[i] = sw[i];
        __syncthreads();
        if (threadIdx.x == 0) ns_patch(L, *cur, which, t);
      }
      __syncthreads();
      const Problem& P = *cur;
      const int ntiles = P.tiles_m * P.tiles_n;
      if (warp == 0) {
        if (lane == 0 && ok) {
          SmemPlan sp;
          plan_problem(P, sp);
          for (int tile = rank; tile < ntiles; tile += L.cs) {
            const TileCoord tc{0, z, tile / P.tiles_n, tile % P.tiles_n};
            filled += sp.ngroups * (P.K / kBK);
            if (!produce_tile(L.maps, P, sp, tc, tiles, stage_bytes, nstages, full, empty, s_prod,
                              ph_prod, 0, 1, e_prod, L.status, lim)) {
              ok = false;
              break;
            }
          }
        }
      } else if (warp == 1) {
        if (ok) {   // the whole warp walks the loop; one elected lane issues
          SmemPlan sp;
          plan_problem(P, sp);
          for (int tile = rank; tile < ntiles; tile += L.cs, ++it_mma) {
            const int buf = it_mma & 1;
            const uint32_t bph = (it_mma >> 1) & 1;
            if (!mbar_wait_w(&acce[buf], bph ^ 1, L.status, lim)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const bool good = mma_tile(P, sp, tiles_saddr, stage_bytes, nstages, full, empty,
                                       tmem + buf * 256, s_mma, ph_mma, L.status, lim);
            umma_commit_w(&accf[buf]);
            if (!good) {
              ok = false;
              break;
            }
          }
        }
      } else {
        float* stage = staging + (warp - 2) * kStageFloats;
        for (int tile = rank; tile < ntiles; tile += L.cs, ++it_epi) {
          const int buf = it_epi & 1;
          const uint32_t bph = (it_epi >> 1) & 1;
          bool got = false;
          if (ok)
            tc_epilogue_tile<false>(P, z, tile / P.tiles_n, tile % P.tiles_n, tmem + buf * 256, &accf[buf],
                             bph, L.status, lim, &got, stage, warp, warp - 2, lane);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acce[buf]);
          if (!got) ok = false;
        }
        fence_proxy_async_global();   // our tiles are read by TMA after the barrier
      }
      __syncthreads();
      cluster_sync_all();
    }
  }

  // W <- L2-Normalize(W - U) over this CTA's share of the matrix rows
  {
    const int d = L.d;
    const int slot = z / L.BH, bh = z % L.BH;
    const long long base = (long long)bh * d * d;
    float* W = L.W[slot] + base;
    __nv_bfloat16* Wb = static_cast<__nv_bfloat16*>(L.Wb[slot]) + base;
    const float* U = L.U + (long long)z * d * d;
    const int rows_per = (d + L.cs - 1) / L.cs;
    const int r0 = rank * rows_per, r1 = min(d, r0 + rows_per);
    for (int r = r0 + warp; r < r1; r += kGemmThreads / 32) {
      float vals[32];
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int c = lane + 32 * i;
        float x = 0.f;
        if (c < d) x = W[(long long)r * d + c] - U[(long long)r * d + c];
        vals[i] = x;
        ss += x * x;
      }
      float scale = 1.f;
      if (L.l2norm) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        scale = 1.0f / fmaxf(sqrtf(ss), 1e-12f);
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int c = lane + 32 * i;
        if (c < d) {
          const float y = vals[i] * scale;
          W[(long long)r * d + c] = y;
          Wb[(long long)r * d + c] = __float2bfloat16_rn(y);
        }
      }
    }
  }

  if (warp == 0 && lane == 0) drain_producer(full, nstages, s_prod, ph_prod, filled, L.status, lim);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- host

static int cluster_ok_cache[64][9];   // 0 unknown, 1 fits, 2 does not

bool ns_cluster_applicable(int d, int* cs_out, int* bn_out) {
  if (d % 64 != 0 || d > 512) return false;
  const int tiles_m = (d + 127) / 128;
  const int bn = d <= 256 ? d : (d % 192 == 0 ? 192 : 256);
  const int tiles_n = (d + bn - 1) / bn;
  const int cs = tiles_m * tiles_n;
  if (cs > 8) return false;
  *cs_out = cs;
  *bn_out = bn;
  return true;
}

static bool cluster_fits(int dev, int cs) {
  if (dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lk(setup_mutex());
  int& c = cluster_ok_cache[dev][cs];
  if (c == 0) {
    c = 2;
    if (cudaFuncSetAttribute(ns_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kUmmaSmemBytes) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = cs;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(cs, 1, 1);
      cfg.blockDim = dim3(kGemmThreads, 1, 1);
      cfg.dynamicSmemBytes = kUmmaSmemBytes;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, ns_cluster_kernel, &cfg) == cudaSuccess && n > 0)
        c = 1;
    }
    cudaGetLastError();
  }
  return c == 1;
}

bool prepare_ns_cluster(int d) {
  int cs = 0, bn = 0;
  if (!ns_cluster_applicable(d, &cs, &bn)) return false;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  return cluster_fits(dev, cs);
}

int launch_ns_cluster(MapCache& cache, const NsArgs& a, int* status, unsigned long long wait_ns,
                      cudaStream_t stream) {
  int cs = 0, bn = 0;
  if (!ns_cluster_applicable(a.d, &cs, &bn)) return 1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -6;
  if (!cluster_fits(dev, cs)) return 1;

  const int d = a.d, Z = 3 * a.BH;
  NsLaunch L;
  std::memset(&L, 0, sizeof(L));
  TensorRef TX0{a.X[0], 1, (long long)Z * d, d};
  TensorRef TX1{a.X[1], 1, (long long)Z * d, d};
  TensorRef TG{a.G, 1, (long long)Z * d, d};
  TensorRef TB{a.Bm, 1, (long long)Z * d, d};
  const struct {
    TensorRef t;
    int box;
  } maps[NM_COUNT] = {{TX0, 128}, {TX0, bn}, {TX0, 64}, {TX1, 128}, {TX1, bn},
                      {TX1, 64},  {TG, 128}, {TG, bn},  {TB, 128}};
  for (int i = 0; i < NM_COUNT; ++i)
    if (!cache.get(maps[i].t, maps[i].box, &L.maps[i])) return -4;

  auto base = [&](int K) {
    Problem p;
    std::memset(&p, 0, sizeof(p));
    p.M = d;
    p.N = d;
    p.K = K;
    p.Z = Z;
    p.nacc = 1;
    p.bn = bn;
    p.tiles_m = (d + 127) / 128;
    p.tiles_n = (d + bn - 1) / bn;
    p.epi.z_div = 1;
    p.epi.out_ld = d;
    p.epi.out_z = (long long)d * d;
    p.epi.normsq = a.normsq;
    p.epi.eps = 1e-7f;
    return p;
  };
  auto op = [&](int map, int mn) {
    OpDesc o;
    std::memset(&o, 0, sizeof(o));
    o.map3 = -1;   // MN-major tiles go as 64-column 2-D boxes (no 3-D map here)
    o.map = map;
    o.mn_major = mn;
    o.z_outer = d;
    o.z_div = 1;
    return o;
  };
  L.gram = base(d);
  L.gram.a[0] = op(NM_X0_A, 0);
  L.gram.b[0] = op(NM_X0_B, 0);
  L.gram.epi.kind = EPI_NS_GRAM;
  L.gram.epi.out[0] = a.G;
  L.poly = base(d);
  L.poly.a[0] = op(NM_G_A, 0);
  L.poly.b[0] = op(NM_G_B, 0);
  L.poly.epi.kind = EPI_NS_POLY;
  L.poly.epi.in0 = a.G;
  L.poly.epi.out[0] = a.Bm;
  L.poly.epi.b = a.ns[1];
  L.poly.epi.c = a.ns[2];
  L.poly.epi.in_tmem = 1;   // each CTA keeps its Gram tile in TMEM for the next product
  L.step = base(d);
  L.step.a[0] = op(NM_BM_A, 0);
  L.step.b[0] = op(NM_X0_MN, 1);
  L.step.epi.kind = EPI_NS_STEP;
  L.step.epi.a = a.ns[0];
  L.X[0] = a.X[0];
  L.X[1] = a.X[1];
  L.U = a.U;
  for (int s = 0; s < 3; ++s) {
    L.W[s] = a.W[s];
    L.Wb[s] = a.Wb[s];
  }
  L.BH = a.BH;
  L.h0 = a.h0;
  L.nh = a.nh;
  L.slot0 = a.slot0;
  L.d = d;
  L.steps = a.steps;
  L.cs = cs;
  L.l2norm = a.l2norm;
  L.status = status;
  L.wait_limit_ns = wait_ns;

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(a.nslots * a.nh * cs, 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = kUmmaSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const double r = d, c = d;
  const double flops = (double)a.nslots * a.nh * a.steps * (4 * r * c * c + 2 * c * c * c);
  ProfScope ps(PT_MUON, stream, flops, 0.0);
  if (cudaLaunchKernelEx(&cfg, ns_cluster_kernel, L) != cudaSuccess) return -6;
  return 0;
}

}  // namespace ttt
