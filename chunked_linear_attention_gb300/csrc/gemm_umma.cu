// Grouped batched GEMM on the 5th-generation tensor cores (tcgen05 + TMEM),
// operands staged by TMA into 128-byte-swizzled shared memory, with the fused
// epilogues of epilogue.cuh.  One CTA computes one 128 x bn output tile of one
// batch index of one problem, holding up to three fp32 accumulators in TMEM.
//
// Warp roles (192 threads): warp 0 issues TMA loads into a ring of stages,
// warp 1 owns the TMEM allocation and issues tcgen05.mma from one thread,
// warps 2..5 drain TMEM (tcgen05.ld) and run the epilogue, warp w reading
// TMEM lanes 32*(w%4)..+31 (one output row per thread).  Every wait is bounded
// and reports TTT_ERR_TIMEOUT into the device status word.
#include "common.cuh"
#include "epilogue.cuh"
#include "launch.h"

namespace ttt {

static_assert(sizeof(GemmLaunch) <= 4096, "kernel parameter block too large");

constexpr int kUmmaThreads = 192;
constexpr int kBM = 128;
constexpr int kBK = 64;                      // one 128-byte swizzle row of bf16
constexpr int kATileBytes = kBM * kBK * 2;   // 16 KB
constexpr int kMaxStages = 8;
constexpr int kCtrlBytes = 1024;             // barriers + TMEM slot

struct TileCoord {
  int prob, z, tm, tn;
};

__device__ __forceinline__ TileCoord decode_tile(const GemmLaunch& L, int t) {
  int p = 0;
#pragma unroll 1
  for (int i = 1; i < L.nprob; ++i)
    if (t >= L.prob[i].tile_start) p = i;
  const Problem& P = L.prob[p];
  int local = t - P.tile_start;
  TileCoord c;
  c.prob = p;
  c.tn = local % P.tiles_n;
  local /= P.tiles_n;
  c.tm = local % P.tiles_m;
  c.z = local / P.tiles_m;
  return c;
}

// Issue the TMA boxes of one operand tile (rows x 64 of K) for k-step ks.
__device__ __forceinline__ void load_operand(const GemmLaunch& L, const OpDesc& op, uint8_t* dst,
                                             int rows, int mn0, int ks, int z, uint64_t* bar) {
  const int zz = op.z_div > 1 ? z / op.z_div : z;
  const CUtensorMap* map = &L.maps[op.map];
  if (!op.mn_major) {
    tma_load_2d(dst, map, op.inner_base + ks * kBK, op.outer_base + zz * op.z_outer + mn0, bar);
  } else {
    for (int i = 0; i < rows / 64; ++i)
      tma_load_2d(dst + i * 8192, map, op.inner_base + mn0 + i * 64,
                  op.outer_base + zz * op.z_outer + ks * kBK, bar);
  }
}

__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int mn_major, int kk) {
  // K-major: a 16-element K slice starts 32 bytes further along the row.
  // MN-major: it starts 16 K-rows (2 KB) further down.
  return mn_major ? smem_desc_sw128(base + kk * 2048, 8192, 1024)
                  : smem_desc_sw128(base + kk * 32, 16, 1024);
}

__global__ void __launch_bounds__(kUmmaThreads, 1)
    umma_gemm_kernel(const __grid_constant__ GemmLaunch L) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxStages;
  uint64_t* accf = empty + kMaxStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accf + 1);
  uint8_t* tiles = smem + kCtrlBytes;

  const TileCoord tc = decode_tile(L, blockIdx.x);
  const Problem& P = L.prob[tc.prob];
  const int nacc = P.nacc, bn = P.bn;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  uint32_t a_off[kMaxAcc], b_off[kMaxAcc], stage_bytes = 0, tx_bytes = 0;
#pragma unroll
  for (int j = 0; j < kMaxAcc; ++j) {
    if (j >= nacc) break;
    if (j > 0 && ((P.a_shared >> j) & 1)) {
      a_off[j] = a_off[j - 1];
    } else {
      a_off[j] = stage_bytes;
      stage_bytes += kATileBytes;
    }
  }
#pragma unroll
  for (int j = 0; j < kMaxAcc; ++j) {
    if (j >= nacc) break;
    b_off[j] = stage_bytes;
    stage_bytes += bn * kBK * 2;
  }
  tx_bytes = stage_bytes;
  int nstages = (kUmmaSmemBytes - 1024 - kCtrlBytes) / (int)stage_bytes;
  if (nstages > kMaxStages) nstages = kMaxStages;
  const int nk = P.K / kBK;
  uint32_t ncols = 32;
  while (ncols < (uint32_t)(nacc * bn)) ncols <<= 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nstages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accf, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int j = 0; j < nacc; ++j) {
      tma_prefetch_map(&L.maps[P.a[j].map]);
      tma_prefetch_map(&L.maps[P.b[j].map]);
    }
  }
  if (warp == 1) tmem_alloc(tmem_slot, ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const unsigned long long lim = L.wait_limit_ns;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    int issued = 0;
    for (int ks = 0; ks < nk; ++ks) {
      const int s = ks % nstages;
      const uint32_t ph = (ks / nstages) & 1;
      if (!mbar_wait(&empty[s], ph ^ 1, L.status, lim)) break;
      mbar_arrive_expect_tx(&full[s], tx_bytes);
      uint8_t* st = tiles + s * stage_bytes;
      for (int j = 0; j < nacc; ++j) {
        if (!(j > 0 && ((P.a_shared >> j) & 1)))
          load_operand(L, P.a[j], st + a_off[j], kBM, tc.tm * kBM, ks, tc.z, &full[s]);
        load_operand(L, P.b[j], st + b_off[j], bn, tc.tn * bn, ks, tc.z, &full[s]);
      }
      issued = ks + 1;
    }
    // wait (bounded) until the copies of the last stages have landed
    for (int ks = issued > nstages ? issued - nstages : 0; ks < issued; ++ks)
      mbar_wait(&full[ks % nstages], (ks / nstages) & 1, L.status, lim);
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer
    uint32_t idesc[kMaxAcc];
    for (int j = 0; j < nacc; ++j) idesc[j] = idesc_bf16_f32(bn, P.a[j].mn_major, P.b[j].mn_major);
    for (int ks = 0; ks < nk; ++ks) {
      const int s = ks % nstages;
      const uint32_t ph = (ks / nstages) & 1;
      if (!mbar_wait(&full[s], ph, L.status, lim)) break;
      tc_fence_after();
      const uint32_t st = smem_u32(tiles + s * stage_bytes);
      for (int j = 0; j < nacc; ++j) {
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          const uint64_t ad = operand_desc(st + a_off[j], P.a[j].mn_major, kk);
          const uint64_t bd = operand_desc(st + b_off[j], P.b[j].mn_major, kk);
          umma_bf16(tmem + j * bn, ad, bd, idesc[j], (ks | kk) != 0);
        }
      }
      umma_commit(&empty[s]);
    }
    umma_commit(accf);
  } else if (warp >= 2) {
    // ---------------- epilogue
    const bool ok = mbar_wait(accf, 0, L.status, lim);
    tc_fence_after();
    const int sub = warp & 3;
    const int row = sub * 32 + lane;
    const int grow = tc.tm * kBM + row;
    const uint32_t tl = tmem + ((uint32_t)(sub * 32) << 16);
    float sumsq = 0.f;
    if (ok) {
      for (int c0 = 0; c0 < bn; c0 += 16) {
        float v0[16], v1[16], v2[16];
        tmem_ld16(tl + c0, v0);
        if (nacc > 1) tmem_ld16(tl + bn + c0, v1);
        if (nacc > 2) tmem_ld16(tl + 2 * bn + c0, v2);
        const int gcol = tc.tn * bn + c0;
        if (grow < P.M && gcol < P.N) {
          const int n = min(16, P.N - gcol);
          sumsq += epilogue_vec<16, __nv_bfloat16, __nv_bfloat16, false>(P.epi, tc.z, grow, gcol,
                                                                        n, v0, v1, v2);
        }
      }
    }
    if (P.epi.kind == EPI_GRAD && P.epi.normsq_out) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sumsq += __shfl_xor_sync(0xffffffffu, sumsq, off);
      if (lane == 0) {
        const int zz = P.epi.z_div > 1 ? tc.z / P.epi.z_div : tc.z;
        atomicAdd(P.epi.normsq_out + zz, sumsq);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

cudaError_t launch_umma_gemm(const GemmLaunch& L, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(umma_gemm_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kUmmaSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (L.total_tiles <= 0) return cudaSuccess;
  umma_gemm_kernel<<<L.total_tiles, kUmmaThreads, kUmmaSmemBytes, stream>>>(L);
  return cudaGetLastError();
}

}  // namespace ttt
