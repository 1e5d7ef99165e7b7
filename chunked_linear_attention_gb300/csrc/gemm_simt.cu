// Grouped batched GEMM in plain fp32 FFMA (no TF32) for the fp32 I/O path.
// Same problem descriptors and epilogues as the tensor-core kernel; 64 x 64
// output tiles, 256 threads, each thread 4 x 4 outputs per accumulator.
// Any M, N, K (bounds-checked loads); operands are fp32.
#include "common.cuh"
#include "epilogue.cuh"
#include "launch.h"

namespace ttt {

constexpr int kSK = 16;

__device__ __forceinline__ float simt_load(const OpDesc& op, int z, int mn, int k, int mn_ext,
                                           int K) {
  if (mn >= mn_ext || k >= K) return 0.f;
  const int zz = op.z_div > 1 ? z / op.z_div : z;
  const float* p = static_cast<const float*>(op.ptr) + (long long)zz * op.z_stride;
  return op.mn_major ? p[(long long)k * op.ld + mn] : p[(long long)mn * op.ld + k];
}

__global__ void __launch_bounds__(256) simt_gemm_kernel(const __grid_constant__ GemmLaunch L) {
  __shared__ float As[kMaxAcc][kSK][kSimtTile + 1];
  __shared__ float Bs[kMaxAcc][kSK][kSimtTile + 1];

  const int t = blockIdx.x;
  int p = 0;
  for (int i = 1; i < L.nprob; ++i)
    if (t >= L.prob[i].tile_start) p = i;
  const Problem& P = L.prob[p];
  int local = t - P.tile_start;
  const int tn = local % P.tiles_n;
  local /= P.tiles_n;
  const int tm = local % P.tiles_m;
  const int z = local / P.tiles_m;
  const int m0 = tm * kSimtTile, n0 = tn * kSimtTile;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;

  float acc[kMaxAcc][4][4];
#pragma unroll
  for (int j = 0; j < kMaxAcc; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[j][i][k] = 0.f;

  for (int k0 = 0; k0 < P.K; k0 += kSK) {
    for (int j = 0; j < P.nacc; ++j) {
      for (int i = threadIdx.x; i < kSimtTile * kSK; i += 256) {
        const int mm = i % kSimtTile, kk = i / kSimtTile;
        As[j][kk][mm] = simt_load(P.a[j], z, m0 + mm, k0 + kk, P.M, P.K);
        Bs[j][kk][mm] = simt_load(P.b[j], z, n0 + mm, k0 + kk, P.N, P.K);
      }
    }
    __syncthreads();
    for (int j = 0; j < P.nacc; ++j) {
#pragma unroll
      for (int kk = 0; kk < kSK; ++kk) {
        float a[4], b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          a[i] = As[j][kk][ty * 4 + i];
          b[i] = Bs[j][kk][tx * 4 + i];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int k = 0; k < 4; ++k) acc[j][i][k] = fmaf(a[i], b[k], acc[j][i][k]);
      }
    }
    __syncthreads();
  }

  float sumsq = 0.f;
  const int gc = n0 + tx * 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gr = m0 + ty * 4 + i;
    if (gr < P.M && gc < P.N) {
      const int n = min(4, P.N - gc);
      sumsq += epilogue_vec<4, float, float, true>(P.epi, z, gr, gc, n, acc[0][i], acc[1][i],
                                                  acc[2][i]);
    }
  }
  if (P.epi.kind == EPI_GRAD && P.epi.normsq_out) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sumsq += __shfl_xor_sync(0xffffffffu, sumsq, off);
    if ((threadIdx.x & 31) == 0) {
      const int zz = P.epi.z_div > 1 ? z / P.epi.z_div : z;
      const int slot = (tm * P.tiles_n + tn) * 8 + (int)(threadIdx.x >> 5);
      P.epi.normsq_out[(long long)zz * P.epi.nslot + slot] = sumsq;
    }
  }
}

cudaError_t launch_simt_gemm(const GemmLaunch& L, cudaStream_t stream) {
  if (L.total_tiles <= 0) return cudaSuccess;
  simt_gemm_kernel<<<L.total_tiles, 256, 0, stream>>>(L);
  return cudaGetLastError();
}

}  // namespace ttt
