// Tensor-core epilogue: drains one tile's TMEM accumulators and applies the
// fused epilogue of epilogue.cuh, with memory traffic shaped for the GPU:
//
//   * each epilogue warp owns 32 rows (its TMEM lane quarter) and the tile's
//     columns, processed in blocks of kBW columns;
//   * per-row scalars (eta, the Newton-Schulz scale) are read once per tile,
//     before waiting for the accumulator;
//   * input tiles (momentum, Newton-Schulz iterates) are fetched with
//     coalesced 16-byte loads one block ahead, then transposed through a
//     padded per-warp staging buffer in shared memory;
//   * outputs go back through the same buffer and leave as coalesced 16-byte
//     stores that cover whole 64/128-byte row segments.
// The staging buffer holds 32 rows x (kBW + 1) floats (the pad spreads both
// the row-wise and the chunk-wise accesses over the banks).
#pragma once

#include "common.cuh"
#include "epilogue.cuh"
#include "umma_core.cuh"

namespace ttt {

constexpr int kBW = 16;                               // columns per epilogue block
constexpr int kStageStride = kBW + 1;                 // floats per staged row (padded)
constexpr int kStageFloats = 32 * kStageStride;       // per warp
// all epilogue warps' staging buffers, rounded up to keep the stage ring 1 KB aligned
constexpr int kStagingBytes = (kEpiWarps * kStageFloats * 4 + 1023) / 1024 * 1024;

// 32 x kBW block of T starting at `base` of a row-major matrix with leading
// dimension ld; one warp, coalesced 16-byte accesses.
template <typename T>
struct BlockRegs {
  static constexpr int kCPR = kBW * (int)sizeof(T) / 16;   // 16-byte chunks per row
  static constexpr int kRPI = 32 / kCPR;                    // rows per warp instruction
  uint4 r[32 / kRPI];
};

template <typename T>
__device__ __forceinline__ void block_load(const T* base, long long ld, int rows_valid,
                                           BlockRegs<T>& g, int lane) {
  constexpr int kCPR = BlockRegs<T>::kCPR;
  constexpr int kRPI = BlockRegs<T>::kRPI;
#pragma unroll
  for (int i = 0; i < 32 / kRPI; ++i) {
    const int r = i * kRPI + lane / kCPR;
    const int ch = lane % kCPR;
    if (r < rows_valid)
      g.r[i] = *reinterpret_cast<const uint4*>(base + (long long)r * ld + ch * (16 / sizeof(T)));
    else
      g.r[i] = make_uint4(0, 0, 0, 0);
  }
}

// Coalesced registers -> staging (as fp32).
template <typename T>
__device__ __forceinline__ void block_to_stage(const BlockRegs<T>& g, float* stage, int lane) {
  constexpr int kCPR = BlockRegs<T>::kCPR;
  constexpr int kRPI = BlockRegs<T>::kRPI;
  constexpr int kEPC = 16 / sizeof(T);  // elements per chunk
#pragma unroll
  for (int i = 0; i < 32 / kRPI; ++i) {
    const int r = i * kRPI + lane / kCPR;
    const int c = (lane % kCPR) * kEPC;
    float* dst = stage + r * kStageStride + c;
    const uint4 v = g.r[i];
    if constexpr (sizeof(T) == 2) {
      dst[0] = bf16lo(v.x); dst[1] = bf16hi(v.x); dst[2] = bf16lo(v.y); dst[3] = bf16hi(v.y);
      dst[4] = bf16lo(v.z); dst[5] = bf16hi(v.z); dst[6] = bf16lo(v.w); dst[7] = bf16hi(v.w);
    } else {
      dst[0] = __uint_as_float(v.x); dst[1] = __uint_as_float(v.y);
      dst[2] = __uint_as_float(v.z); dst[3] = __uint_as_float(v.w);
    }
  }
}

// Staging -> global, coalesced, converting to T.
template <typename T>
__device__ __forceinline__ void stage_to_global(const float* stage, T* base, long long ld,
                                                int rows_valid, int lane) {
  constexpr int kCPR = BlockRegs<T>::kCPR;
  constexpr int kRPI = BlockRegs<T>::kRPI;
  constexpr int kEPC = 16 / sizeof(T);
#pragma unroll
  for (int i = 0; i < 32 / kRPI; ++i) {
    const int r = i * kRPI + lane / kCPR;
    const int c = (lane % kCPR) * kEPC;
    const float* s = stage + r * kStageStride + c;
    uint4 v;
    if constexpr (sizeof(T) == 2) {
      v = make_uint4(pack_bf16x2(s[0], s[1]), pack_bf16x2(s[2], s[3]), pack_bf16x2(s[4], s[5]),
                     pack_bf16x2(s[6], s[7]));
    } else {
      v = make_uint4(__float_as_uint(s[0]), __float_as_uint(s[1]), __float_as_uint(s[2]),
                     __float_as_uint(s[3]));
    }
    if (r < rows_valid) *reinterpret_cast<uint4*>(base + (long long)r * ld + c) = v;
  }
}

// This thread's row of kBW values: registers -> staging row / staging row -> registers.
__device__ __forceinline__ void row_to_stage(const float (&v)[kBW], float* stage, int lane) {
#pragma unroll
  for (int j = 0; j < kBW; ++j) stage[lane * kStageStride + j] = v[j];
}
__device__ __forceinline__ void stage_to_row(const float* stage, float (&v)[kBW], int lane) {
#pragma unroll
  for (int j = 0; j < kBW; ++j) v[j] = stage[lane * kStageStride + j];
}

// Writes a row-held block through the staging buffer to global memory.
template <typename T>
__device__ __forceinline__ void store_rows(const float (&v)[kBW], float* stage, T* base, long long ld,
                                           int rows_valid, int lane) {
  row_to_stage(v, stage, lane);
  __syncwarp();
  stage_to_global<T>(stage, base, ld, rows_valid, lane);
  __syncwarp();
}

// One block of a gradient epilogue: M = beta M + g (momentum present), then
// the fp32 update source and/or the bf16 Newton-Schulz input with its squared
// norm.  `x` holds the old momentum when e.mom is set.
__device__ __forceinline__ float grad_block(const EpiDesc& e, float (&v0)[kBW],
                                            const float (&x)[kBW], long long off, int rows_valid,
                                            float* stage, int lane) {
  float sumsq = 0.f;
  if (e.mom) {
#pragma unroll
    for (int i = 0; i < kBW; ++i) v0[i] = e.a * x[i] + v0[i];
    store_rows<float>(v0, stage, e.mom + off, e.out_ld, rows_valid, lane);
  }
  if (e.out[0])
    store_rows<float>(v0, stage, static_cast<float*>(e.out[0]) + off, e.out_ld, rows_valid, lane);
  if (e.out[1]) {
    store_rows<__nv_bfloat16>(v0, stage, static_cast<__nv_bfloat16*>(e.out[1]) + off, e.out_ld,
                              rows_valid, lane);
    if (lane < rows_valid) {
#pragma unroll
      for (int i = 0; i < kBW; ++i) sumsq += v0[i] * v0[i];
    }
  }
  return sumsq;
}

// Blocks of one tile for one epilogue kind (the kind is uniform per tile, so
// each kind is its own non-inlined loop and keeps only the registers it needs).
template <int KIND>
__device__ __noinline__ float tc_epilogue_blocks(const Problem& P, int tn, uint32_t tl,
                                                    int c_begin, int c_end, long long tile_base,
                                                    int rows_valid, float eta, float scale,
                                                    float* stage, int lane, uint64_t* accf,
                                                    uint32_t accf_parity, int* status,
                                                    unsigned long long lim, bool* ok_out) {
  const EpiDesc& e = P.epi;
  const int bn = P.bn;
  constexpr bool kInBf16 = KIND == EPI_NS_STEP || (KIND == EPI_NS_POLY);
  constexpr bool kInF32 = KIND == EPI_GRAD;   // used only when e.mom is set
  constexpr int kAcc = KIND == EPI_PROJ_K ? 3 : (KIND == EPI_PROJ_Q ? 2 : 1);
  const bool has_mom = kInF32 && e.mom != nullptr;
  // the polynomial product may take G from the other TMEM accumulator buffer
  const bool x_tmem = KIND == EPI_NS_POLY && e.in_tmem;
  BlockRegs<__nv_bfloat16> gin16;
  BlockRegs<float> gin32;
  auto prefetch = [&](int c0) {
    const int gcol = tn * bn + c0;
    if (rows_valid <= 0 || gcol >= P.N || x_tmem) return;
    if constexpr (kInBf16)
      block_load(static_cast<const __nv_bfloat16*>(e.in0) + tile_base + gcol, e.out_ld,
                 rows_valid, gin16, lane);
    if constexpr (kInF32)
      if (has_mom) block_load(e.mom + tile_base + gcol, e.out_ld, rows_valid, gin32, lane);
  };
  // the first input block is requested before the accumulator is ready, then
  // inputs run one block ahead
  prefetch(c_begin);
  const bool ok = mbar_wait(accf, accf_parity, status, lim);
  *ok_out = ok;
  tc_fence_after();
  float sumsq = 0.f;
  if (!ok) return sumsq;
  for (int c0 = c_begin; c0 < c_end; c0 += kBW) {
    float v0[kBW];
    float v1[kAcc > 1 ? kBW : 1];
    float v2[kAcc > 2 ? kBW : 1];
    float x[(kInBf16 || kInF32) ? kBW : 1];
    tmem_ld16_nowait(tl + c0, v0);
    if constexpr (kAcc > 1) tmem_ld16_nowait(tl + bn + c0, v1);
    if constexpr (kAcc > 2) tmem_ld16_nowait(tl + 2 * bn + c0, v2);
    const int gcol = tn * bn + c0;
    const bool active = rows_valid > 0 && gcol < P.N;
    if constexpr (kInBf16 || kInF32) {
      if (x_tmem) {
        if constexpr (KIND == EPI_NS_POLY) {
          tmem_ld16_nowait((tl + c0) ^ 256u, x);
          tmem_wait_bind(x);
#pragma unroll
          for (int i = 0; i < kBW; ++i) x[i] *= scale * scale;
        }
      } else if (active && (kInBf16 || has_mom)) {
        if constexpr (kInBf16) block_to_stage(gin16, stage, lane);
        else block_to_stage(gin32, stage, lane);
        __syncwarp();
        stage_to_row(stage, x, lane);
        __syncwarp();
      }
    }
    if (c0 + kBW < c_end) prefetch(c0 + kBW);
    tmem_wait_bind(v0);
    if constexpr (kAcc > 1) tmem_wait_bind(v1);
    if constexpr (kAcc > 2) tmem_wait_bind(v2);
    if (!active) continue;
    const long long off = tile_base + gcol;
    if constexpr (KIND == EPI_STORE_F32) {
      store_rows<float>(v0, stage, static_cast<float*>(e.out[0]) + off, e.out_ld, rows_valid, lane);
    } else if constexpr (KIND == EPI_PROJ_Q) {
#pragma unroll
      for (int i = 0; i < kBW; ++i) v0[i] = v0[i] * sigmoid_f(v0[i]) * v1[i];
      store_rows<__nv_bfloat16>(v0, stage, static_cast<__nv_bfloat16*>(e.out[0]) + off, e.out_ld,
                                rows_valid, lane);
    } else if constexpr (KIND == EPI_PROJ_K) {
#pragma unroll
      for (int i = 0; i < kBW; ++i) {
        const float h1 = v0[i], h3 = v1[i];
        const float s = sigmoid_f(h1);
        const float sl = h1 * s;
        const float dA = -eta * v2[i];
        v0[i] = dA * h3 * s * (1.0f + h1 * (1.0f - s));   // dH1
        v1[i] = dA * sl;                                   // dH3
        v2[i] = -eta * sl * h3;                            // P
      }
      store_rows<__nv_bfloat16>(v0, stage, static_cast<__nv_bfloat16*>(e.out[0]) + off, e.out_ld,
                                rows_valid, lane);
      store_rows<__nv_bfloat16>(v1, stage, static_cast<__nv_bfloat16*>(e.out[1]) + off, e.out_ld,
                                rows_valid, lane);
      store_rows<__nv_bfloat16>(v2, stage, static_cast<__nv_bfloat16*>(e.out[2]) + off, e.out_ld,
                                rows_valid, lane);
    } else if constexpr (KIND == EPI_GRAD) {
      sumsq += grad_block(e, v0, x, off, rows_valid, stage, lane);
    } else if constexpr (KIND == EPI_OUT) {
      store_rows<__nv_bfloat16>(v0, stage, static_cast<__nv_bfloat16*>(e.out[0]) + off, e.out_ld,
                                rows_valid, lane);
    } else if constexpr (KIND == EPI_NS_GRAM) {
      const float s2 = scale * scale;
#pragma unroll
      for (int i = 0; i < kBW; ++i) v0[i] *= s2;
      store_rows<__nv_bfloat16>(v0, stage, static_cast<__nv_bfloat16*>(e.out[0]) + off, e.out_ld,
                                rows_valid, lane);
    } else if constexpr (KIND == EPI_NS_POLY) {
#pragma unroll
      for (int i = 0; i < kBW; ++i) v0[i] = e.b * x[i] + e.c * v0[i];
      store_rows<__nv_bfloat16>(v0, stage, static_cast<__nv_bfloat16*>(e.out[0]) + off, e.out_ld,
                                rows_valid, lane);
    } else if constexpr (KIND == EPI_NS_STEP) {
#pragma unroll
      for (int i = 0; i < kBW; ++i) v0[i] = scale * (e.a * x[i] + v0[i]);
      if (e.out[1])
        store_rows<float>(v0, stage, static_cast<float*>(e.out[1]) + off, e.out_ld, rows_valid,
                          lane);
      else
        store_rows<__nv_bfloat16>(v0, stage, static_cast<__nv_bfloat16*>(e.out[0]) + off,
                                  e.out_ld, rows_valid, lane);
    }
  }
  return sumsq;
}

// Epilogue of one tile on the tensor-core path (bf16 work tensors and I/O).
// Waits for the accumulator (bounded) after reading the per-row scalars.
// `warp` is 2..9; `stage` is this warp's staging buffer.  Returns this
// thread's share of the EPI_GRAD sum of squares.
__device__ __forceinline__ float tc_epilogue_tile(const Problem& P, int z, int tm, int tn,
                                                  uint32_t tmem_acc, uint64_t* accf,
                                                  uint32_t accf_parity, int* status,
                                                  unsigned long long lim, bool* ok_out,
                                                  float* stage, int warp, int lane) {
  const EpiDesc& e = P.epi;
  const int sub = warp & 3;
  constexpr int kSplit = kEpiWarps / 4;                 // column slices per lane quarter
  const int slice = (warp - 2) / 4;
  const int bn = P.bn;
  const int row0 = tm * kBM + sub * 32;                 // first row of this warp
  const int rows_valid = min(32, P.M - row0);           // may be <= 0
  const int myrow = row0 + lane;
  const int zz = e.z_div > 1 ? z / e.z_div : z;
  const long long tile_base = (long long)zz * e.out_z + (e.out_row0 + row0) * e.out_ld;
  const uint32_t tl = tmem_acc + ((uint32_t)(sub * 32) << 16);
  const int c_begin = slice * (bn / kSplit), c_end = c_begin + bn / kSplit;

  float eta = 0.f, scale = 1.f;
  if (e.kind == EPI_PROJ_K && myrow < P.M)
    eta = e.eta[(long long)zz * e.eta_z + e.eta_row0 + myrow];
  if ((e.kind == EPI_NS_GRAM || e.kind == EPI_NS_STEP || (e.kind == EPI_NS_POLY && e.in_tmem)) &&
      e.first)
    scale = ns_scale(e, zz);

  switch (e.kind) {
    case EPI_STORE_F32:
      return tc_epilogue_blocks<EPI_STORE_F32>(P, tn, tl, c_begin, c_end, tile_base, rows_valid,
                                               eta, scale, stage, lane, accf, accf_parity, status, lim, ok_out);
    case EPI_PROJ_Q:
      return tc_epilogue_blocks<EPI_PROJ_Q>(P, tn, tl, c_begin, c_end, tile_base, rows_valid, eta,
                                            scale, stage, lane, accf, accf_parity, status, lim, ok_out);
    case EPI_PROJ_K:
      return tc_epilogue_blocks<EPI_PROJ_K>(P, tn, tl, c_begin, c_end, tile_base, rows_valid, eta,
                                            scale, stage, lane, accf, accf_parity, status, lim, ok_out);
    case EPI_GRAD:
      return tc_epilogue_blocks<EPI_GRAD>(P, tn, tl, c_begin, c_end, tile_base, rows_valid, eta,
                                          scale, stage, lane, accf, accf_parity, status, lim, ok_out);
    case EPI_OUT:
      return tc_epilogue_blocks<EPI_OUT>(P, tn, tl, c_begin, c_end, tile_base, rows_valid, eta,
                                         scale, stage, lane, accf, accf_parity, status, lim, ok_out);
    case EPI_NS_GRAM:
      return tc_epilogue_blocks<EPI_NS_GRAM>(P, tn, tl, c_begin, c_end, tile_base, rows_valid,
                                             eta, scale, stage, lane, accf, accf_parity, status, lim, ok_out);
    case EPI_NS_POLY:
      return tc_epilogue_blocks<EPI_NS_POLY>(P, tn, tl, c_begin, c_end, tile_base, rows_valid,
                                             eta, scale, stage, lane, accf, accf_parity, status, lim, ok_out);
    case EPI_NS_STEP:
      return tc_epilogue_blocks<EPI_NS_STEP>(P, tn, tl, c_begin, c_end, tile_base, rows_valid,
                                             eta, scale, stage, lane, accf, accf_parity, status, lim, ok_out);
    default:
      *ok_out = mbar_wait(accf, accf_parity, status, lim);
      tc_fence_after();
      return 0.f;
  }
}

}  // namespace ttt
