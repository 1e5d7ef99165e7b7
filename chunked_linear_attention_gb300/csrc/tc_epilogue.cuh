// Tensor-core epilogue: drains one tile's TMEM accumulators and applies the
// fused epilogue of epilogue.cuh, with memory traffic shaped for the GPU:
//
//   * each epilogue warp owns 32 rows (its TMEM lane quarter) and about a
//     third of the tile's columns (three warps per lane quarter keep enough
//     loads and stores in flight), processed in blocks of 16 columns;
//   * per-row scalars (eta, the Newton-Schulz scale) are read once per tile,
//     and the first input block is requested, before waiting for the
//     accumulator;
//   * where rows are 32-byte aligned (the usual case), every lane moves its
//     own row segment of a block (32 bytes of bf16, 64 of fp32) with 32-byte
//     global loads and stores straight from registers: one instruction per 32
//     bytes instead of a pass through shared memory;
//   * otherwise rows move between a lane's registers and coalesced 16-byte
//     global accesses through a 2 KB per-warp staging block in shared memory,
//     with an XOR swizzle that keeps both the row-wise and the coalesced
//     passes free of bank conflicts.
#pragma once

#include "common.cuh"
#include "epilogue.cuh"
#include "umma_core.cuh"

namespace ttt {

constexpr int kStageBytesPerWarp = 2048;                 // 32 rows x 64 bytes
constexpr int kStageFloats = kStageBytesPerWarp / 4;     // per-warp stride in floats
constexpr int kStagingBytes = kEpiWarps * kStageBytesPerWarp;
static_assert(kStagingBytes % 1024 == 0, "keeps the stage ring 1 KB aligned");

// Byte offset of 16-byte unit u of row r in a 32-row staging block whose rows
// are RB bytes (RB = 32 or 64).  The XOR spreads the 8 lanes of one shared
// memory phase over all banks, for the row-wise and the coalesced pattern.
template <int RB>
__device__ __forceinline__ uint32_t stage_off(int r, int u) {
  static_assert(RB == 32 || RB == 64, "row bytes");
  if constexpr (RB == 32) return (uint32_t)(r * 32 + ((u ^ ((r >> 2) & 1)) << 4));
  else return (uint32_t)(r * 64 + ((u ^ ((r >> 1) & 3)) << 4));
}

template <int BW>
__device__ __forceinline__ void tmem_load_block(uint32_t taddr, float (&v)[BW]) {
  static_assert(BW == 16 || BW == 32, "block width");
  if constexpr (BW == 16) tmem_ld16_nowait(taddr, v);
  else tmem_ld32(taddr, v);
}
template <int BW>
__device__ __forceinline__ void tmem_wait_block(float (&v)[BW]) {
  if constexpr (BW == 16) tmem_wait_bind(v);
  else tmem_wait32(v);
}

// 16-byte units of a 32-row block of T, BW columns, held as coalesced
// registers: unit i of this lane is unit (i * 32 + lane) of the block.
template <typename T, int BW>
struct BlockIn {
  static constexpr int kRB = BW * (int)sizeof(T);   // bytes per row
  static constexpr int kU = kRB / 16;               // units per row
  uint4 w[kU];
};

// Global -> registers (rows >= rows_valid read as zero).  V8 (32-byte
// aligned rows): this lane's own row segment, in order; else coalesced
// 16-byte units for block_to_row.
template <typename T, int BW, bool V8>
__device__ __forceinline__ void block_fetch(const T* base, long long ld, int rows_valid,
                                            BlockIn<T, BW>& g, int lane) {
  constexpr int U = BlockIn<T, BW>::kU;
  static_assert(U % 2 == 0, "whole 32-byte row segments");
  if constexpr (V8) {
    const char* rowp = reinterpret_cast<const char*>(base + (long long)lane * ld);
#pragma unroll
    for (int h = 0; h < U / 2; ++h) {
      uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (lane < rows_valid) ldg256(rowp + 32 * h, w);
      g.w[2 * h] = make_uint4(w[0], w[1], w[2], w[3]);
      g.w[2 * h + 1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
    return;
  }
#pragma unroll
  for (int i = 0; i < U; ++i) {
    const int idx = i * 32 + lane, r = idx / U, u = idx % U;
    g.w[i] = r < rows_valid ? *reinterpret_cast<const uint4*>(
                                  reinterpret_cast<const char*>(base + (long long)r * ld) + u * 16)
                            : make_uint4(0, 0, 0, 0);
  }
}

// Fetched block -> this lane's row (as fp32); through the staging block
// unless it was fetched lane-per-row (V8).
template <typename T, int BW, bool V8>
__device__ __forceinline__ void block_to_row(const BlockIn<T, BW>& g, uint32_t st, float (&x)[BW],
                                             int lane) {
  constexpr int RB = BlockIn<T, BW>::kRB, U = BlockIn<T, BW>::kU;
  if constexpr (!V8) {
#pragma unroll
    for (int i = 0; i < U; ++i) {
      const int idx = i * 32 + lane;
      sts128(st + stage_off<RB>(idx / U, idx % U), g.w[i]);
    }
    __syncwarp();
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    uint4 w;
    if constexpr (V8) w = g.w[u];
    else w = lds128(st + stage_off<RB>(lane, u));
    if constexpr (sizeof(T) == 2) {
      x[8 * u + 0] = bf16lo(w.x); x[8 * u + 1] = bf16hi(w.x);
      x[8 * u + 2] = bf16lo(w.y); x[8 * u + 3] = bf16hi(w.y);
      x[8 * u + 4] = bf16lo(w.z); x[8 * u + 5] = bf16hi(w.z);
      x[8 * u + 6] = bf16lo(w.w); x[8 * u + 7] = bf16hi(w.w);
    } else {
      x[4 * u + 0] = __uint_as_float(w.x); x[4 * u + 1] = __uint_as_float(w.y);
      x[4 * u + 2] = __uint_as_float(w.z); x[4 * u + 3] = __uint_as_float(w.w);
    }
  }
  if constexpr (!V8) __syncwarp();
}

// This lane's row (BW values) -> global as T: with 32-byte stores of the
// lane's own row where rows are 32-byte aligned (V8), else through the
// staging block as coalesced 16-byte stores.
template <typename T, int BW, bool V8>
__device__ __forceinline__ void store_rows(const float (&v)[BW], uint32_t st, T* base, long long ld,
                                           int rows_valid, int lane) {
  constexpr int RB = BlockIn<T, BW>::kRB, U = BlockIn<T, BW>::kU;
  if constexpr (V8) {
    if (lane < rows_valid) {
      char* rowp = reinterpret_cast<char*>(base + (long long)lane * ld);
#pragma unroll
      for (int h = 0; h < RB / 32; ++h) {
        uint32_t w[8];
        if constexpr (sizeof(T) == 2) {
#pragma unroll
          for (int i = 0; i < 8; ++i) w[i] = pack_bf16x2(v[16 * h + 2 * i], v[16 * h + 2 * i + 1]);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) w[i] = __float_as_uint(v[8 * h + i]);
        }
        stg256(rowp + 32 * h, w);
      }
    }
    return;
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    uint4 w;
    if constexpr (sizeof(T) == 2) {
      w = make_uint4(pack_bf16x2(v[8 * u], v[8 * u + 1]), pack_bf16x2(v[8 * u + 2], v[8 * u + 3]),
                     pack_bf16x2(v[8 * u + 4], v[8 * u + 5]),
                     pack_bf16x2(v[8 * u + 6], v[8 * u + 7]));
    } else {
      w = make_uint4(__float_as_uint(v[4 * u]), __float_as_uint(v[4 * u + 1]),
                     __float_as_uint(v[4 * u + 2]), __float_as_uint(v[4 * u + 3]));
    }
    sts128(st + stage_off<RB>(lane, u), w);
  }
  __syncwarp();
#pragma unroll
  for (int i = 0; i < U; ++i) {
    const int idx = i * 32 + lane, r = idx / U, u = idx % U;
    const uint4 w = lds128(st + stage_off<RB>(r, u));
    if (r < rows_valid)
      *reinterpret_cast<uint4*>(reinterpret_cast<char*>(base + (long long)r * ld) + u * 16) = w;
  }
  __syncwarp();
}

// Columns per block for each epilogue kind: 16 where three accumulators or
// fp32 rows must fit the registers and the 2 KB staging block.
template <int KIND>
constexpr int epi_block_width() {
  return (kEpiWarps == 8 && (KIND == EPI_PROJ_Q || KIND == EPI_OUT)) ? 32 : 16;
}

// One block of a gradient epilogue: M = beta M + g (momentum present), then
// the fp32 update source and/or the bf16 Newton-Schulz input with its squared
// norm.  `x` holds the old momentum when e.mom is set.
template <bool V8>
__device__ __forceinline__ float grad_block(const EpiDesc& e, float (&v0)[16], const float (&x)[16],
                                            long long off, int rows_valid, uint32_t st, int lane) {
  float sumsq = 0.f;
  if (e.mom) {
#pragma unroll
    for (int i = 0; i < 16; ++i) v0[i] = e.a * x[i] + v0[i];
    store_rows<float, 16, V8>(v0, st, e.mom + off, e.out_ld, rows_valid, lane);
  }
  if (e.out[0])
    store_rows<float, 16, V8>(v0, st, static_cast<float*>(e.out[0]) + off, e.out_ld, rows_valid, lane);
  if (e.out[1]) {
    store_rows<__nv_bfloat16, 16, V8>(v0, st, static_cast<__nv_bfloat16*>(e.out[1]) + off, e.out_ld,
                                  rows_valid, lane);
    if (lane < rows_valid) {
#pragma unroll
      for (int i = 0; i < 16; ++i) sumsq += v0[i] * v0[i];
    }
  }
  return sumsq;
}

// Gradient epilogue with momentum on the lane-per-row path, for a warp slice
// of at most four 16-column blocks: the old momentum of every block is loaded
// before the accumulator wait, so the loads overlap the main loop (a tile's
// 2048-deep K loop takes ~20 us) instead of following it one block at a time.
__device__ __forceinline__ float grad_blocks_prefetched(const Problem& P, int tn, uint32_t tl,
                                                        int c_begin, int c_end,
                                                        long long tile_base, int rows_valid,
                                                        uint32_t st, int lane, uint64_t* accf,
                                                        uint32_t accf_parity, int* status,
                                                        unsigned long long lim, bool* ok_out) {
  const EpiDesc& e = P.epi;
  const int bn = P.bn;
  float m[4][16];
#pragma unroll
  for (int bi = 0; bi < 4; ++bi) {
    const int c0 = c_begin + 16 * bi;
    const int gcol = tn * bn + c0;
    BlockIn<float, 16> g;
    if (c0 < c_end && rows_valid > 0 && gcol < P.N) {
      block_fetch<float, 16, true>(e.mom + tile_base + gcol, e.out_ld, rows_valid, g, lane);
    } else {
#pragma unroll
      for (int u = 0; u < BlockIn<float, 16>::kU; ++u) g.w[u] = make_uint4(0, 0, 0, 0);
    }
    block_to_row<float, 16, true>(g, st, m[bi], lane);
  }
  const bool ok = mbar_wait(accf, accf_parity, status, lim);
  *ok_out = ok;
  tc_fence_after();
  float sumsq = 0.f;
  if (!ok) return sumsq;
#pragma unroll
  for (int bi = 0; bi < 4; ++bi) {
    const int c0 = c_begin + 16 * bi;
    if (c0 >= c_end) break;
    float v0[16];
    tmem_load_block<16>(tl + c0, v0);
    tmem_wait_block<16>(v0);
    const int gcol = tn * bn + c0;
    if (rows_valid <= 0 || gcol >= P.N) continue;
    sumsq += grad_block<true>(e, v0, m[bi], tile_base + gcol, rows_valid, st, lane);
  }
  return sumsq;
}

// Blocks of one tile for one epilogue kind (the kind is uniform per tile, so
// each kind is its own non-inlined loop and keeps only the registers it needs).
// V8: every row the problem touches is 32-byte aligned (decided on the host).
// Waits (bounded) for the accumulator after requesting the first input block.
template <int KIND, bool V8>
__device__ __noinline__ float tc_epilogue_blocks(const Problem& P, int tn, uint32_t tl,
                                                    int c_begin, int c_end, long long tile_base,
                                                    int rows_valid, float eta, float scale,
                                                    float* stage, int lane, uint64_t* accf,
                                                    uint32_t accf_parity, int* status,
                                                    unsigned long long lim, bool* ok_out) {
  constexpr int BW = epi_block_width<KIND>();
  const EpiDesc& e = P.epi;
  const int bn = P.bn;
  const uint32_t st = smem_u32(stage);
  constexpr bool kInBf16 = KIND == EPI_NS_STEP || KIND == EPI_NS_POLY;
  constexpr bool kInF32 = KIND == EPI_GRAD;   // used only when e.mom is set
  constexpr int kAcc = KIND == EPI_PROJ_K ? 3 : (KIND == EPI_PROJ_Q ? 2 : 1);
  const bool has_mom = kInF32 && e.mom != nullptr;
  // the polynomial product may take G from the other TMEM accumulator buffer
  const bool x_tmem = KIND == EPI_NS_POLY && e.in_tmem;
  if constexpr (KIND == EPI_GRAD && V8 && BW == 16) {
    if (has_mom && c_end - c_begin <= 64)
      return grad_blocks_prefetched(P, tn, tl, c_begin, c_end, tile_base, rows_valid, st, lane,
                                    accf, accf_parity, status, lim, ok_out);
  }
  BlockIn<__nv_bfloat16, BW> gin16;
  BlockIn<float, BW> gin32;
  auto prefetch = [&](int c0) {
    const int gcol = tn * bn + c0;
    if (rows_valid <= 0 || gcol >= P.N || x_tmem) return;
    if constexpr (kInBf16)
      block_fetch<__nv_bfloat16, BW, V8>(static_cast<const __nv_bfloat16*>(e.in0) + tile_base + gcol,
                                         e.out_ld, rows_valid, gin16, lane);
    if constexpr (kInF32)
      if (has_mom)
        block_fetch<float, BW, V8>(e.mom + tile_base + gcol, e.out_ld, rows_valid, gin32, lane);
  };
  // the first input block is requested before the accumulator is ready, then
  // inputs run one block ahead
  prefetch(c_begin);
  const bool ok = mbar_wait(accf, accf_parity, status, lim);
  *ok_out = ok;
  tc_fence_after();
  float sumsq = 0.f;
  if (!ok) return sumsq;
  for (int c0 = c_begin; c0 < c_end; c0 += BW) {
    float v0[BW];
    float v1[kAcc > 1 ? BW : 1];
    float v2[kAcc > 2 ? BW : 1];
    float x[(kInBf16 || kInF32) ? BW : 1];
    tmem_load_block<BW>(tl + c0, v0);
    if constexpr (kAcc > 1) tmem_load_block<BW>(tl + bn + c0, v1);
    if constexpr (kAcc > 2) tmem_load_block<BW>(tl + 2 * bn + c0, v2);
    const int gcol = tn * bn + c0;
    const bool active = rows_valid > 0 && gcol < P.N;
    if constexpr (kInBf16 || kInF32) {
      if (x_tmem) {
        if constexpr (KIND == EPI_NS_POLY) {
          tmem_load_block<BW>((tl + c0) ^ 256u, x);
          tmem_wait_block<BW>(x);
#pragma unroll
          for (int i = 0; i < BW; ++i) x[i] *= scale * scale;
        }
      } else if (active && (kInBf16 || has_mom)) {
        if constexpr (kInBf16) block_to_row<__nv_bfloat16, BW, V8>(gin16, st, x, lane);
        else block_to_row<float, BW, V8>(gin32, st, x, lane);
      }
    }
    if (c0 + BW < c_end) prefetch(c0 + BW);
    tmem_wait_block<BW>(v0);
    if constexpr (kAcc > 1) tmem_wait_block<BW>(v1);
    if constexpr (kAcc > 2) tmem_wait_block<BW>(v2);
    if (!active) continue;
    const long long off = tile_base + gcol;
    if constexpr (KIND == EPI_STORE_F32) {
      store_rows<float, BW, V8>(v0, st, static_cast<float*>(e.out[0]) + off, e.out_ld, rows_valid,
                            lane);
    } else if constexpr (KIND == EPI_PROJ_Q) {
      // optional row factor: -eta of the row (e.eta set) or the constant e.a
      const float f = e.eta ? -eta : (e.a != 0.f ? e.a : 1.0f);
#pragma unroll
      for (int i = 0; i < BW; ++i) v0[i] = v0[i] * sigmoid_f(v0[i]) * v1[i] * f;
      store_rows<__nv_bfloat16, BW, V8>(v0, st, static_cast<__nv_bfloat16*>(e.out[0]) + off, e.out_ld,
                                    rows_valid, lane);
    } else if constexpr (KIND == EPI_PROJ_K) {
#pragma unroll
      for (int i = 0; i < BW; ++i) {
        const float h1 = v0[i], h3 = v1[i];
        const float s = sigmoid_f(h1);
        const float sl = h1 * s;
        const float dA = -eta * v2[i];
        v0[i] = dA * h3 * s * (1.0f + h1 * (1.0f - s));   // dH1
        v1[i] = dA * sl;                                   // dH3
        v2[i] = -eta * sl * h3;                            // P
      }
      store_rows<__nv_bfloat16, BW, V8>(v0, st, static_cast<__nv_bfloat16*>(e.out[0]) + off, e.out_ld,
                                    rows_valid, lane);
      store_rows<__nv_bfloat16, BW, V8>(v1, st, static_cast<__nv_bfloat16*>(e.out[1]) + off, e.out_ld,
                                    rows_valid, lane);
      store_rows<__nv_bfloat16, BW, V8>(v2, st, static_cast<__nv_bfloat16*>(e.out[2]) + off, e.out_ld,
                                    rows_valid, lane);
    } else if constexpr (KIND == EPI_GRAD) {
      sumsq += grad_block<V8>(e, v0, x, off, rows_valid, st, lane);
    } else if constexpr (KIND == EPI_OUT) {
      store_rows<__nv_bfloat16, BW, V8>(v0, st, static_cast<__nv_bfloat16*>(e.out[0]) + off, e.out_ld,
                                    rows_valid, lane);
    } else if constexpr (KIND == EPI_NS_GRAM) {
      const float s2 = scale * scale;
#pragma unroll
      for (int i = 0; i < BW; ++i) v0[i] *= s2;
      store_rows<__nv_bfloat16, BW, V8>(v0, st, static_cast<__nv_bfloat16*>(e.out[0]) + off, e.out_ld,
                                    rows_valid, lane);
    } else if constexpr (KIND == EPI_NS_POLY) {
#pragma unroll
      for (int i = 0; i < BW; ++i) v0[i] = e.b * x[i] + e.c * v0[i];
      store_rows<__nv_bfloat16, BW, V8>(v0, st, static_cast<__nv_bfloat16*>(e.out[0]) + off, e.out_ld,
                                    rows_valid, lane);
    } else if constexpr (KIND == EPI_NS_STEP) {
#pragma unroll
      for (int i = 0; i < BW; ++i) v0[i] = scale * (e.a * x[i] + v0[i]);
      if (e.out[1])
        store_rows<float, BW, V8>(v0, st, static_cast<float*>(e.out[1]) + off, e.out_ld, rows_valid,
                              lane);
      else
        store_rows<__nv_bfloat16, BW, V8>(v0, st, static_cast<__nv_bfloat16*>(e.out[0]) + off,
                                      e.out_ld, rows_valid, lane);
    }
  }
  return sumsq;
}

// Epilogue of one tile on the tensor-core path (bf16 work tensors and I/O).
// `warp` is the hardware warp index (its TMEM lane quarter is warp % 4), `ew`
// the epilogue warp index 0 .. kEpiWarps-1 (consecutive warps: every lane
// quarter gets kEpiWarps / 4 column slices); `stage` is this warp's staging
// block.  Sets *ok_out to the outcome of the (bounded) accumulator wait.
// Returns this thread's share of the EPI_GRAD sum of squares.  V8: every
// problem of the launch has 32-byte aligned rows (EpiDesc::rows32).
template <bool V8>
__device__ __forceinline__ float tc_epilogue_tile(const Problem& P, int z, int tm, int tn,
                                                  uint32_t tmem_acc, uint64_t* accf,
                                                  uint32_t accf_parity, int* status,
                                                  unsigned long long lim, bool* ok_out,
                                                  float* stage, int warp, int ew, int lane) {
  const EpiDesc& e = P.epi;
  const int sub = warp & 3;
  constexpr int kSplit = kEpiWarps / 4;                 // column slices per lane quarter
  const int slice = ew / 4;
  const int bn = P.bn;
  const int row0 = tm * kBM + sub * 32;                 // first row of this warp
  const int rows_valid = min(32, P.M - row0);           // may be <= 0
  const int myrow = row0 + lane;
  const int zz = e.z_div > 1 ? z / e.z_div : z;
  const long long tile_base = (long long)zz * e.out_z + (e.out_row0 + row0) * e.out_ld;
  const uint32_t tl = tmem_acc + ((uint32_t)(sub * 32) << 16);
  // the tile's 16-column blocks are shared out in contiguous runs
  const int nblk = bn / 16;
  const int c_begin = 16 * (slice * nblk / kSplit), c_end = 16 * ((slice + 1) * nblk / kSplit);

  float eta = 0.f, scale = 1.f;
  if ((e.kind == EPI_PROJ_K || (e.kind == EPI_PROJ_Q && e.eta)) && myrow < P.M)
    eta = e.eta[(long long)zz * e.eta_z + e.eta_row0 + myrow];
  if ((e.kind == EPI_NS_GRAM || e.kind == EPI_NS_STEP || (e.kind == EPI_NS_POLY && e.in_tmem)) &&
      e.first)
    scale = ns_scale(e, zz);

#define TTT_EPI_CASE(K)                                                                       \
  case K:                                                                                     \
    return tc_epilogue_blocks<K, V8>(P, tn, tl, c_begin, c_end, tile_base, rows_valid, eta,   \
                                     scale, stage, lane, accf, accf_parity, status, lim, ok_out);
  switch (e.kind) {
    TTT_EPI_CASE(EPI_STORE_F32)
    TTT_EPI_CASE(EPI_PROJ_Q)
    TTT_EPI_CASE(EPI_PROJ_K)
    TTT_EPI_CASE(EPI_GRAD)
    TTT_EPI_CASE(EPI_OUT)
    TTT_EPI_CASE(EPI_NS_GRAM)
    TTT_EPI_CASE(EPI_NS_POLY)
    TTT_EPI_CASE(EPI_NS_STEP)
    default:
      *ok_out = mbar_wait(accf, accf_parity, status, lim);
      tc_fence_after();
      return 0.f;
  }
#undef TTT_EPI_CASE
}

}  // namespace ttt
