// Building blocks of the tensor-core kernels: tile decoding, the shared-memory
// stage plan of a problem, and the three warp roles (TMA producer, tcgen05
// MMA issuer, TMEM epilogue) for one 128 x bn output tile.  The persistent
// grouped GEMM (gemm_umma.cu) and the cluster Newton-Schulz kernel
// (ns_cluster.cu) run these roles over their own tile sequences; the
// pipeline counters (k-step and tile iteration) carry across tiles so the
// mbarrier phases stay consistent.
#pragma once

#include "common.cuh"
#include "epilogue.cuh"

namespace ttt {

constexpr int kBM = 128;
constexpr int kBK = 64;                      // one 128-byte swizzle row of bf16
constexpr int kATileBytes = kBM * kBK * 2;   // 16 KB
constexpr int kMaxStages = 8;
constexpr int kCtrlBytes = 3072;             // barriers, TMEM slot, problem descriptors
constexpr int kProbOffset = 256;             // problem descriptors inside the control region
constexpr int kPlanOffset = 2304;            // per-problem stage plans inside the control region
constexpr int kEpiWarps = 12;           // three warps per TMEM lane quarter (column thirds)
constexpr int kGemmThreads = 64 + 32 * kEpiWarps;
constexpr int kProdLanes = 2;           // TMA-issuing threads (lane 0 of two producer warps)

struct TileCoord {
  int prob, z, tm, tn;
};

__device__ __forceinline__ TileCoord decode_tile(const Problem* probs, int nprob, int t) {
  int p = 0;
#pragma unroll 1
  for (int i = 1; i < nprob; ++i)
    if (t >= probs[i].tile_start) p = i;
  const Problem& P = probs[p];
  int local = t - P.tile_start;
  TileCoord c;
  c.prob = p;
  c.tn = local % P.tiles_n;
  local /= P.tiles_n;
  c.tm = local % P.tiles_m;
  c.z = local / P.tiles_m;
  return c;
}

// Accumulator groups of a problem.  Accumulators that share one A tile form a
// group; a group's k-steps stream A plus the group's B tiles through one
// pipeline stage (A at offset 0, B tiles after it), and the groups run one
// after the other, so a stage never holds more than one A tile.  A group
// whose B tiles are of the same major-ness and total N <= 256 is issued as a
// single MMA (TMEM columns of its accumulators are adjacent).
struct SmemPlan {
  int kd;               // 64-deep K steps per stage (1 or 2)
  int ngroups;
  int g_first[kMaxAcc], g_count[kMaxAcc], g_merged[kMaxAcc];
  uint32_t g_bytes[kMaxAcc];
  uint32_t max_bytes;
};

__device__ __forceinline__ void plan_problem(const Problem& P, SmemPlan& sp) {
  sp.kd = P.kd == 2 ? 2 : 1;
  sp.ngroups = 0;
  sp.max_bytes = 0;
  int j = 0;
#pragma unroll 1
  while (j < P.nacc) {
    int cnt = 1;
    while (j + cnt < P.nacc && ((P.a_shared >> (j + cnt)) & 1)) ++cnt;
    bool same = true;
    for (int i = 1; i < cnt; ++i) same = same && P.b[j + i].mn_major == P.b[j].mn_major;
    const int g = sp.ngroups++;
    sp.g_first[g] = j;
    sp.g_count[g] = cnt;
    sp.g_merged[g] = cnt > 1 && same && cnt * P.bn <= 256;
    sp.g_bytes[g] = sp.kd * (kATileBytes + cnt * P.bn * kBK * 2);
    sp.max_bytes = max(sp.max_bytes, sp.g_bytes[g]);
    j += cnt;
  }
}

// Issue the TMA boxes of one operand tile (rows x 64 of K) for k-step ks.
__device__ __forceinline__ void load_operand(const CUtensorMap* maps, const OpDesc& op,
                                             uint8_t* dst, int rows, int mn0, int ks, int z,
                                             uint64_t* bar) {
  const int zz = op.z_div > 1 ? z / op.z_div : z;
  const CUtensorMap* map = &maps[op.map];
  if (!op.mn_major) {
    tma_load_2d(dst, map, op.inner_base + ks * kBK, op.outer_base + zz * op.z_outer + mn0, bar);
  } else {
    for (int i = 0; i < rows / 64; ++i)
      tma_load_2d(dst + i * 8192, map, op.inner_base + mn0 + i * 64,
                  op.outer_base + zz * op.z_outer + ks * kBK, bar);
  }
}

// Descriptor of an operand tile at `base` for kd K steps per stage: MN-major
// blocks of 64 M/N columns are 8 KB x kd apart.
__device__ __forceinline__ uint64_t operand_desc_kd(uint32_t base, int mn_major, int kd) {
  return mn_major ? smem_desc_sw128(base, 8192 * kd, 1024) : smem_desc_sw128(base, 16, 1024);
}

__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int mn_major, int kk) {
  // K-major: a 16-element K slice starts 32 bytes further along the row.
  // MN-major: it starts 16 K-rows (2 KB) further down.
  return mn_major ? smem_desc_sw128(base + kk * 2048, 8192, 1024)
                  : smem_desc_sw128(base + kk * 32, 16, 1024);
}

// ---------------------------------------------------------------- roles

// Precomputed TMA coordinates of one operand tile: the k-step ks box(es) are
// at (x0 + ks * dx, y0 + ks * dy) and, for MN-major operands, nbox boxes of 64
// M/N columns 64 apart along x.
//
// With kd = 2 a stage covers 128 of K: a K-major tile is two boxes of 64 K
// columns, one after the other (`kbytes` apart), and an MN-major tile's boxes
// are 128 K rows deep (`bbytes` = 16 KB apart instead of 8 KB).
struct OpCoords {
  const CUtensorMap* map;
  const CUtensorMap* map3;   // MN-major: the whole stage tile as one 3-D box, or NULL
  int x0, y0, dx, dy, nbox, kd, kbytes, bbytes;
};

__device__ __forceinline__ OpCoords op_coords(const CUtensorMap* maps, const OpDesc& op, int rows,
                                              int mn0, int z, int kd) {
  const int zz = op.z_div > 1 ? z / op.z_div : z;
  OpCoords c;
  c.map = &maps[op.map];
  c.map3 = (op.mn_major && op.map3 >= 0) ? &maps[op.map3] : nullptr;
  c.kd = kd;
  c.kbytes = rows * kBK * 2;
  c.bbytes = 8192 * kd;
  if (!op.mn_major) {
    c.x0 = op.inner_base;
    c.y0 = op.outer_base + zz * op.z_outer + mn0;
    c.dx = kBK * kd;
    c.dy = 0;
    c.nbox = 1;
  } else {
    c.x0 = op.inner_base + mn0;
    c.y0 = op.outer_base + zz * op.z_outer;
    c.dx = 0;
    c.dy = kBK * kd;
    c.nbox = rows / 64;
  }
  return c;
}

__device__ __forceinline__ void issue_op(const OpCoords& c, uint8_t* dst, int ks, uint64_t* bar) {
  const int x = c.x0 + ks * c.dx, y = c.y0 + ks * c.dy;
  if (c.dy == 0) {   // K-major: kd boxes of 64 K columns
    tma_load_2d(dst, c.map, x, y, bar);
    if (c.kd == 2) tma_load_2d(dst + c.kbytes, c.map, x + kBK, y, bar);
  } else if (c.map3) {   // blocks of 64 columns land c.bbytes apart, as below
    tma_load_3d(dst, c.map3, 0, y, x >> 6, bar);
  } else {
    for (int i = 0; i < c.nbox; ++i) tma_load_2d(dst + i * c.bbytes, c.map, x + i * 64, y, bar);
  }
}

// TMA producer (one thread): streams every (group, k-step) of one tile through
// the ring.  `s`/`ph` are the ring position carried across tiles.  Per-operand
// coordinates live in scalars (no runtime-indexed local arrays in the loop).
//
// Several lanes of the producer warp may share the work: every lane walks
// every ring entry (`e` counts them across tiles) and issues those with
// e % nlanes == lane, so consecutive entries are in flight from different
// threads (one thread alone cannot issue TMA fast enough).  nlanes is 1 or 2.
static __device__ __forceinline__ bool produce_tile(const CUtensorMap* maps, const Problem& P,
                                             const SmemPlan& sp, const TileCoord& tc,
                                             uint8_t* tiles, uint32_t stage_bytes, int nstages,
                                             uint64_t* full, uint64_t* empty, int& s,
                                             uint32_t& ph, int lane, int nlanes, int& e,
                                             int* status, unsigned long long lim) {
  const int kd = sp.kd;
  const int nk = P.K / (kBK * kd);
  const uint32_t a_bytes = kATileBytes * kd;
  const uint32_t b_step = P.bn * kBK * 2 * kd;
  if (lane == 0 && P.epi.kind == EPI_GRAD && P.epi.mom) {
    // the epilogue reads this tile's momentum rows: bring them into L2 while
    // the main loop runs (whole rows, contiguous)
    const EpiDesc& e = P.epi;
    const int zz = e.z_div > 1 ? tc.z / e.z_div : tc.z;
    const int row0 = tc.tm * kBM;
    const int rows = min(kBM, P.M - row0);
    if (rows > 0) {
      const char* base = reinterpret_cast<const char*>(
          e.mom + (long long)zz * e.out_z + (e.out_row0 + row0) * e.out_ld);
      const uint32_t bytes = (uint32_t)rows * (uint32_t)e.out_ld * 4u;
      if ((reinterpret_cast<uintptr_t>(base) & 15) == 0 && (bytes & 15) == 0)
        for (uint32_t o = 0; o < bytes; o += 16384u)
          prefetch_l2_bulk(base + o, min(16384u, bytes - o));
    }
  }
  for (int g = 0; g < sp.ngroups; ++g) {
    const int j0 = sp.g_first[g], cnt = sp.g_count[g];
    const uint32_t bytes = sp.g_bytes[g];
    const OpCoords ca = op_coords(maps, P.a[j0], kBM, tc.tm * kBM, tc.z, kd);
    const OpCoords cb0 = op_coords(maps, P.b[j0], P.bn, tc.tn * P.bn, tc.z, kd);
    OpCoords cb1 = cb0, cb2 = cb0;
    if (cnt > 1) cb1 = op_coords(maps, P.b[j0 + 1], P.bn, tc.tn * P.bn, tc.z, kd);
    if (cnt > 2) cb2 = op_coords(maps, P.b[j0 + 2], P.bn, tc.tn * P.bn, tc.z, kd);
    for (int ks = 0; ks < nk; ++ks, ++e) {
      if ((e & (nlanes - 1)) == lane) {
        if (!mbar_wait(&empty[s], ph ^ 1, status, lim)) return false;
        mbar_arrive_expect_tx(&full[s], bytes);
        uint8_t* st = tiles + s * stage_bytes;
        issue_op(ca, st, ks, &full[s]);
        issue_op(cb0, st + a_bytes, ks, &full[s]);
        if (cnt > 1) issue_op(cb1, st + a_bytes + b_step, ks, &full[s]);
        if (cnt > 2) issue_op(cb2, st + a_bytes + 2 * b_step, ks, &full[s]);
      }
      if (++s == nstages) {
        s = 0;
        ph ^= 1;
      }
    }
  }
  return true;
}

// Waits (bounded) until the copies of the last stages issued have landed:
// the ring position (s, ph) is one past the last stage filled.
__device__ __forceinline__ void drain_producer(uint64_t* full, int nstages, int s, uint32_t ph,
                                               int filled, int* status, unsigned long long lim) {
  for (int k = 0; k < nstages && k < filled; ++k) {
    if (--s < 0) {
      s = nstages - 1;
      ph ^= 1;
    }
    mbar_wait(&full[s], ph, status, lim);
  }
}

// MMA issue loop, run by a whole warp (one elected lane issues each
// tcgen05 operation): accumulates one tile into TMEM at column tmem_acc
// (accumulator j at tmem_acc + j * bn).  Descriptors are scalars built once
// per group; no runtime-indexed arrays in the k-step loop.
static __device__ __forceinline__ bool mma_tile(const Problem& P, const SmemPlan& sp,
                                         uint32_t tiles_saddr, uint32_t stage_bytes, int nstages,
                                         uint64_t* full, uint64_t* empty, uint32_t tmem_acc,
                                         int& s, uint32_t& ph, int* status,
                                         unsigned long long lim) {
  const int kd = sp.kd;
  const int nk = P.K / (kBK * kd);
  const uint32_t a_bytes = kATileBytes * kd;
  const uint32_t b_step = P.bn * kBK * 2 * kd;
  for (int g = 0; g < sp.ngroups; ++g) {
    const int j0 = sp.g_first[g], cnt = sp.g_count[g];
    const bool merged = sp.g_merged[g];
    const int nmma = merged ? 1 : cnt;
    const int a_mn = P.a[j0].mn_major;
    const int bmn0 = P.b[j0].mn_major;
    const int bmn1 = cnt > 1 ? P.b[j0 + 1].mn_major : bmn0;
    const int bmn2 = cnt > 2 ? P.b[j0 + 2].mn_major : bmn0;
    const uint32_t n0 = (merged ? cnt : 1) * P.bn;
    const uint32_t id0 = idesc_bf16_f32(n0, a_mn, bmn0);
    const uint32_t id1 = idesc_bf16_f32(P.bn, a_mn, bmn1);
    const uint32_t id2 = idesc_bf16_f32(P.bn, a_mn, bmn2);
    const uint32_t d0 = tmem_acc + j0 * P.bn, d1 = d0 + P.bn, d2 = d0 + 2 * P.bn;
    const uint32_t bo0 = a_bytes, bo1 = a_bytes + b_step, bo2 = a_bytes + 2 * b_step;
    // Stage-0 descriptors, advanced by adding byte offsets / 16 to the start
    // address field (shared addresses < 256 KB: the 14-bit field never
    // carries); a 16-deep K slice is 32 B further (K-major) or 2 KB (MN-major),
    // and with kd = 2 the second 64 of K is one K-major tile (rows x 128 B)
    // further or 8 KB deeper into the MN-major blocks (16 KB apart).
    // Keeping this loop short keeps the tensor core fed.
    const uint64_t a0 = operand_desc_kd(tiles_saddr, a_mn, kd);
    const uint64_t b0 = operand_desc_kd(tiles_saddr + bo0, bmn0, kd);
    const uint64_t b1 = operand_desc_kd(tiles_saddr + bo1, bmn1, kd);
    const uint64_t b2 = operand_desc_kd(tiles_saddr + bo2, bmn2, kd);
    const uint32_t ka = a_mn ? 128 : 2, kb0 = bmn0 ? 128 : 2, kb1 = bmn1 ? 128 : 2,
                   kb2 = bmn2 ? 128 : 2;
    const uint32_t ha = a_mn ? 512 : kBM * 8, hb0 = bmn0 ? 512 : P.bn * 8;   // next 64 of K
    const uint32_t stage16 = stage_bytes >> 4;
    for (int ks = 0; ks < nk; ++ks) {
      if (!mbar_wait_w(&full[s], ph, status, lim)) return false;
      tc_fence_after();
      const uint64_t so = (uint64_t)(s * stage16);
      for (int kh = 0; kh < kd; ++kh) {
        const uint64_t ah = a0 + so + kh * ha, bh = b0 + so + kh * hb0;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          const uint32_t acc = (ks | kh | kk) != 0;
          const uint64_t ad = ah + kk * ka;
          umma_bf16_w(d0, ad, bh + kk * kb0, id0, acc);
          if (nmma > 1) umma_bf16_w(d1, ad, b1 + so + kk * kb1, id1, acc);
          if (nmma > 2) umma_bf16_w(d2, ad, b2 + so + kk * kb2, id2, acc);
        }
      }
      umma_commit_w(&empty[s]);
      if (++s == nstages) {
        s = 0;
        ph ^= 1;
      }
    }
  }
  return true;
}

}  // namespace ttt
