// Muon for square fast-weight matrices of order d = 128 R (R = 1..4): every
// Newton-Schulz step (eq 6 of the LaCT notes; the quintic of the Muon write-up)
// and the final W <- L2-Normalize(W - U) (eq 5) in one launch, one
// thread-block cluster of 2 R CTAs per matrix.
//
// CTA (r, h) of a cluster (rank h R + r) computes the 128 x d/2 block of row
// panel r and column half h of every product:
//     G  = X X^T              (first step: scaled by 1/(|M|_F + eps)^2)
//     P  = a I + b G + c G G
//     X' = P X                (first step: scaled by 1/(|M|_F + eps))
// Its A operand is the whole 128-row panel r of the previous product, kept in
// shared memory (128-byte swizzle, K-major): each epilogue writes its own half
// of the panel, and a bulk shared-to-shared copy sends that half to the
// partner (r, 1-h), completing on the partner's panel barrier.  The B operand
// is column half h of the previous product (rows of X or G for the Gram and
// polynomial products, X as MN-major for the step); it streams from L2
// through a ring of 64-deep K slices that every CTA fetches for itself (a
// slice multicast to the R CTAs of the half measured slower: a stage could
// only be refilled once all of them had consumed it).  Every CTA thus reads
// half of B per product (the work per CTA is half a row panel).  G and
// X' also go to global memory by TMA store for the next products' B
// operands, followed by a cluster barrier (two per step; P stays in shared
// memory).  The MMA commits of a product arrive at both partners, so neither
// overwrites a panel the other is still reading.  The last product applies the
// update from TMEM; partners exchange per-row partial sums for the norm.
//
// The K loop of every product takes the CTA's own half of the panel first and
// waits for the partner's half only before the rest.
//
// Warp roles (320 threads): warp 0 lane 0 issues the TMA loads, warp 1
// the tcgen05 MMAs (M = 128, N = d/2; one elected lane issues), warps 2..9 drain TMEM (warp w
// reads lanes 32 (w % 4) .., column quarter (w - 2) / 4 of the half).  Every
// mbarrier wait is bounded and reports TTT_ERR_TIMEOUT; every thread reaches
// every cluster barrier.
#include <cstring>

#include "builder.h"
#include "common.cuh"
#include "exec.h"
#include "launch.h"
#include "ns_cluster.h"
#include "ns_half.h"
#include "prof.h"

namespace ttt {

namespace {

constexpr int kHThreads = 320;
constexpr int kHCtrl = 3072;                 // barriers, TMEM slot, row sums (own [2][128], peer [128])
constexpr int kHMaxStages = 8;
constexpr int kHMaxR = 4;                    // largest order d = 128 kHMaxR
constexpr int kHChunk = 128 * 64 * 2;        // one 64-column chunk of a 128-row bf16 panel
constexpr int kHProdLanes = 1;               // TMA-issuing lanes of warp 0 (2 measured no faster)

enum HalfMap : int {
  HM_X0 = 0, HM_X1, HM_G,        // 64 x (d/2) boxes: one K slice of a column half (K-major B)
  HM_X0_MN, HM_X1_MN,            // MN-major B slices: 64 K rows x d/2 columns as R blocks of
                                 // 64 columns (3-D map), or 64 x 64 shares (2-D, mn_split)
  HM_X0_P, HM_X1_P, HM_G_P,      // 64 x 128 boxes: panel chunks (A load, stores)
  HM_W0, HM_W1, HM_W2,           // fp32 32 x 128 boxes: fast-weight blocks per slot
  HM_COUNT
};

struct NsHalfLaunch {
  CUtensorMap maps[HM_COUNT];
  const float* normsq_part;  // partial sums of the squared Frobenius norms of M
  int nslot;                 // partials per matrix
  float* W[3];              // fp32 state per slot (W1, W3, W2), [B*H][d*d]
  void* Wb[3];              // bf16 operand copies per slot
  int BH, d, steps, l2norm, h0, nh, R, nstages;
  int slot0;                // first matrix slot of this launch (its slots are slot0 ..)
  int mn_split;             // MN-major slices fetched as R shares of 64 columns
  float a, b, c, eps;
  int* status;
  unsigned long long wait_limit_ns;
};

static_assert(sizeof(NsHalfLaunch) <= 4096, "kernel parameter block too large");

int half_stages(int d) {
  const int R = d / 128;
  int n = (kUmmaSmemBytes - 1024 - kHCtrl - (d / 64) * kHChunk) / (8192 * R);
  return n > kHMaxStages ? kHMaxStages : n;
}

__device__ __forceinline__ uint32_t hpack(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 hunpack(uint32_t u) {
  return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u));
}

// 32 columns of this thread's panel row: TMEM -> bf16 -> shared panel (row at
// `row_saddr` of the chunk holding column gcol, 128-byte swizzle).  kind 0/2:
// sc * acc; kind 1: a [diagonal] + b G + c acc, G read from the panel.
__device__ __forceinline__ void half_block(int kind, float a, float b, float c, float sc,
                                           uint32_t taddr, uint32_t row_saddr, int rl, int grow,
                                           int gcol) {
  float v[32];
  tmem_ld32(taddr, v);
  const int u0 = (gcol & 63) >> 3;
  uint4 g[4];
  if (kind == 1) {
#pragma unroll
    for (int j = 0; j < 4; ++j) g[j] = lds128(row_saddr + ((uint32_t)((u0 + j) ^ (rl & 7)) << 4));
  }
  tmem_wait32(v);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float x[8];
    if (kind == 1) {
      const uint32_t gw[4] = {g[j].x, g[j].y, g[j].z, g[j].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 gf = hunpack(gw[i]);
        x[2 * i] = b * gf.x + c * v[8 * j + 2 * i];
        x[2 * i + 1] = b * gf.y + c * v[8 * j + 2 * i + 1];
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (grow == gcol + 8 * j + i) x[i] += a;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = sc * v[8 * j + i];
    }
    sts128(row_saddr + ((uint32_t)((u0 + j) ^ (rl & 7)) << 4),
           make_uint4(hpack(x[0], x[1]), hpack(x[2], x[3]), hpack(x[4], x[5]), hpack(x[6], x[7])));
  }
}

// Final update of this CTA's 128 x d/2 block: W <- (W - sc U) / |row| (or
// W - sc U), U in TMEM.  The fp32 W block is staged through shared memory
// (`wtile`, 32-column chunks of 128 rows, 128-byte swizzle, TMA in and out);
// row norms combine the two column quarters of this CTA and, through the
// partner's shared memory, the partner's half.  All 256 epilogue threads.
__device__ __noinline__ void half_update(const NsHalfLaunch& L, int z, int r, int h, int rl, int c2,
                                         int e_warp, int lane, uint32_t tl, float sc, bool got,
                                         float* rs_own, float* rs_peer, uint8_t* wtile,
                                         uint64_t* wbar, uint64_t* rsbar, uint32_t peer_rs,
                                         uint32_t peer_rsbar) {
  const int d = L.d, half = d / 2, nwc = half / 32, qc = half / 2;
  const int slot = z / L.BH, bh = z % L.BH;
  const CUtensorMap* wmap = &L.maps[HM_W0 + slot];
  const int wrow = bh * d + r * 128, wcol = h * half;
  const bool leader = e_warp == 0 && lane == 0;
  const uint32_t wsaddr = smem_u32(wtile);
  if (leader && got) {
    mbar_arrive_expect_tx(wbar, (uint32_t)(nwc * 16384));
    for (int ch = 0; ch < nwc; ++ch) tma_load_2d(wtile + ch * 16384, wmap, wcol + ch * 32, wrow, wbar);
  }
  const bool okw = got && mbar_wait(wbar, 0, L.status, L.wait_limit_ns);
  float ss = 0.f;
  if (okw) {
    for (int c0 = 0; c0 < qc; c0 += 32) {
      float v[32];
      tmem_ld32(tl + c0, v);
      tmem_wait32(v);
      const uint32_t row = wsaddr + ((c2 * qc + c0) >> 5) * 16384 + rl * 128;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t ad = row + ((uint32_t)(u ^ (rl & 7)) << 4);
        const uint4 w = lds128(ad);
        const float y0 = __uint_as_float(w.x) - sc * v[4 * u];
        const float y1 = __uint_as_float(w.y) - sc * v[4 * u + 1];
        const float y2 = __uint_as_float(w.z) - sc * v[4 * u + 2];
        const float y3 = __uint_as_float(w.w) - sc * v[4 * u + 3];
        ss += y0 * y0 + y1 * y1 + y2 * y2 + y3 * y3;
        sts128(ad, make_uint4(__float_as_uint(y0), __float_as_uint(y1), __float_as_uint(y2),
                              __float_as_uint(y3)));
      }
    }
  }
  if (L.l2norm) {
    // this CTA's two column quarters, then the partner's half of the row
    rs_own[c2 * 128 + rl] = ss;
    named_bar_sync(2, 256);
    const float mine = rs_own[rl] + rs_own[128 + rl];
    if (c2 == 0) {
      st_cluster_f32(peer_rs + (uint32_t)rl * 4u, mine);
      fence_acq_rel_cluster();
    }
    named_bar_sync(2, 256);
    if (leader) mbar_arrive_cluster(peer_rsbar);
    const bool okr = mbar_wait_cluster(rsbar, 0, L.status, L.wait_limit_ns);
    const float inv = okr ? 1.0f / fmaxf(sqrtf(mine + rs_peer[rl]), 1e-12f) : 1.0f;
    if (okw) {
      for (int c0 = 0; c0 < qc; c0 += 32) {
        const uint32_t row = wsaddr + ((c2 * qc + c0) >> 5) * 16384 + rl * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint32_t ad = row + ((uint32_t)(u ^ (rl & 7)) << 4);
          const uint4 w = lds128(ad);
          sts128(ad, make_uint4(__float_as_uint(__uint_as_float(w.x) * inv),
                                __float_as_uint(__uint_as_float(w.y) * inv),
                                __float_as_uint(__uint_as_float(w.z) * inv),
                                __float_as_uint(__uint_as_float(w.w) * inv)));
        }
      }
    }
  }
  fence_proxy_async_smem();
  named_bar_sync(2, 256);
  if (leader && okw) {
    for (int ch = 0; ch < nwc; ++ch) tma_store_2d(wmap, wcol + ch * 32, wrow, wtile + ch * 16384);
    bulk_commit_group();
  }
  if (okw) {   // bf16 operand copy: warp e_warp writes rows 16 e_warp .. + 15 of the block
    // lane l converts columns 8 l .. 8 l + 7 (two 16-byte shared loads, one
    // 16-byte store); four rows are in flight per iteration
    __nv_bfloat16* Wb = static_cast<__nv_bfloat16*>(L.Wb[slot]) + (long long)wrow * d + wcol;
    const int ch = lane >> 2, g = 2 * (lane & 3);
    if (lane < half / 8) {
      for (int r0 = e_warp * 16; r0 < e_warp * 16 + 16; r0 += 4) {
        uint4 w0[4], w1[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int rr = r0 + i;
          const uint32_t row = wsaddr + ch * 16384 + rr * 128;
          w0[i] = lds128(row + ((uint32_t)(g ^ (rr & 7)) << 4));
          w1[i] = lds128(row + ((uint32_t)((g + 1) ^ (rr & 7)) << 4));
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 o = make_uint4(hpack(__uint_as_float(w0[i].x), __uint_as_float(w0[i].y)),
                                     hpack(__uint_as_float(w0[i].z), __uint_as_float(w0[i].w)),
                                     hpack(__uint_as_float(w1[i].x), __uint_as_float(w1[i].y)),
                                     hpack(__uint_as_float(w1[i].z), __uint_as_float(w1[i].w)));
          *reinterpret_cast<uint4*>(Wb + (long long)(r0 + i) * d + 8 * lane) = o;
        }
      }
    }
  }
  if (leader && okw) bulk_wait_all();
}

// One instantiation per order d = 128 R: the loop bounds over panel chunks,
// K slices and epilogue columns are compile-time (measured 0.8% faster per
// layer step at d = 384 than one kernel for all d).
template <int R>
__global__ void __launch_bounds__(kHThreads, 1)
    ns_half_kernel(const __grid_constant__ NsHalfLaunch L) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kHMaxStages;
  uint64_t* mma_done = empty + kHMaxStages;   // both partners' MMAs of a product complete
  uint64_t* own_ready = mma_done + 1;         // this CTA's half of the next A panel written
  uint64_t* pready = own_ready + 1;           // [R] chunk j of the partner's half landed
  uint64_t* abar = pready + kHMaxR;           // first A panel loaded
  uint64_t* wbar = abar + 1;                  // fp32 W block loaded (final update)
  uint64_t* rsbar = wbar + 1;                 // partner's row sums written
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rsbar + 1);
  float* rs_own = reinterpret_cast<float*>(smem + 1024);   // [2][128]
  float* rs_peer = rs_own + 256;                           // [128], written by the partner
  static_assert(1024 + 3 * 128 * 4 <= kHCtrl, "row sums inside the control region");
  static_assert(R <= kHMaxR && (2 * kHMaxStages + kHMaxR + 6) * 8 + 4 <= 1024,
                "barriers and TMEM slot below the row sums");
  uint8_t* apanel = smem + kHCtrl;

  constexpr int d = 128 * R, nk = d / 64, half = d / 2;
  const int nstages = L.nstages;
  const uint32_t stage_bytes = 8192u * (uint32_t)R;
  uint8_t* ring = apanel + nk * kHChunk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)cluster_ctarank();
  const int h = rank / R, r = rank % R;        // column half, row panel
  const int partner = (1 - h) * R + r;
  const uint16_t pmask = (uint16_t)((1u << rank) | (1u << partner));
  const int zl = blockIdx.x / (2 * R);
  const int z = (L.slot0 + zl / L.nh) * L.BH + L.h0 + (zl % L.nh);
  const int mrow = z * d;                     // first row of this matrix in the stacked buffers
  const int prow = mrow + r * 128;            // first row of this CTA's panel
  const unsigned long long lim = L.wait_limit_ns;
  if (threadIdx.x == 0) {
    for (int s = 0; s < nstages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(mma_done, 2);
    mbar_init(own_ready, 1);
    for (int j = 0; j < R; ++j) mbar_init(&pready[j], 1);
    mbar_init(abar, 1);
    mbar_init(wbar, 1);
    mbar_init(rsbar, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0)
    for (int i = 0; i < HM_COUNT; ++i) tma_prefetch_map(&L.maps[i]);
  if (warp == 1) tmem_alloc(tmem_slot, 256);
  tc_fence_before();
  cluster_sync_all();   // peers signal our barriers: initialise them first
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the setup above touches no global memory; the gradient launch before this
  // one in the stream wrote the iterates and the norm partials read below
  pdl_wait();
  // every warp sums the partials in the same fixed order (same value everywhere)
  const float s1 =
      1.0f / (sqrtf(sum_partials_warp(L.normsq_part + (long long)z * L.nslot, L.nslot)) + L.eps);
  const uint32_t peer_pready = map_cluster(smem_u32(pready), (uint32_t)partner);   // + 8 j: chunk j
  const uint32_t peer_panel = map_cluster(smem_u32(apanel), (uint32_t)partner);
  const uint32_t peer_rs = map_cluster(smem_u32(rs_peer), (uint32_t)partner);
  const uint32_t peer_rsbar = map_cluster(smem_u32(rsbar), (uint32_t)partner);

  int s_prod = 0, s_mma = 0, issued = 0;
  uint32_t ph_prod = 0, ph_mma = 0;
  bool ok = true;
  bool copy_after_arrive = false;   // epilogue leader: panel copy deferred past the barrier arrival
  const int nprod = 3 * L.steps;
  const int nint = 2 * L.steps;
  // intervals: {G(t)} and {P(t), X(t+1)}; a cluster barrier closes each but the last
  for (int iv = 0; iv < nint; ++iv) {
    const int t = iv >> 1;
    const int p_begin = (iv & 1) ? 3 * t + 1 : 3 * t;
    const int p_end = (iv & 1) ? 3 * t + 3 : 3 * t + 1;
    if (warp == 0) {
      if (lane < kHProdLanes && ok) {
        fence_proxy_async_global();
        if (iv == 0 && lane == 0) {
          mbar_arrive_expect_tx(abar, (uint32_t)(nk * kHChunk));
          for (int c = 0; c < nk; ++c)
            tma_load_2d(apanel + c * kHChunk, &L.maps[HM_X0_P], c * 64, prow, abar);
        }
        if (iv == nint - 1 && lane == 0) {   // the final update reads these fp32 W rows
          const int slot = z / L.BH, bh = z % L.BH;
          const char* wp = reinterpret_cast<const char*>(
              L.W[slot] + ((long long)bh * d + r * 128) * d);
          const int bytes = 128 * d * 4;
          for (int o = 0; o < bytes; o += 16384)
            prefetch_l2_bulk(wp + o, (uint32_t)min(16384, bytes - o));
        }
        for (int p = p_begin; p < p_end && ok; ++p) {
          const int kind = p % 3, tp = p / 3;
          const CUtensorMap* map =
              kind == 1 ? &L.maps[HM_G]
                        : &L.maps[kind == 2 ? ((tp & 1) ? HM_X1_MN : HM_X0_MN)
                                            : ((tp & 1) ? HM_X1 : HM_X0)];
          for (int i = 0; i < nk; ++i) {
            const int ks = i < R ? h * R + i : (1 - h) * R + i - R;   // own half of K first
            if ((issued % kHProdLanes) == lane) {
              if (!mbar_wait(&empty[s_prod], ph_prod ^ 1, L.status, lim)) {
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(&full[s_prod], stage_bytes);
              uint8_t* dst = ring + s_prod * stage_bytes;
              // the whole K slice of this CTA's column half (one box, or R shares)
              if (kind == 2) {   // X as MN-major B: K = rows of X, N = its columns of half h
                if (L.mn_split) {
                  for (int j = 0; j < R; ++j)
                    tma_load_2d(dst + j * 8192, map, h * half + j * 64, mrow + ks * 64,
                                &full[s_prod]);
                } else {
                  tma_load_3d(dst, map, 0, mrow + ks * 64, h * R, &full[s_prod]);
                }
              } else {   // rows of X or G of half h as K-major B
                tma_load_2d(dst, map, ks * 64, mrow + h * half, &full[s_prod]);
              }
            }
            ++issued;   // every producer lane walks every entry
            if (++s_prod == nstages) {
              s_prod = 0;
              ph_prod ^= 1;
            }
          }
        }
      }
    } else if (warp == 1) {
      if (ok) {   // the whole warp walks the loop; one elected lane issues
        // descriptors advanced by byte offset / 16 in the start-address field
        const uint64_t a_desc0 = smem_desc_sw128(smem_u32(apanel), 16, 1024);
        const uint64_t bk_desc0 = smem_desc_sw128(smem_u32(ring), 16, 1024);     // K-major B
        const uint64_t bm_desc0 = smem_desc_sw128(smem_u32(ring), 8192, 1024);   // MN-major B
        const uint32_t stage16 = stage_bytes >> 4;
        for (int p = p_begin; p < p_end && ok; ++p) {
          const int kind = p % 3;
          // The K slices of this CTA's own half of the A panel come first (its
          // own epilogue wrote them); the partner's half is waited for only
          // before the remaining slices, so the exchange hides behind them.
          ok = p == 0 ? mbar_wait_w(abar, 0, L.status, lim)
                      : mbar_wait_w(own_ready, (uint32_t)((p - 1) & 1), L.status, lim);
          if (!ok) break;
          tc_fence_after();
          const uint32_t idesc = idesc_bf16_f32(half, 0, kind == 2 ? 1 : 0);
          const uint64_t b_desc0 = kind == 2 ? bm_desc0 : bk_desc0;
          const uint32_t bkk = kind == 2 ? 2048 / 16 : 32 / 16;
          for (int i = 0; i < nk; ++i) {
            const int ks = i < R ? h * R + i : (1 - h) * R + i - R;
            if (i >= R && p > 0) {   // chunk i - R of the partner's half
              if (!mbar_wait_cluster_w(&pready[i - R], (uint32_t)((p - 1) & 1), L.status, lim)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            if (!mbar_wait_w(&full[s_mma], ph_mma, L.status, lim)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t ad = a_desc0 + (uint64_t)(ks * (kHChunk / 16));
            const uint64_t bd = b_desc0 + (uint64_t)(s_mma * stage16);
            umma_bf16_w(tmem, ad, bd, idesc, i != 0);
            umma_bf16_w(tmem, ad + 2, bd + bkk, idesc, 1);
            umma_bf16_w(tmem, ad + 4, bd + 2 * bkk, idesc, 1);
            umma_bf16_w(tmem, ad + 6, bd + 3 * bkk, idesc, 1);
            umma_commit_w(&empty[s_mma]);
            if (++s_mma == nstages) {
              s_mma = 0;
              ph_mma ^= 1;
            }
          }
          if (ok) umma_commit_mc_w(mma_done, pmask);   // this product done, at both partners
        }
      }
    } else {
      const int e_warp = warp - 2;
      const int q = warp & 3, c2 = e_warp >> 2;
      const int rl = q * 32 + lane;
      const int grow = r * 128 + rl;                  // row inside the matrix
      const int qc = half / 2;                        // columns per thread
      const uint32_t tlb = tmem + ((uint32_t)(q * 32) << 16);       // this warp's TMEM lanes
      const uint32_t tl = tlb + (uint32_t)(c2 * qc);
      const bool leader = e_warp == 0 && lane == 0;
      const float ca = L.a, cb = L.b, cc = L.c;
      const uint32_t a_saddr = smem_u32(apanel);
      for (int p = p_begin; p < p_end; ++p) {
        const int kind = p % 3, tp = p / 3;
        const bool last = p == nprod - 1;
        const bool got = ok && mbar_wait_cluster(mma_done, (uint32_t)(p & 1), L.status, lim);
        tc_fence_after();
        const float sc = tp == 0 ? (kind == 0 ? s1 * s1 : s1) : 1.f;
        if (last) {
          half_update(L, z, r, h, rl, c2, e_warp, lane, tl, sc, got, rs_own, rs_peer, apanel, wbar,
                      rsbar, peer_rs, peer_rsbar);
        } else {
          // The half panel is drained one 64-column chunk at a time (each
          // warp takes 32 columns of it); G and X', which the other CTAs read
          // as B operands, leave chunk by chunk by TMA store as soon as every
          // warp has written the chunk, under the drain of the next ones.  P
          // needs no store; each chunk goes straight to the partner instead,
          // landing on that chunk's own barrier there.
          const int map = kind == 0 ? HM_G_P : (((tp + 1) & 1) ? HM_X1_P : HM_X0_P);
#pragma unroll
          for (int j = 0; j < R; ++j) {
            const int lc = 64 * j + 32 * c2;   // column inside this CTA's half
            if (got)
              half_block(kind, ca, cb, cc, sc, tlb + (uint32_t)lc,
                         a_saddr + (h * R + j) * kHChunk + rl * 128, rl, grow, h * half + lc);
            fence_proxy_async_smem();
            named_bar_sync(1, 256);
            if (leader && got) {
              const uint32_t off = (uint32_t)((h * R + j) * kHChunk);
              if (kind != 1)
                tma_store_2d(&L.maps[map], (h * R + j) * 64, prow, apanel + off);
              else
                bulk_copy_s2c(peer_panel + off, a_saddr + off, (uint32_t)kHChunk,
                              peer_pready + 8u * (uint32_t)j);
            }
          }
          if (leader && got) {
            if (kind != 1) bulk_commit_group();
            // Before a cluster barrier (G, X') the copies to the partner are
            // issued after the barrier arrival: a release-ordered arrival would
            // wait for them.
            if (kind != 1) copy_after_arrive = true;
            for (int j = 0; j < R; ++j) mbar_arrive_expect_tx(&pready[j], (uint32_t)kHChunk);
            mbar_arrive(own_ready);
            if (kind != 1) {
              bulk_wait_all();
              fence_proxy_async_global();
            }
          }
        }
        if (!got) ok = false;
      }
    }
    if (iv + 1 < nint) {
      cluster_arrive();
      if (copy_after_arrive) {
        for (int j = 0; j < R; ++j) {
          const uint32_t off = (uint32_t)((h * R + j) * kHChunk);
          bulk_copy_s2c(peer_panel + off, smem_u32(apanel) + off, (uint32_t)kHChunk,
                        peer_pready + 8u * (uint32_t)j);
        }
        copy_after_arrive = false;
      }
      cluster_wait();
    }
  }

  // the last product's MMAs are issued: the next launch may start its setup
  // while the update finishes
  if (warp == 1 && lane == 0) pdl_launch_dependents();

  // the last commits into our ring barriers must have landed before the exit
  if (warp == 0 && lane == 0 && ok) {
    const int n = issued < nstages ? issued : nstages;
    for (int i = 0; i < n; ++i) {
      if (!mbar_wait(&empty[s_prod], ph_prod ^ 1, L.status, lim)) break;
      if (++s_prod == nstages) {
        s_prod = 0;
        ph_prod ^= 1;
      }
    }
  }
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

int g_half_fit[64][9];   // per device and cluster size: 0 unknown, 1 fits, 2 does not

using HalfKernel = void (*)(NsHalfLaunch);

// The instantiation for d = 128 R (R = 1..4), else null.
HalfKernel half_kernel(int R) {
  switch (R) {
    case 1: return ns_half_kernel<1>;
    case 2: return ns_half_kernel<2>;
    case 3: return ns_half_kernel<3>;
    case 4: return ns_half_kernel<4>;
    default: return nullptr;
  }
}

}  // namespace

bool ns_half_applicable(int d) {
  return d % 128 == 0 && d >= 128 && d <= 512 && half_stages(d) >= 2;
}

bool prepare_ns_half(int d) {
  if (!ns_half_applicable(d)) return false;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  const int cs = 2 * (d / 128);
  std::lock_guard<std::mutex> lk(setup_mutex());
  int& c = g_half_fit[dev][cs];
  if (c == 0) {
    c = 2;
    if (cudaFuncSetAttribute(half_kernel(d / 128), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kUmmaSmemBytes) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = cs;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(cs, 1, 1);
      cfg.blockDim = dim3(kHThreads, 1, 1);
      cfg.dynamicSmemBytes = kUmmaSmemBytes;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, half_kernel(d / 128), &cfg) == cudaSuccess && n > 0)
        c = 1;
    }
    cudaGetLastError();
  }
  return c == 1;
}

int launch_ns_half(MapCache& cache, const NsArgs& a, int* status, unsigned long long wait_ns,
                   cudaStream_t stream) {
  if (!prepare_ns_half(a.d) || a.steps < 1) return 1;
  const int d = a.d, R = d / 128, cs = 2 * R, Z = a.zcount > 0 ? a.zcount : 3 * a.BH;
  NsHalfLaunch L;
  std::memset(&L, 0, sizeof(L));
  const TensorRef TX0{a.X[0], 1, (long long)Z * d, d};
  const TensorRef TX1{a.X[1], 1, (long long)Z * d, d};
  const TensorRef TG{a.G, 1, (long long)Z * d, d};
  const TensorRef TW0{a.W[0], 0, (long long)a.BH * d, d};
  const TensorRef TW1{a.W[1], 0, (long long)a.BH * d, d};
  const TensorRef TW2{a.W[2], 0, (long long)a.BH * d, d};
  const struct {
    TensorRef t;
    int box;
  } maps[HM_COUNT] = {{TX0, 64 * R}, {TX1, 64 * R}, {TG, 64 * R}, {TX0, 64},  {TX1, 64},
                      {TX0, 128},    {TX1, 128},    {TG, 128},    {TW0, 128}, {TW1, 128},
                      {TW2, 128}};
  // MN-major slices as one 3-D box of R column blocks where the driver takes
  // the blocked view, else as R shares of 64 columns
  L.mn_split = !(cache.get_blocked(TX0, 64, R, &L.maps[HM_X0_MN]) &&
                 cache.get_blocked(TX1, 64, R, &L.maps[HM_X1_MN]));
  for (int i = 0; i < HM_COUNT; ++i) {
    if (!L.mn_split && (i == HM_X0_MN || i == HM_X1_MN)) continue;
    if (!cache.get(maps[i].t, maps[i].box, &L.maps[i])) return -4;
  }
  L.normsq_part = a.normsq_part;
  L.nslot = a.nslot;
  for (int s = 0; s < 3; ++s) {
    L.W[s] = a.W[s];
    L.Wb[s] = a.Wb[s];
  }
  L.BH = a.BH;
  L.d = d;
  L.steps = a.steps;
  L.l2norm = a.l2norm;
  L.slot0 = a.slot0;
  L.h0 = a.h0;
  L.nh = a.nh;
  L.R = R;
  L.nstages = half_stages(d);
  L.a = a.ns[0];
  L.b = a.ns[1];
  L.c = a.ns[2];
  L.eps = 1e-7f;
  L.status = status;
  L.wait_limit_ns = wait_ns;

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[3];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  attr[2].id = cudaLaunchAttributePriority;
  attr[2].val.priority = a.priority;
  cfg.gridDim = dim3(a.nslots * a.nh * cs, 1, 1);
  cfg.blockDim = dim3(kHThreads, 1, 1);
  cfg.dynamicSmemBytes = kUmmaSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = a.priority != 0 ? 3 : 2;
  const double n3 = (double)d * d * d;
  const double flops = (double)a.nslots * a.nh * a.steps * 6.0 * n3;
  const int sms = device_sm_count();
  ProfScope ps(PT_MUON_HALF, stream, flops, 0.0,
               sms > 0 ? (double)(a.nslots * a.nh * cs) / sms : 1.0);
  if (cudaLaunchKernelEx(&cfg, half_kernel(R), L) != cudaSuccess) return -6;
  return 0;
}

}  // namespace ttt
