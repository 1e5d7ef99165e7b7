// Muon for square fast-weight matrices whose order d is a multiple of 128
// (d <= 384): every Newton-Schulz step (eq 6 of the LaCT notes; the quintic of
// the Muon write-up) and the final W <- L2-Normalize(W - U) (eq 5) in one
// launch, one thread-block cluster of d / 128 CTAs per matrix.
//
// CTA r of a cluster owns rows [128 r, 128 r + 128) of every product, i.e.
// a full 128 x d row panel, accumulated in TMEM (d fp32 columns).  Per step:
//     G  = X X^T              (first step: scaled by 1/(|M|_F + eps)^2)
//     P  = a I + b G + c G G
//     X' = P X                (first step: scaled by 1/(|M|_F + eps))
// which is a X + (b G + c G G) X with the a-term folded into P.  The A operand
// of every product is this CTA's own panel of the previous product (X, G or
// P), so it never leaves shared memory: each epilogue writes its bf16 result
// into the A panel in the 128-byte-swizzled layout the MMA reads.  The B
// operand is the whole d x d matrix of the previous product (X rows for G,
// G rows for G G, X as MN-major for P X); it streams from L2 through a ring of
// shared-memory stages, each stage one 64-deep K slice of one column half,
// every CTA of the cluster fetching a 64-row share and multicasting it to all
// of them.  Panels that peers read (G and X') are written to global memory by
// TMA stores; a cluster barrier follows G and X' (P stays local), so a step
// costs two cluster barriers.  The last step's epilogue applies the update
// and row normalisation directly from TMEM.
//
// Warp roles (320 threads): warp 0 lanes 0-1 issue the TMA loads, warp 1 lane 0
// the tcgen05 MMAs, warps 2..9 drain TMEM (warp w reads lanes 32 (w % 4) ..,
// column half (w - 2) / 4).  Every mbarrier wait is bounded and reports
// TTT_ERR_TIMEOUT; every thread reaches every cluster barrier.
#include <cstring>

#include "builder.h"
#include "common.cuh"
#include "launch.h"
#include "ns_cluster.h"
#include "ns_panel.h"
#include "prof.h"

namespace ttt {

namespace {

constexpr int kPanelThreads = 320;
constexpr int kPanelCtrl = 2048;        // barriers, TMEM slot, row sums
constexpr int kPanelMaxStages = 8;
constexpr int kPanelChunk = 128 * 64 * 2;   // one 64-column chunk of a 128-row panel
constexpr int kProdLanes = 2;               // TMA-issuing lanes of warp 0

enum PanelMap : int {
  PM_X0 = 0, PM_X1, PM_G,        // 64 x 64 boxes: B-operand shares
  PM_X0_P, PM_X1_P, PM_G_P,      // 64 x 128 boxes: row panels (A load, panel stores)
  PM_W0, PM_W1, PM_W2,           // fp32 32 x 128 boxes: fast-weight row panels per slot
  PM_COUNT
};

struct NsPanelLaunch {
  CUtensorMap maps[PM_COUNT];
  const float* normsq_part;  // partial sums of the squared Frobenius norms of M
  int nslot;                 // partials per matrix
  float* W[3];              // fp32 state per slot (W1, W3, W2), [B*H][d*d]
  void* Wb[3];              // bf16 operand copies per slot
  int BH, d, steps, l2norm, h0, nh, cs, nstages;
  float a, b, c, eps;
  int* status;
  unsigned long long wait_limit_ns;
};

static_assert(sizeof(NsPanelLaunch) <= 4096, "kernel parameter block too large");

int panel_stages(int d) {
  const int nk = d / 64;
  const int stage = 8192 * (d / 128);
  int n = (kUmmaSmemBytes - 1024 - kPanelCtrl - nk * kPanelChunk) / stage;
  return n > kPanelMaxStages ? kPanelMaxStages : n;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t u) {
  return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u));
}

// One 64-column chunk of this thread's panel row: TMEM -> bf16 -> A panel
// (row r of the chunk at `row_saddr`, 128-byte swizzle).  kind 0 and 2:
// sc * acc; kind 1: a [diagonal] + b G + c acc with G read from the panel.
// `col0` is the chunk's first column, `grow` this row, both in the matrix.
__device__ __forceinline__ void panel_chunk(int kind, float a, float b, float c, float sc,
                                            uint32_t tl, uint32_t row_saddr, int r, int grow,
                                            int col0) {
#pragma unroll
  for (int hb = 0; hb < 2; ++hb) {
    float v[32];
    tmem_ld32(tl + hb * 32, v);
    uint4 g[4];
    if (kind == 1) {
#pragma unroll
      for (int j = 0; j < 4; ++j) g[j] = lds128(row_saddr + ((uint32_t)((hb * 4 + j) ^ (r & 7)) << 4));
    }
    tmem_wait32(v);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int unit = hb * 4 + j;
      float x[8];
      if (kind == 1) {
        const uint32_t gw[4] = {g[j].x, g[j].y, g[j].z, g[j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 gf = unpack_bf16x2(gw[i]);
          x[2 * i] = b * gf.x + c * v[8 * j + 2 * i];
          x[2 * i + 1] = b * gf.y + c * v[8 * j + 2 * i + 1];
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (grow == col0 + unit * 8 + i) x[i] += a;
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = sc * v[8 * j + i];
      }
      sts128(row_saddr + ((uint32_t)(unit ^ (r & 7)) << 4),
             make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]),
                        pack_bf16x2(x[4], x[5]), pack_bf16x2(x[6], x[7])));
    }
  }
}

// Final update of this CTA's 128 rows: W <- (W - sc U) / |row| (or W - sc U),
// U in TMEM.  The fp32 W panel is staged through shared memory (`wpanel`,
// 32-column chunks of 128 rows in the 128-byte swizzle, loaded and stored by
// TMA); the bf16 copy leaves with coalesced stores.  All 256 epilogue threads
// take part; `h` is this thread's column half.
__device__ __noinline__ void panel_update(const NsPanelLaunch& L, int z, int rank, int r, int h,
                                          int e_warp, int lane, uint32_t tl, float sc, bool got,
                                          float* rowss, uint8_t* wpanel, uint64_t* wbar) {
  const int d = L.d, half = d / 2, nwc = d / 32;
  const int slot = z / L.BH, bh = z % L.BH;
  const CUtensorMap* wmap = &L.maps[PM_W0 + slot];
  const int wrow = bh * d + rank * 128;
  const bool leader = e_warp == 0 && lane == 0;
  const uint32_t wsaddr = smem_u32(wpanel);
  if (leader && got) {
    mbar_arrive_expect_tx(wbar, (uint32_t)(nwc * 16384));
    for (int ch = 0; ch < nwc; ++ch)
      tma_load_2d(wpanel + ch * 16384, wmap, ch * 32, wrow, wbar);
  }
  const bool okw = got && mbar_wait(wbar, 0, L.status, L.wait_limit_ns);
  float ss = 0.f;
  if (okw) {
    for (int c0 = 0; c0 < half; c0 += 32) {
      float v[32];
      tmem_ld32(tl + c0, v);
      tmem_wait32(v);
      const uint32_t row = wsaddr + ((h * half + c0) >> 5) * 16384 + r * 128;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t ad = row + ((uint32_t)(u ^ (r & 7)) << 4);
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
  if (L.l2norm) {   // the two halves of a row meet in shared memory
    rowss[h * 128 + r] = ss;
    named_bar_sync(2, 256);
    const float inv = 1.0f / fmaxf(sqrtf(rowss[r] + rowss[128 + r]), 1e-12f);
    if (okw) {
      for (int c0 = 0; c0 < half; c0 += 32) {
        const uint32_t row = wsaddr + ((h * half + c0) >> 5) * 16384 + r * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint32_t ad = row + ((uint32_t)(u ^ (r & 7)) << 4);
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
    for (int ch = 0; ch < nwc; ch++) tma_store_2d(wmap, ch * 32, wrow, wpanel + ch * 16384);
    bulk_commit_group();
  }
  if (okw) {   // bf16 operand copy: warp e_warp writes rows 16 e_warp .. + 15, whole rows per pass
    __nv_bfloat16* Wb = static_cast<__nv_bfloat16*>(L.Wb[slot]) + (long long)wrow * d;
    const int sub = lane >> 3, u = lane & 7;
    for (int rr = e_warp * 16; rr < e_warp * 16 + 16; ++rr) {
      for (int c4 = 0; c4 < nwc; c4 += 4) {
        const int ch = c4 + sub;
        const uint4 w = lds128(wsaddr + ch * 16384 + rr * 128 + ((uint32_t)(u ^ (rr & 7)) << 4));
        const uint2 o = make_uint2(pack_bf16x2(__uint_as_float(w.x), __uint_as_float(w.y)),
                                   pack_bf16x2(__uint_as_float(w.z), __uint_as_float(w.w)));
        *reinterpret_cast<uint2*>(Wb + (long long)rr * d + ch * 32 + u * 4) = o;
      }
    }
  }
  if (leader && okw) bulk_wait_all();
}

__global__ void __launch_bounds__(kPanelThreads, 1)
    ns_panel_kernel(const __grid_constant__ NsPanelLaunch L) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kPanelMaxStages;
  uint64_t* accf = empty + kPanelMaxStages;   // accumulator complete (MMA -> epilogue)
  uint64_t* aready = accf + 1;                // panel rewritten, TMEM drained (epilogue -> MMA)
  uint64_t* abar = aready + 1;                // first A panel loaded
  uint64_t* wbar = abar + 1;                  // fp32 W panel loaded (final update)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(wbar + 1);
  float* rowss = reinterpret_cast<float*>(smem + 1024);   // [2][128]
  uint8_t* apanel = smem + kPanelCtrl;

  const int d = L.d, cs = L.cs, nk = d / 64, half = d / 2, nstages = L.nstages;
  const uint32_t stage_bytes = 8192u * (uint32_t)cs;
  uint8_t* ring = apanel + nk * kPanelChunk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)cluster_ctarank();
  const int zl = blockIdx.x / cs;
  const int z = (zl / L.nh) * L.BH + L.h0 + (zl % L.nh);
  const int mrow = z * d;                     // first row of this matrix in the stacked buffers
  const int prow = mrow + rank * 128;         // first row of this CTA's panel
  const uint16_t mask = (uint16_t)((1u << cs) - 1u);
  const unsigned long long lim = L.wait_limit_ns;
  // every warp sums the partials in the same fixed order (same value everywhere)
  const float s1 =
      1.0f / (sqrtf(sum_partials_warp(L.normsq_part + (long long)z * L.nslot, L.nslot)) + L.eps);

  if (threadIdx.x == 0) {
    for (int s = 0; s < nstages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], cs);
    }
    mbar_init(accf, 1);
    mbar_init(aready, 1);
    mbar_init(abar, 1);
    mbar_init(wbar, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0)
    for (int i = 0; i < PM_COUNT; ++i) tma_prefetch_map(&L.maps[i]);
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  cluster_sync_all();   // peers signal our barriers: initialise them first
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  int s_prod = 0, s_mma = 0, issued = 0;
  uint32_t ph_prod = 0, ph_mma = 0;
  bool ok = true;
  const int nprod = 3 * L.steps;
  const int nint = 2 * L.steps;
  // intervals: {G(t)} and {P(t), X(t+1)}; a cluster barrier closes each but the last
  for (int iv = 0; iv < nint; ++iv) {
    const int t = iv >> 1;
    const int p_begin = (iv & 1) ? 3 * t + 1 : 3 * t;
    const int p_end = (iv & 1) ? 3 * t + 3 : 3 * t + 1;
    if (warp == 0) {
      // kProdLanes lanes share the ring entries round robin: one thread cannot
      // issue the multicast boxes fast enough to keep the tensor cores busy
      if (lane < kProdLanes && ok) {
        fence_proxy_async_global();
        if (iv == 0 && lane == 0) {
          mbar_arrive_expect_tx(abar, (uint32_t)(nk * kPanelChunk));
          for (int c = 0; c < nk; ++c)
            tma_load_2d(apanel + c * kPanelChunk, &L.maps[PM_X0_P], c * 64, prow, abar);
        }
        if (iv == nint - 1 && lane == 0) {   // the final update reads this CTA's fp32 W rows
          const int slot = z / L.BH, bh = z % L.BH;
          const char* wp = reinterpret_cast<const char*>(
              L.W[slot] + ((long long)bh * d + rank * 128) * d);
          const int bytes = 128 * d * 4;
          for (int o = 0; o < bytes; o += 16384)
            prefetch_l2_bulk(wp + o, (uint32_t)min(16384, bytes - o));
        }
        for (int p = p_begin; p < p_end && ok; ++p) {
          const int kind = p % 3, tp = p / 3;
          const CUtensorMap* map = kind == 1 ? &L.maps[PM_G] : &L.maps[(tp & 1) ? PM_X1 : PM_X0];
          for (int h = 0; h < 2 && ok; ++h) {
            for (int ks = 0; ks < nk; ++ks) {
              if ((issued % kProdLanes) == lane) {
                if (!mbar_wait(&empty[s_prod], ph_prod ^ 1, L.status, lim)) {
                  ok = false;
                  break;
                }
                mbar_arrive_expect_tx(&full[s_prod], stage_bytes);
                uint8_t* dst = ring + s_prod * stage_bytes + rank * 8192;
                if (kind == 2)   // X as MN-major B: K = rows of X, N = its columns
                  tma_load_2d_mc(dst, map, h * half + rank * 64, mrow + ks * 64, &full[s_prod], mask);
                else             // rows of X or G as K-major B
                  tma_load_2d_mc(dst, map, ks * 64, mrow + h * half + rank * 64, &full[s_prod], mask);
              }
              ++issued;   // every producer lane walks every entry
              if (++s_prod == nstages) {
                s_prod = 0;
                ph_prod ^= 1;
              }
            }
          }
        }
      }
    } else if (warp == 1) {
      if (lane == 0 && ok) {
        // Base descriptors, advanced per operand slice by adding the byte
        // offset / 16 to the start-address field (shared addresses < 256 KB,
        // so the 14-bit field cannot carry).  The issue loop stays short: the
        // tensor core runs only as fast as this thread feeds it.
        const uint64_t a_desc0 = smem_desc_sw128(smem_u32(apanel), 16, 1024);
        const uint64_t bk_desc0 = smem_desc_sw128(smem_u32(ring), 16, 1024);     // K-major B
        const uint64_t bm_desc0 = smem_desc_sw128(smem_u32(ring), 8192, 1024);   // MN-major B
        const uint32_t stage16 = stage_bytes >> 4;
        for (int p = p_begin; p < p_end && ok; ++p) {
          const int kind = p % 3;
          ok = p == 0 ? mbar_wait(abar, 0, L.status, lim)
                      : mbar_wait(aready, (uint32_t)((p - 1) & 1), L.status, lim);
          if (!ok) break;
          tc_fence_after();
          const uint32_t idesc = idesc_bf16_f32(half, 0, kind == 2 ? 1 : 0);
          const uint64_t b_desc0 = kind == 2 ? bm_desc0 : bk_desc0;
          const uint32_t bkk = kind == 2 ? 2048 / 16 : 32 / 16;   // one 16-deep K slice
          for (int h = 0; h < 2 && ok; ++h) {
            const uint32_t dcol = tmem + (uint32_t)(h * half);
            for (int ks = 0; ks < nk; ++ks) {
              if (!mbar_wait(&full[s_mma], ph_mma, L.status, lim)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t ad = a_desc0 + (uint64_t)(ks * (kPanelChunk / 16));
              const uint64_t bd = b_desc0 + (uint64_t)(s_mma * stage16);
              umma_bf16(dcol, ad, bd, idesc, ks != 0);
              umma_bf16(dcol, ad + 2, bd + bkk, idesc, 1);
              umma_bf16(dcol, ad + 4, bd + 2 * bkk, idesc, 1);
              umma_bf16(dcol, ad + 6, bd + 3 * bkk, idesc, 1);
              umma_commit_mc(&empty[s_mma], mask);
              if (++s_mma == nstages) {
                s_mma = 0;
                ph_mma ^= 1;
              }
            }
          }
          umma_commit(accf);
        }
      }
    } else {
      const int e_warp = warp - 2;
      const int q = warp & 3, h = e_warp >> 2;
      const int r = q * 32 + lane;
      const int grow = rank * 128 + r;   // row inside the matrix
      const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * half);
      const bool lead = (e_warp & 3) == 0 && lane == 0;   // one thread per column half
      const int nch = half / 64;                          // 64-column chunks per half
      const float ca = L.a, cb = L.b, cc = L.c;
      const uint32_t a_saddr = smem_u32(apanel);
      for (int p = p_begin; p < p_end; ++p) {
        const int kind = p % 3, tp = p / 3;
        const bool last = p == nprod - 1;
        const bool got = ok && mbar_wait(accf, (uint32_t)(p & 1), L.status, lim);
        tc_fence_after();
        const float sc = tp == 0 ? (kind == 0 ? s1 * s1 : s1) : 1.f;
        if (last) {
          panel_update(L, z, rank, r, h, e_warp, lane, tl, sc, got, rowss, apanel, wbar);
        } else {
          // G and X' are read by the peers: each finished 64-column chunk of
          // a half leaves by TMA store while the next one is computed
          const int map = kind == 0 ? PM_G_P : (((tp + 1) & 1) ? PM_X1_P : PM_X0_P);
          for (int k = 0; k < nch; ++k) {
            const int ch = h * nch + k;
            if (got)
              panel_chunk(kind, ca, cb, cc, sc, tl + k * 64, a_saddr + ch * kPanelChunk + r * 128,
                          r, grow, ch * 64);
            if (kind != 1) {
              fence_proxy_async_smem();
              named_bar_sync(3 + h, 128);
              if (lead && got) {
                tma_store_2d(&L.maps[map], ch * 64, prow, apanel + ch * kPanelChunk);
                bulk_commit_group();
              }
            }
          }
          if (kind != 1 && lead && got) {
            bulk_wait_all();
            fence_proxy_async_global();
          }
        }
        tc_fence_before();
        fence_proxy_async_smem();
        named_bar_sync(1, 256);
        if (e_warp == 0 && lane == 0) mbar_arrive(aready);
        if (!got) ok = false;
      }
    }
    if (iv + 1 < nint) cluster_sync_all();
  }

  // every peer's multicast commit into our ring barriers must have landed
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
    tmem_dealloc(tmem, 512);
  }
}

int g_panel_fit[64][5];   // per device and cluster size: 0 unknown, 1 fits, 2 does not

}  // namespace

bool ns_panel_applicable(int d) {
  // the final update stages the 128 x d fp32 W panel in the A panel + ring
  return d % 128 == 0 && d >= 128 && d <= 384 && panel_stages(d) >= 2 &&
         d * 128 * 4 <= (d / 64) * kPanelChunk + panel_stages(d) * 8192 * (d / 128);
}

bool prepare_ns_panel(int d) {
  if (!ns_panel_applicable(d)) return false;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  const int cs = d / 128;
  int& c = g_panel_fit[dev][cs];
  if (c == 0) {
    c = 2;
    if (cudaFuncSetAttribute(ns_panel_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kUmmaSmemBytes) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = cs;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(cs, 1, 1);
      cfg.blockDim = dim3(kPanelThreads, 1, 1);
      cfg.dynamicSmemBytes = kUmmaSmemBytes;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, ns_panel_kernel, &cfg) == cudaSuccess && n > 0) c = 1;
    }
    cudaGetLastError();
  }
  return c == 1;
}

int launch_ns_panel(MapCache& cache, const NsArgs& a, int* status, unsigned long long wait_ns,
                    cudaStream_t stream) {
  if (!prepare_ns_panel(a.d) || a.steps < 1) return 1;
  const int d = a.d, cs = d / 128, Z = 3 * a.BH;
  NsPanelLaunch L;
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
  } maps[PM_COUNT] = {{TX0, 64},  {TX1, 64},  {TG, 64},   {TX0, 128}, {TX1, 128},
                      {TG, 128},  {TW0, 128}, {TW1, 128}, {TW2, 128}};
  for (int i = 0; i < PM_COUNT; ++i)
    if (!cache.get(maps[i].t, maps[i].box, &L.maps[i])) return -4;
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
  L.h0 = a.h0;
  L.nh = a.nh;
  L.cs = cs;
  L.nstages = panel_stages(d);
  L.a = a.ns[0];
  L.b = a.ns[1];
  L.c = a.ns[2];
  L.eps = 1e-7f;
  L.status = status;
  L.wait_limit_ns = wait_ns;

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(3 * a.nh * cs, 1, 1);
  cfg.blockDim = dim3(kPanelThreads, 1, 1);
  cfg.dynamicSmemBytes = kUmmaSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const double n3 = (double)d * d * d;
  const double flops = 3.0 * a.nh * a.steps * 6.0 * n3;
  ProfScope ps(PT_MUON_PANEL, stream, flops, 0.0);
  if (cudaLaunchKernelEx(&cfg, ns_panel_kernel, L) != cudaSuccess) return -6;
  return 0;
}

}  // namespace ttt
