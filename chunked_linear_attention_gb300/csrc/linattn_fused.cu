// Chunked linear attention in one cooperative launch on the tensor cores
// ("Test-Time Training with KV Binding Is Secretly Linear Attention", Thm 5.2
// and App. H with alpha = 0): per (batch, head) the state after chunk c is
// S0 + sum over visible chunks of V~_c^T K_c with V~ = eta * V, and the
// chunk's outputs are O_c = Q_c S_c^T (S_c before or after chunk c's own
// update, by mask mode).
//
// The work of a call is one ordered list of items, split statically over one
// CTA per SM (every CTA resident: cooperative launch):
//   A (batch-head, chunk, split): the partial state V~^T K over `slen` tokens
//     of an updating chunk.  The producer loads the token rows of V and K
//     (MN-major tiles, 128 tokens per stage); four warps scale the V rows by
//     eta in shared memory, then the MMA accumulates M = d_v by N = d_k over
//     the tokens in TMEM; the same warps store the fp32 partial.
//   P (batch-head, part): a slice of the state elements: the prefix over the
//     chunks of the partials, the bf16 state each chunk reads and the final
//     fp32 state.
//   B (batch-head, chunk, row block): O rows = Q rows S_c^T: the state is
//     loaded once per item, then 128-row tiles of Q stream through the MMA
//     (M = 128, N = d_v, K = d_k) and the epilogue writes bf16 rows.
// Items are listed A, then P, then B; CTA b takes items b, b + G, b + 2G...
// A P item waits for its batch-head's A items and a B item for its P items
// through counters in global memory (release after the stores, acquire before
// the reads; bounded waits).  Since every item an item waits for has a
// smaller index and every CTA walks its items in order, the waits end.
//
// Warp roles (192 threads): warp 0 lane 0 issues TMA loads, warp 1 the MMAs
// (one elected lane issues), warps 2..5 scale, drain TMEM (warp w reads lanes 32 (w % 4) ..) and
// run the prefix items.  Every mbarrier and counter wait is bounded and
// reports TTT_ERR_TIMEOUT.
#include <atomic>
#include <cstring>

#include "builder.h"
#include "common.cuh"
#include "exec.h"
#include "launch.h"
#include "linattn_fused.h"
#include "prof.h"

namespace ttt {

namespace {

constexpr int kLThreads = 192;
constexpr int kLCtrl = 1024;
constexpr int kLMaxStages = 8;
constexpr int kLTok = 128;                 // tokens (A) or rows (B) per pipeline stage

enum LinMap : int { LM_V = 0, LM_K, LM_Q, LM_S, LM_COUNT };

struct LinFusedLaunch {
  CUtensorMap maps[LM_COUNT];
  const float* eta;           // [BH][N]
  const float* S0;            // [BH][dv][dk] or NULL
  float* partials;            // [BH][nc][splits][dv][dk]
  __nv_bfloat16* s_read;      // [BH][nc][dv][dk]
  float* s_final;             // [BH][dv][dk] or NULL
  __nv_bfloat16* out;         // [BH][N][dv]
  const __nv_bfloat16* q;     // [BH][N][dk] (L2 prefetch; the loads use the maps)
  const __nv_bfloat16* k;     // [BH][N][dk]
  const __nv_bfloat16* v;     // [BH][N][dv]
  int* counters;              // [2][BH] items done: A, P (zero at launch)
  int BH, N, dk, dv, chunk, nc, splits, slen, pparts, rb, apply_first, n_upd;
  int nA, nP, nB, nstages;
  uint32_t stage_bytes;
  UpdateFlags flags;
  LinRule rule;               // momentum and per-chunk learning rates of the state update
  int* status;
  unsigned long long wait_limit_ns;
  int withhold_bh;            // test hook: this batch-head's A items never release (-1: none)
  int blocked;                // maps are 3-D blocked views: one box per tile (all 64-column
                              // blocks), else 2-D maps and one box per 64-column block
};

static_assert(sizeof(LinFusedLaunch) <= 4096, "kernel parameter block too large");

__device__ __forceinline__ bool chunk_updates(const LinFusedLaunch& L, int c) {
  return L.flags.all || ((L.flags.bits[c >> 5] >> (c & 31)) & 1u);
}

// Bounded wait until *p >= target (acquire at GPU scope).
__device__ __forceinline__ bool wait_count(const int* p, int target, int* status,
                                           unsigned long long lim) {
  unsigned long long t0 = 0;
  for (;;) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    if (v >= target) return true;
    const unsigned long long now = global_ns();
    if (t0 == 0) {
      t0 = now;
    } else if (now - t0 > lim) {
      report_status(status, kStatusTimeout);
      return false;
    }
    __nanosleep(128);
  }
}

struct Item {
  int kind;   // 0 = A, 1 = P, 2 = B
  int bh, c, sub;
};

__device__ __forceinline__ Item decode_item(const LinFusedLaunch& L, int i) {
  Item it;
  if (i < L.nA) {
    it.kind = 0;
    it.bh = i / (L.nc * L.splits);
    const int r = i - it.bh * L.nc * L.splits;
    it.c = r / L.splits;
    it.sub = r - it.c * L.splits;
  } else if (i < L.nA + L.nP) {
    const int j = i - L.nA;
    it.kind = 1;
    it.bh = j / L.pparts;
    it.c = 0;
    it.sub = j - it.bh * L.pparts;
  } else {
    const int j = i - L.nA - L.nP;
    const int rbs = L.chunk / L.rb;
    it.kind = 2;
    it.bh = j / (L.nc * rbs);
    const int r = j - it.bh * L.nc * rbs;
    it.c = r / rbs;
    it.sub = r - it.c * rbs;
  }
  return it;
}

// L2 prefetch of `bytes` contiguous bytes (16-byte multiple) in 32 KB pieces.
__device__ __forceinline__ void prefetch_rows_l2(const void* p, uint32_t bytes) {
  const char* c = static_cast<const char*>(p);
  for (uint32_t o = 0; o < bytes; o += 32768u) prefetch_l2_bulk(c + o, min(32768u, bytes - o));
}

__device__ __forceinline__ void ring_next(int& s, uint32_t& ph, int nstages) {
  if (++s == nstages) {
    s = 0;
    ph ^= 1;
  }
}

// One prefix item: the `per` (<= 2048) elements from e0 of batch-head bh's
// state.  Thread t owns the element groups (4 elements) e0 + 4 t + 512 g,
// g < kPG, and carries their running states across the chunks.  The
// producer warp brings the item's (chunk, split) partial slices into the
// ring by bulk copies, as many per stage as fit (generic loads of those
// partials measured slow: they finished ~9.5 us after the last A item,
// wherever they were issued).
constexpr int kPG = 4;

__device__ __forceinline__ void store_bf16x4(__nv_bfloat16* r, float4 v) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&lo);
  u.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(r) = u;
}

__device__ __forceinline__ void fma4(float4& y, float a, const float4& x) {
  y.x = fmaf(a, x.x, y.x); y.y = fmaf(a, x.y, y.y); y.z = fmaf(a, x.z, y.z); y.w = fmaf(a, x.w, y.w);
}

// Per updating chunk c: M <- alpha_c M + G_c, S <- S + lr_c M (rule.mom), or
// S <- S + lr_c G_c; chunks that do not update leave both unchanged.  Run by
// the four epilogue warps together (tid 0..127); walks the item's ring stages
// in step with the producer (s, ph) and releases each one.
__device__ __forceinline__ void prefix_item(const LinFusedLaunch& L, int bh, int e0, int per,
                                            int tid, const uint8_t* ring, uint64_t* full,
                                            uint64_t* empty, int& s, uint32_t& ph, bool& ok) {
  const long long E = (long long)L.dv * L.dk;
  const int npairs = L.nc * L.splits;
  const uint32_t sl = (uint32_t)per * 4;
  const int pps = (int)(L.stage_bytes / sl);
  const LinRule& R = L.rule;
  float4 s4[kPG], add[kPG], m[kPG];
  bool own[kPG];
#pragma unroll
  for (int g = 0; g < kPG; ++g) {
    const int off = 4 * tid + 512 * g;
    own[g] = off < per;
    s4[g] = (own[g] && L.S0) ? *reinterpret_cast<const float4*>(L.S0 + bh * E + e0 + off)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
    m[g] = (own[g] && R.M0) ? *reinterpret_cast<const float4*>(R.M0 + bh * E + e0 + off)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
    add[g] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int p0 = 0; p0 < npairs; p0 += pps) {
    if (ok) ok = mbar_wait(&full[s], ph, L.status, L.wait_limit_ns);
    ok = __all_sync(0xffffffffu, ok);
    const uint32_t st = smem_u32(ring + s * L.stage_bytes) + (uint32_t)tid * 16u;
    for (int j = 0; j < pps; ++j) {
      const int pr = p0 + j;
      if (pr >= npairs) break;
      if (ok && chunk_updates(L, pr / L.splits)) {
#pragma unroll
        for (int g = 0; g < kPG; ++g) {
          if (!own[g]) continue;
          const uint4 w = lds128(st + (uint32_t)j * sl + 2048u * g);
          add[g].x += __uint_as_float(w.x); add[g].y += __uint_as_float(w.y);
          add[g].z += __uint_as_float(w.z); add[g].w += __uint_as_float(w.w);
        }
      }
      if ((pr + 1) % L.splits != 0) continue;
      // chunk pr / splits complete: the state it reads, then the running state
      const int c = pr / L.splits;
      const bool upd = chunk_updates(L, c);
      const float lr = (upd && R.lr) ? R.lr[(long long)bh * L.nc + c] : R.lr_const;
      const float al = (upd && R.mom && R.alpha) ? R.alpha[(long long)bh * L.nc + c]
                                                 : R.alpha_const;
#pragma unroll
      for (int g = 0; g < kPG; ++g) {
        if (!own[g]) continue;
        float4 inc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (upd) {
          if (R.mom) {
            float4 mm = add[g];
            fma4(mm, al, m[g]);
            m[g] = mm;
            fma4(inc, lr, mm);
          } else {
            fma4(inc, lr, add[g]);
          }
        }
        float4 rd = s4[g];
        if (!L.apply_first) {
          rd.x += inc.x; rd.y += inc.y; rd.z += inc.z; rd.w += inc.w;
        }
        if (ok)
          store_bf16x4(L.s_read + (long long)(bh * L.nc + c) * E + e0 + 4 * tid + 512 * g, rd);
        s4[g].x += inc.x; s4[g].y += inc.y; s4[g].z += inc.z; s4[g].w += inc.w;
        add[g] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    named_bar_sync(1, 128);   // every thread is done with the stage
    if (tid == 0 && ok) mbar_arrive(&empty[s]);
    ring_next(s, ph, L.nstages);
  }
  if (!ok) return;
#pragma unroll
  for (int g = 0; g < kPG; ++g) {
    if (!own[g]) continue;
    const long long o = bh * E + e0 + 4 * tid + 512 * g;
    if (L.s_final) *reinterpret_cast<float4*>(L.s_final + o) = s4[g];
    if (R.M_final) *reinterpret_cast<float4*>(R.M_final + o) = m[g];
  }
}

__global__ void __launch_bounds__(kLThreads, 1)
    linattn_fused_kernel(const __grid_constant__ LinFusedLaunch L) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kLMaxStages;
  uint64_t* scaled = empty + kLMaxStages;
  uint64_t* accf = scaled + kLMaxStages;   // [2]
  uint64_t* acce = accf + 2;               // [2]
  uint64_t* sfull = acce + 2;              // state tile of a B item loaded
  uint64_t* sempty = sfull + 1;            // state tile no longer read
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sempty + 1);
  uint8_t* sreg = smem + kLCtrl;                           // state tile (d_v rows x d_k)
  const uint32_t s_bytes = (uint32_t)L.dv * L.dk * 2;
  uint8_t* ring = sreg + ((s_bytes + 1023) & ~1023u);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nstages = L.nstages;
  const uint32_t stage_bytes = L.stage_bytes;
  const unsigned long long lim = L.wait_limit_ns;
  const int total = L.nA + L.nP + L.nB;
  int* doneA = L.counters;
  int* doneP = L.counters + L.BH;
  const int dvb = L.dv / 64, dkb = L.dk / 64;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nstages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&scaled[s], 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], 4);
    }
    mbar_init(sfull, 1);
    mbar_init(sempty, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0)
    for (int i = 0; i < LM_COUNT; ++i) tma_prefetch_map(&L.maps[i]);
  if (warp == 1) tmem_alloc(tmem_slot, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int s = 0, nb = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int i = blockIdx.x; i < total && ok; i += gridDim.x) {
        const Item it = decode_item(L, i);
        if (it.kind == 0) {
          if (!chunk_updates(L, it.c)) continue;
          const int row0 = it.bh * L.N + it.c * L.chunk + it.sub * L.slen;
          const int nst = L.slen / kLTok;
          for (int j = 0; j < nst && ok; ++j) {
            // keep one more ring's depth of this item's rows on the way into L2
            if (j + nstages < nst) {
              const long long pr = (long long)row0 + (j + nstages) * kLTok;
              prefetch_rows_l2(L.v + pr * L.dv, (uint32_t)kLTok * L.dv * 2);
              prefetch_rows_l2(L.k + pr * L.dk, (uint32_t)kLTok * L.dk * 2);
            }
            if (!mbar_wait(&empty[s], ph ^ 1, L.status, lim)) { ok = false; break; }
            mbar_arrive_expect_tx(&full[s], (uint32_t)(L.dv + L.dk) * kLTok * 2);
            uint8_t* st = ring + s * stage_bytes;
            if (L.blocked) {
              tma_load_3d(st, &L.maps[LM_V], 0, row0 + j * kLTok, 0, &full[s]);
              tma_load_3d(st + dvb * 16384, &L.maps[LM_K], 0, row0 + j * kLTok, 0, &full[s]);
            } else {
              for (int b = 0; b < dvb; ++b)
                tma_load_2d(st + b * 16384, &L.maps[LM_V], b * 64, row0 + j * kLTok, &full[s]);
              for (int b = 0; b < dkb; ++b)
                tma_load_2d(st + (dvb + b) * 16384, &L.maps[LM_K], b * 64, row0 + j * kLTok,
                            &full[s]);
            }
            ring_next(s, ph, nstages);
          }
        } else if (it.kind == 1) {
          // the batch-head's partial slices for this item, through the ring;
          // chunks that do not update wrote none and are skipped
          if (!wait_count(doneA + it.bh, L.n_upd * L.splits, L.status, lim)) { ok = false; break; }
          fence_proxy_async_global();
          const int E = L.dv * L.dk, per = E / L.pparts, npairs = L.nc * L.splits;
          const uint32_t sl = (uint32_t)per * 4;
          const int pps = (int)(stage_bytes / sl);
          const float* base = L.partials + (long long)it.bh * npairs * E + (long long)it.sub * per;
          for (int p0 = 0; p0 < npairs && ok; p0 += pps) {
            if (!mbar_wait(&empty[s], ph ^ 1, L.status, lim)) { ok = false; break; }
            const int n = min(pps, npairs - p0);
            uint32_t bytes = 0;
            for (int j = 0; j < n; ++j)
              if (chunk_updates(L, (p0 + j) / L.splits)) bytes += sl;
            mbar_arrive_expect_tx(&full[s], bytes);
            uint8_t* st = ring + s * stage_bytes;
            for (int j = 0; j < n; ++j)
              if (chunk_updates(L, (p0 + j) / L.splits))
                bulk_load_g2s(st + j * sl, base + (long long)(p0 + j) * E, sl, &full[s]);
            ring_next(s, ph, nstages);
          }
        } else if (it.kind == 2) {
          const int qrow0 = it.bh * L.N + it.c * L.chunk + it.sub * L.rb;
          prefetch_rows_l2(L.q + (long long)qrow0 * L.dk, (uint32_t)L.rb * L.dk * 2);
          // the state this chunk reads is written by the batch-head's P items
          if (!wait_count(doneP + it.bh, L.pparts, L.status, lim)) { ok = false; break; }
          fence_proxy_async_global();
          if (!mbar_wait(sempty, (nb & 1) ^ 1, L.status, lim)) { ok = false; break; }
          mbar_arrive_expect_tx(sfull, s_bytes);
          if (L.blocked)
            tma_load_3d(sreg, &L.maps[LM_S], 0, (it.bh * L.nc + it.c) * L.dv, 0, sfull);
          else
            for (int b = 0; b < dkb; ++b)
              tma_load_2d(sreg + b * L.dv * 128, &L.maps[LM_S], b * 64,
                          (it.bh * L.nc + it.c) * L.dv, sfull);
          ++nb;
          const int row0 = it.bh * L.N + it.c * L.chunk + it.sub * L.rb;
          for (int mt = 0; mt < L.rb / kLTok && ok; ++mt) {
            if (!mbar_wait(&empty[s], ph ^ 1, L.status, lim)) { ok = false; break; }
            mbar_arrive_expect_tx(&full[s], (uint32_t)L.dk * kLTok * 2);
            uint8_t* st = ring + s * stage_bytes;
            if (L.blocked)
              tma_load_3d(st, &L.maps[LM_Q], 0, row0 + mt * kLTok, 0, &full[s]);
            else
              for (int b = 0; b < dkb; ++b)
                tma_load_2d(st + b * 16384, &L.maps[LM_Q], b * 64, row0 + mt * kLTok, &full[s]);
            ring_next(s, ph, nstages);
          }
        }
      }
    }
  } else if (warp == 1) {
    {   // the whole warp walks the items; one elected lane issues
      int s = 0, u = 0, nb = 0;
      uint32_t ph = 0;
      bool ok = true;
      const uint32_t ring_saddr = smem_u32(ring), s_saddr = smem_u32(sreg);
      const uint32_t stage16 = stage_bytes >> 4;
      for (int i = blockIdx.x; i < total && ok; i += gridDim.x) {
        const Item it = decode_item(L, i);
        if (it.kind == 0) {
          if (!chunk_updates(L, it.c)) continue;
          const int buf = u & 1;
          if (!mbar_wait_w(&acce[buf], ((u >> 1) & 1) ^ 1, L.status, lim)) { ok = false; break; }
          tc_fence_after();
          // A = V~^T (M = d_v, K = tokens), B = K^T (N = d_k): both MN-major,
          // 64-column blocks of 128 token rows 16 KB apart
          const uint32_t idesc = idesc_bf16_f32(L.dk, 1, 1);
          const uint64_t a0 = smem_desc_sw128(ring_saddr, 16384, 1024);
          const uint64_t b0 = smem_desc_sw128(ring_saddr + dvb * 16384, 16384, 1024);
          const uint32_t d = tmem + buf * 128;
          for (int j = 0; j < L.slen / kLTok; ++j) {
            // scaled[s] completes once per A-stage use of slot s; a CTA's A
            // items all come before its B items, so its A stages fill the first
            // ring rounds and the ring phase is the barrier's phase
            if (!mbar_wait_w(&scaled[s], ph, L.status, lim)) { ok = false; break; }
            tc_fence_after();
            const uint64_t so = (uint64_t)(s * stage16);
#pragma unroll
            for (int kk = 0; kk < kLTok / 16; ++kk)   // 16 token rows = 2 KB
              umma_bf16_w(d, a0 + so + kk * 128, b0 + so + kk * 128, idesc, (j | kk) != 0);
            umma_commit_w(&empty[s]);
            ring_next(s, ph, nstages);
          }
          umma_commit_w(&accf[buf]);
          ++u;
        } else if (it.kind == 1) {   // the prefix warps consume these stages
          const int per = L.dv * L.dk / L.pparts;
          const int pps = (int)(stage_bytes / ((uint32_t)per * 4));
          for (int p0 = 0; p0 < L.nc * L.splits; p0 += pps) ring_next(s, ph, nstages);
        } else if (it.kind == 2) {
          if (!mbar_wait_w(sfull, nb & 1, L.status, lim)) { ok = false; break; }
          ++nb;
          // A = Q rows (K-major, K = d_k), B = S (K-major: N = d_v rows, K = d_k)
          const uint32_t idesc = idesc_bf16_f32(L.dv, 0, 0);
          const uint64_t a0 = smem_desc_sw128(ring_saddr, 16, 1024);
          const uint64_t b0 = smem_desc_sw128(s_saddr, 16, 1024);
          for (int mt = 0; mt < L.rb / kLTok && ok; ++mt) {
            const int buf = u & 1;
            if (!mbar_wait_w(&acce[buf], ((u >> 1) & 1) ^ 1, L.status, lim)) { ok = false; break; }
            if (!mbar_wait_w(&full[s], ph, L.status, lim)) { ok = false; break; }
            tc_fence_after();
            const uint64_t so = (uint64_t)(s * stage16);
            const uint32_t d = tmem + buf * 128;
            for (int b = 0; b < dkb; ++b) {   // 64 of K per block: A 16 KB, S d_v x 128 B apart
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_bf16_w(d, a0 + so + b * 1024 + kk * 2, b0 + b * (L.dv * 8) + kk * 2, idesc,
                          (b | kk) != 0);
            }
            umma_commit_w(&empty[s]);
            umma_commit_w(&accf[buf]);
            ring_next(s, ph, nstages);
            ++u;
          }
          umma_commit_w(sempty);
        }
      }
    }
  } else {
    // warps 2..5: row = TMEM lane of this thread.  `ok` stays uniform across
    // the warp (TMEM loads are warp-collective) and, after a failed wait, the
    // warps keep walking their items without waiting or storing, so that all
    // four reach every named barrier.
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const int tid = threadIdx.x - 64;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    int s = 0, u = 0;
    uint32_t ph = 0;
    bool ok = true;
    auto wait_uniform = [&](uint64_t* bar, uint32_t parity) {
      if (ok) ok = mbar_wait(bar, parity, L.status, lim);
      ok = __all_sync(0xffffffffu, ok);
    };
    for (int i = blockIdx.x; i < total; i += gridDim.x) {
      const Item it = decode_item(L, i);
      if (it.kind == 0) {
        if (!chunk_updates(L, it.c)) continue;
        const int tok0 = it.c * L.chunk + it.sub * L.slen;
        const float* eta = L.eta + (long long)it.bh * L.N + tok0;
        const int nst = L.slen / kLTok;
        // this thread's token-row eta for the next three stages, loaded ahead
        // (a DRAM round trip is several microseconds while the whole GPU streams)
        float e0 = eta[tid];
        float e1 = nst > 1 ? eta[kLTok + tid] : 0.f;
        float e2 = nst > 2 ? eta[2 * kLTok + tid] : 0.f;
        for (int j = 0; j < nst; ++j) {
          const float e = e0;
          e0 = e1;
          e1 = e2;
          e2 = j + 3 < nst ? eta[(j + 3) * kLTok + tid] : 0.f;
          wait_uniform(&full[s], ph);
          if (ok) {
            const uint32_t st = smem_u32(ring + s * stage_bytes) + tid * 128;
            for (int b = 0; b < dvb; ++b) {
              // the whole 128-byte row: eight 16-byte chunks loaded together, in
              // a lane-rotated order so that the 8 lanes of a shared-memory
              // phase hit 8 different chunks
              uint4 w[8];
#pragma unroll
              for (int q = 0; q < 8; ++q) w[q] = lds128(st + b * 16384 + (((q + tid) & 7) << 4));
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                uint32_t* wp = reinterpret_cast<uint32_t*>(&w[q]);
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                  const float2 f = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&wp[h]));
                  __nv_bfloat162 r = __floats2bfloat162_rn(f.x * e, f.y * e);
                  wp[h] = *reinterpret_cast<uint32_t*>(&r);
                }
              }
#pragma unroll
              for (int q = 0; q < 8; ++q) sts128(st + b * 16384 + (((q + tid) & 7) << 4), w[q]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&scaled[s]);
          }
          ring_next(s, ph, nstages);
        }
        const int buf = u & 1;
        wait_uniform(&accf[buf], (u >> 1) & 1);
        if (ok) {
          tc_fence_after();
          float* dst = L.partials +
                       ((long long)(it.bh * L.nc + it.c) * L.splits + it.sub) * L.dv * L.dk +
                       (long long)row * L.dk;
          for (int c0 = 0; c0 < L.dk; c0 += 32) {
            float v[32];
            tmem_ld32(tmem + buf * 128 + lane_off + c0, v);
            tmem_wait32(v);
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              uint32_t w[8];
#pragma unroll
              for (int q = 0; q < 8; ++q) w[q] = __float_as_uint(v[8 * h + q]);
              stg256(dst + c0 + 8 * h, w);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acce[buf]);
        }
        ++u;
        named_bar_sync(1, 128);
        if (tid == 0 && ok && it.bh != L.withhold_bh) {
          __threadfence();
          atomicAdd(doneA + it.bh, 1);
        }
      } else if (it.kind == 1) {
        const int per = L.dv * L.dk / L.pparts;
        prefix_item(L, it.bh, it.sub * per, per, tid, ring, full, empty, s, ph, ok);
        named_bar_sync(1, 128);
        if (tid == 0 && ok) {
          __threadfence();
          atomicAdd(doneP + it.bh, 1);
        }
      } else {
        const long long rowbase = (long long)it.bh * L.N + it.c * L.chunk + it.sub * L.rb;
        for (int mt = 0; mt < L.rb / kLTok; ++mt) {
          const int buf = u & 1;
          wait_uniform(&accf[buf], (u >> 1) & 1);
          if (ok) {
            tc_fence_after();
            __nv_bfloat16* dst = L.out + (rowbase + mt * kLTok + row) * L.dv;
            for (int c0 = 0; c0 < L.dv; c0 += 32) {
              float v[32];
              tmem_ld32(tmem + buf * 128 + lane_off + c0, v);
              tmem_wait32(v);
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                uint32_t w[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                  __nv_bfloat162 r =
                      __floats2bfloat162_rn(v[16 * h + 2 * q], v[16 * h + 2 * q + 1]);
                  w[q] = *reinterpret_cast<uint32_t*>(&r);
                }
                stg256(dst + c0 + 16 * h, w);
              }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[buf]);
          }
          ++u;
          ring_next(s, ph, nstages);   // keep the ring position in step (the stage is Q's)
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

int g_fused_ready[64] = {0};   // 0 unknown, 1 usable, 2 not usable
int g_fused_sms[64] = {0};
std::atomic<int> g_withhold_bh{-1};

}  // namespace

void linattn_fused_withhold_release(int bh) { g_withhold_bh.store(bh < 0 ? -1 : bh); }

bool linattn_fused_applicable(const LinDims& D) {
  if (!D.bf16) return false;
  // the state MMA has M = d_v = 128; d_k (its N) may be 64 or 128
  if ((D.dk != 64 && D.dk != 128) || D.dv != 128) return false;
  if (D.chunk % kLTok != 0 || D.N % D.chunk != 0) return false;
  if (D.N / D.chunk > kMaxFlagChunks) return false;
  // a prefix item's slice of the state (d_v d_k / 8 elements, eight items per
  // batch-head) is one pass of its 128 threads
  if (D.dv * D.dk / 8 > 4 * 128 * kPG) return false;
  return true;
}

LinFusedPlan linattn_fused_plan(const LinDims& D) {
  LinFusedPlan p;
  const int BH = D.B * D.H, nc = D.N / D.chunk;
  // token splits: enough A items for most of the SMs, split length a multiple of 128
  p.splits = 1;
  while ((long long)BH * nc * p.splits < 120 && D.chunk % (2 * p.splits * kLTok) == 0 &&
         D.chunk / (2 * p.splits) >= 512)
    p.splits *= 2;
  p.rb = D.chunk % 512 == 0 ? 512 : (D.chunk % 256 == 0 ? 256 : 128);
  p.pparts = 8;
  return p;
}

size_t linattn_fused_scratch(const LinDims& D, const LinFusedPlan& p) {
  const size_t BH = (size_t)D.B * D.H, nc = D.N / D.chunk, E = (size_t)D.dv * D.dk;
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  return al(BH * nc * p.splits * E * 4) + al(BH * nc * E * 2) + al(2 * BH * 4);
}

bool prepare_linattn_fused() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lk(setup_mutex());
  int& r = g_fused_ready[dev];
  if (r == 0) {
    r = 2;
    int coop = 0;
    if (cudaFuncSetAttribute(linattn_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kUmmaSmemBytes) == cudaSuccess &&
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess && coop &&
        cudaDeviceGetAttribute(&g_fused_sms[dev], cudaDevAttrMultiProcessorCount, dev) ==
            cudaSuccess) {
      int per_sm = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, linattn_fused_kernel, kLThreads,
                                                        kUmmaSmemBytes) == cudaSuccess &&
          per_sm >= 1)
        r = 1;
    }
    cudaGetLastError();
  }
  return r == 1;
}

int launch_linattn_fused(MapCache& cache, const LinFusedArgs& a, int* status,
                         unsigned long long wait_ns, cudaStream_t stream) {
  const LinDims& D = *a.D;
  if (!linattn_fused_applicable(D) || !prepare_linattn_fused()) return 1;
  // output rows are written with 32-byte stores
  if ((reinterpret_cast<uintptr_t>(a.out) & 31) != 0) return 1;
  int dev = 0;
  cudaGetDevice(&dev);
  const LinFusedPlan p = linattn_fused_plan(D);
  const int BH = D.B * D.H, nc = D.N / D.chunk;
  const size_t E = (size_t)D.dv * D.dk;
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  char* ws = static_cast<char*>(a.scratch);
  LinFusedLaunch L;
  std::memset(&L, 0, sizeof(L));
  L.partials = reinterpret_cast<float*>(ws);
  ws += al((size_t)BH * nc * p.splits * E * 4);
  L.s_read = reinterpret_cast<__nv_bfloat16*>(ws);
  ws += al((size_t)BH * nc * E * 2);
  L.counters = reinterpret_cast<int*>(ws);
  const TensorRef TV{a.v, 1, (long long)BH * D.N, D.dv};
  const TensorRef TK{a.k, 1, (long long)BH * D.N, D.dk};
  const TensorRef TQ{a.q, 1, (long long)BH * D.N, D.dk};
  const TensorRef TS{L.s_read, 1, (long long)BH * nc * D.dv, D.dk};
  // one box per tile where the driver takes the blocked view, else one per 64 columns
  L.blocked = cache.get_blocked(TV, kLTok, D.dv / 64, &L.maps[LM_V]) &&
              cache.get_blocked(TK, kLTok, D.dk / 64, &L.maps[LM_K]) &&
              cache.get_blocked(TQ, kLTok, D.dk / 64, &L.maps[LM_Q]) &&
              cache.get_blocked(TS, D.dv, D.dk / 64, &L.maps[LM_S]);
  if (!L.blocked &&
      (!cache.get(TV, kLTok, &L.maps[LM_V]) || !cache.get(TK, kLTok, &L.maps[LM_K]) ||
       !cache.get(TQ, kLTok, &L.maps[LM_Q]) || !cache.get(TS, D.dv, &L.maps[LM_S])))
    return -4;
  L.eta = a.eta;
  L.S0 = a.S0;
  L.s_final = a.S_final;
  L.out = static_cast<__nv_bfloat16*>(a.out);
  L.q = static_cast<const __nv_bfloat16*>(a.q);
  L.k = static_cast<const __nv_bfloat16*>(a.k);
  L.v = static_cast<const __nv_bfloat16*>(a.v);
  L.BH = BH;
  L.N = D.N;
  L.dk = D.dk;
  L.dv = D.dv;
  L.chunk = D.chunk;
  L.nc = nc;
  L.splits = p.splits;
  L.slen = D.chunk / p.splits;
  L.pparts = p.pparts;
  L.rb = p.rb;
  L.apply_first = D.mode == 0;
  L.flags = *a.flags;
  L.rule = a.rule;
  int n_upd = 0;
  for (int c = 0; c < nc; ++c)
    if (L.flags.all || ((L.flags.bits[c >> 5] >> (c & 31)) & 1u)) ++n_upd;
  L.n_upd = n_upd;
  L.nA = BH * nc * p.splits;
  L.nP = BH * p.pparts;
  L.nB = BH * nc * (D.chunk / p.rb);
  L.stage_bytes = (uint32_t)(D.dv + D.dk) * kLTok * 2;
  const int s_bytes = (int)((E * 2 + 1023) / 1024 * 1024);
  int nst = (kUmmaSmemBytes - 1024 - kLCtrl - s_bytes) / (int)L.stage_bytes;
  if (nst > kLMaxStages) nst = kLMaxStages;
  if (nst < 2) return 1;
  L.nstages = nst;
  L.status = status;
  L.wait_limit_ns = wait_ns;
  L.withhold_bh = g_withhold_bh.load();

  if (cudaMemsetAsync(L.counters, 0, 2 * (size_t)BH * sizeof(int), stream) != cudaSuccess)
    return -6;
  const int total = L.nA + L.nP + L.nB;
  const int grid = total < g_fused_sms[dev] ? total : g_fused_sms[dev];
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kLThreads, 1, 1);
  cfg.dynamicSmemBytes = kUmmaSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const double flops = 2.0 * (double)n_upd * BH * D.chunk * E + 2.0 * (double)BH * D.N * E;
  const double bytes = (double)BH * D.N * (2.0 * (D.dk * 2 + D.dv) + 4);
  ProfScope ps(PT_LIN_FUSED, stream, flops, bytes);
  if (cudaLaunchKernelEx(&cfg, linattn_fused_kernel, L) != cudaSuccess) return -6;
  return 0;
}

}  // namespace ttt
