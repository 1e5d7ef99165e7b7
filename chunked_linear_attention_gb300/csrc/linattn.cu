// Host orchestration of chunked linear attention ("Test-Time Training with KV
// Binding Is Secretly Linear Attention", Thm 5.2 and App. H with alpha = 0;
// the causal state update of "From Linear Attention to Test-Time Training").
//
// The state after chunk c is S0 + sum over visible chunks of V~_c^T K_c with
// V~ = eta * V.  The chunk sums are independent, so the scan is three
// parallel passes over all (batch, head, chunk) at once:
//   1. V~ = eta * V (bf16 rows), then per (batch, head, chunk, split) the
//      partial state V~_split^T K_split on the tensor cores (K = split tokens)
//   2. a prefix over chunks: the state each chunk reads (bf16 operand copy)
//      and the final fp32 state
//   3. O_c = Q_c S_c^T on the tensor cores, all chunks in one launch.
#include <algorithm>
#include <cstring>

#include "builder.h"
#include "launch.h"
#include "layer.h"
#include "linattn_fused.h"
#include "linattn_kernels.h"
#include "ns_half.h"
#include "ns_products.h"
#include "prof.h"

namespace ttt {

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Token splits of each chunk's state sum: enough tiles for one wave over the
// SMs, each split at least 512 tokens and a multiple of 128 (two 64-deep K
// steps per pipeline stage); fewer splits also mean fewer fp32 partials for
// the prefix pass to read.
int choose_splits(const LinDims& D, int tiles_per_z) {
  const long long pairs = (long long)D.B * D.H * (D.N / D.chunk);
  int splits = 1;
  while (pairs * splits * tiles_per_z < 152) {
    const int next = splits * 2;
    if (D.chunk % next != 0) break;
    const int len = D.chunk / next;
    if (len < 512 || len % 128 != 0) break;
    splits = next;
  }
  return splits;
}

struct LinWs {
  void* Vt;
  float* partials;
  void* Sread;
  int splits;
  // Muon of the momentum (one matrix per update of every sequence)
  void* X[2];
  void* G;
  void* Bm;
  float* U;
  void* Ub;            // bf16 copy the half-panel kernel writes beside U (unused)
  float* normsq;
  float* norm_part;
  int nslot;
};

size_t lin_layout(const LinDims& D, LinWs* w, char* base) {
  const size_t BH = (size_t)D.B * D.H;
  const size_t nc = D.N / D.chunk;
  const size_t es = D.bf16 ? 2 : 4;
  const int tiles = D.bf16 ? ((D.dv + 127) / 128) * ((D.dk + 127) / 128)
                           : ((D.dv + 63) / 64) * ((D.dk + 63) / 64);
  const int splits = choose_splits(D, tiles);
  size_t off = 0;
  auto take = [&](size_t bytes) -> char* {
    char* p = base ? base + off : nullptr;
    off += align_up(bytes);
    return p;
  };
  LinWs tmp;
  LinWs& o = w ? *w : tmp;
  o.splits = splits;
  o.Vt = take(BH * D.N * D.dv * es);
  o.partials = reinterpret_cast<float*>(take(BH * nc * splits * D.dv * D.dk * 4));
  o.Sread = take(BH * nc * D.dv * D.dk * es);
  o.nslot = linattn_momentum_slots(D.dv * D.dk);
  if (D.muon_steps > 0) {   // sized for every chunk updating
    const size_t Z = BH * nc, E = (size_t)D.dv * D.dk, sm = std::min(D.dv, D.dk);
    o.X[0] = take(Z * E * es);
    o.X[1] = take(Z * E * es);
    o.G = take(Z * sm * sm * es);
    o.Bm = take(Z * sm * sm * es);
    o.U = reinterpret_cast<float*>(take(Z * E * 4));
    o.Ub = take(Z * E * 2);
    o.normsq = reinterpret_cast<float*>(take(Z * 4));
    o.norm_part = reinterpret_cast<float*>(take(Z * o.nslot * 4));
  } else {
    o.X[0] = o.X[1] = o.G = o.Bm = o.Ub = nullptr;
    o.U = o.normsq = o.norm_part = nullptr;
  }
  return off;
}

Problem prob0(int M, int N, int K, int Z, int nacc, int bn) {
  Problem p;
  std::memset(&p, 0, sizeof(p));
  p.M = M;
  p.N = N;
  p.K = K;
  p.Z = Z;
  p.nacc = nacc;
  p.bn = bn;
  p.epi.z_div = 1;
  return p;
}

}  // namespace

// Room for either path: the one-launch kernel where it applies, the
// multi-launch path otherwise (and as the fallback on devices without
// cooperative launch).
size_t linattn_workspace_bytes(const LinDims& D) {
  size_t n = lin_layout(D, nullptr, nullptr);
  if (D.muon_steps == 0 && linattn_fused_applicable(D))
    n = std::max(n, linattn_fused_scratch(D, linattn_fused_plan(D)));
  return n;
}

int linattn_forward(const LinArgs& a, const LinDims& D, int* status, unsigned long long wait_ns) {
  cudaStream_t st = a.stream;
  const bool tc = D.bf16;
  const int BH = D.B * D.H, N = D.N, dk = D.dk, dv = D.dv, b = D.chunk;
  const int nc = N / b;
  const int wb16 = tc ? 1 : 0;

  UpdateFlags flags;
  std::memset(&flags, 0, sizeof(flags));
  flags.all = D.mode != 3;
  int n_upd = nc;
  if (D.mode == 3) {
    n_upd = 0;
    for (int c = 0; c < nc; ++c)
      if (a.update_chunks[c]) {
        flags.bits[c >> 5] |= 1u << (c & 31);
        ++n_upd;
      }
  }
  LinRule rule;
  rule.alpha = a.alpha;
  rule.lr = a.lr;
  rule.M0 = a.M0;
  rule.M_final = a.M_final;
  rule.mom = D.mom;
  rule.alpha_const = a.alpha_const;
  rule.lr_const = a.lr_const;
  const bool muon = D.muon_steps > 0;

  if (!muon && linattn_fused_applicable(D)) {
    MapCache fcache;
    LinFusedArgs fa;
    fa.D = &D;
    fa.q = a.q;
    fa.k = a.k;
    fa.v = a.v;
    fa.eta = a.eta;
    fa.S0 = a.S0;
    fa.flags = &flags;
    fa.rule = rule;
    fa.out = a.out;
    fa.S_final = a.S_final;
    fa.scratch = a.workspace;
    const int rc = launch_linattn_fused(fcache, fa, status, wait_ns, st);
    if (rc <= 0) return rc;
  }

  LinWs w;
  lin_layout(D, &w, static_cast<char*>(a.workspace));
  const int splits = w.splits, slen = b / splits;
  {
    const size_t es = tc ? 2 : 4;
    ProfScope ps(PT_LIN_SCALE, st, 0.0, (double)BH * N * (dv * es * 2 + 4));
    if (launch_scale_rows(a.v, a.eta, w.Vt, (long long)BH * N, dv, tc, st) != cudaSuccess)
      return -6;
  }

  MapCache cache;
  LaunchBuilder LB(tc, &cache, status, wait_ns);
  const int BM = LB.bm();
  TensorRef TVt{w.Vt, wb16, (long long)BH * N, dv};
  TensorRef Tk{a.k, wb16, (long long)BH * N, dk};
  TensorRef Tq{a.q, wb16, (long long)BH * N, dk};
  TensorRef TS{w.Sread, wb16, (long long)BH * nc * dv, dk};

  {  // partial states
    const int bn = LB.choose_bn(dk, 1);
    Problem p = prob0(dv, dk, slen, BH * nc * splits, 1, bn);
    // MN-major operands (token rows): 16 KB boxes of 128 K rows when the split allows
    const int kd = (tc && slen % 128 == 0) ? 2 : 1;
    p.a[0] = LB.op(TVt, 1, 0, slen, 64, 64 * kd);
    p.b[0] = LB.op(Tk, 1, 0, slen, 64, 64 * kd);
    p.kd = kd;
    p.epi.kind = EPI_STORE_F32;
    p.epi.out[0] = w.partials;
    p.epi.out_ld = dk;
    p.epi.out_z = (long long)dv * dk;
    LB.add(p);
    if (!LB.ok()) return -4;
    if (LB.launch(st, PT_LIN_PARTIAL) != cudaSuccess) return -6;
  }
  const int dvdk = dv * dk;
  if (!muon) {
    ProfScope ps(PT_LIN_PREFIX, st, 0.0,
                 (double)BH * nc * dvdk * (4.0 * splits + (tc ? 2 : 4)));
    if (launch_linattn_prefix(w.partials, a.S0, w.Sread, a.S_final, BH, nc, splits, dvdk,
                              D.mode == 0, flags, rule, 0, n_upd, tc, st) != cudaSuccess)
      return -6;
  } else if (n_upd == 0) {   // nothing updates: every chunk reads S0
    LinRule none;
    if (launch_linattn_prefix(w.partials, a.S0, w.Sread, a.S_final, BH, nc, splits, dvdk,
                              D.mode == 0, flags, none, 0, 0, tc, st) != cudaSuccess)
      return -6;
    if (a.M_final && launch_copy_f32(a.M_final, a.M0, (long long)BH * dvdk, st) != cudaSuccess)
      return -6;
  } else {
    // Muon of every update's momentum ("Test-Time Training with KV Binding Is
    // Secretly Linear Attention", App. E.3): the momenta M_u of all updates
    // at once, their squared norms, the Newton-Schulz products over all of
    // them, then the state prefix of lr_c Muon(M_u)
    {
      ProfScope ps(PT_LIN_PREFIX, st, 0.0, (double)BH * nc * dvdk * (4.0 * splits + (tc ? 2 : 4)));
      if (launch_linattn_momentum(w.partials, splits, rule, w.X[0], w.norm_part, BH, nc, n_upd,
                                  dvdk, flags, tc, st) != cudaSuccess)
        return -6;
    }
    const int Z = BH * n_upd;
    float sign = 1.f;
    int rc = 1;
    if (tc && dv == dk && ns_half_applicable(dv) && prepare_ns_half(dv)) {
      // all updates through the half-panel cluster kernel: its update step
      // W <- W - Muon(M) without normalisation, over a zeroed fp32 W, leaves
      // -Muon(M_u) in U (its bf16 copy goes to Ub)
      if (cudaMemsetAsync(w.U, 0, (size_t)Z * dvdk * 4, st) != cudaSuccess) return -6;
      NsArgs na;
      na.X[0] = w.X[0];
      na.X[1] = w.X[1];
      na.G = w.G;
      na.Bm = w.Bm;
      na.U = nullptr;
      na.normsq = w.normsq;
      na.normsq_part = w.norm_part;
      na.nslot = w.nslot;
      for (int s = 0; s < 3; ++s) {
        na.W[s] = w.U;
        na.Wb[s] = w.Ub;
      }
      na.BH = Z;
      na.d = dv;
      na.steps = D.muon_steps;
      na.l2norm = 0;
      na.h0 = 0;
      na.nh = Z;
      for (int i = 0; i < 3; ++i) na.ns[i] = D.ns[i];
      na.slot0 = 0;
      na.nslots = 1;
      na.zcount = Z;
      MapCache ncache;
      rc = launch_ns_half(ncache, na, status, wait_ns, st);
      if (rc < 0) return rc;
      if (rc == 0) sign = -1.f;
    }
    if (rc != 0) {   // the per-product launches
      if (launch_normsq_sum(w.norm_part, w.nslot, w.normsq, Z, st) != cudaSuccess) return -6;
      NsGroup g;
      g.X[0] = w.X[0];
      g.X[1] = w.X[1];
      g.G = w.G;
      g.Bm = w.Bm;
      g.U = w.U;
      g.normsq = w.normsq;
      g.Z = Z;
      g.R = dv;
      g.C = dk;
      LB.reset();
      rc = enqueue_ns_products(LB, &g, 1, D.muon_steps, D.ns, st);
      if (rc != 0) return rc;
    }
    LinRule upd_rule;
    upd_rule.lr = a.lr;
    upd_rule.lr_const = a.lr_const;
    upd_rule.inc_scale = sign;
    ProfScope ps(PT_LIN_PREFIX, st, 0.0, (double)BH * nc * dvdk * (4.0 + (tc ? 2 : 4)));
    if (launch_linattn_prefix(w.U, a.S0, w.Sread, a.S_final, BH, nc, 1, dvdk, D.mode == 0, flags,
                              upd_rule, 1, n_upd, tc, st) != cudaSuccess)
      return -6;
  }
  {  // outputs
    const int bn = LB.choose_bn(dv, 1);
    Problem p = prob0(b, dv, dk, BH * nc, 1, bn);
    p.a[0] = LB.op(Tq, 0, 0, b, BM);
    p.b[0] = LB.op(TS, 0, 0, dv, bn);
    p.kd = (tc && dk % 128 == 0) ? 2 : 1;   // one 128-deep stage per tile for dk = 128
    p.epi.kind = EPI_OUT;
    p.epi.out[0] = a.out;
    p.epi.out_ld = dv;
    p.epi.out_z = (long long)b * dv;
    LB.add(p);
    if (!LB.ok()) return -4;
    if (LB.launch(st, PT_LIN_OUT) != cudaSuccess) return -6;
  }
  return 0;
}

int selftest_gemm(const void* A, const void* Bp, float* Dp, int Z, int M, int N, int K, int a_mn,
                  int b_mn, bool bf16, int tile_n, cudaStream_t stream, int* status,
                  unsigned long long wait_ns) {
  MapCache cache;
  LaunchBuilder LB(bf16, &cache, status, wait_ns);
  const int wb16 = bf16 ? 1 : 0;
  const int bn = bf16 ? tile_n : kSimtTile;
  // A: K-major [Z*M, K] or MN-major [Z*K, M]; B: K-major [Z*N, K] or [Z*K, N]
  TensorRef TA = a_mn ? TensorRef{A, wb16, (long long)Z * K, M} : TensorRef{A, wb16, (long long)Z * M, K};
  TensorRef TB = b_mn ? TensorRef{Bp, wb16, (long long)Z * K, N} : TensorRef{Bp, wb16, (long long)Z * N, K};
  Problem p = prob0(M, N, K, Z, 1, bn);
  p.a[0] = LB.op(TA, a_mn, 0, a_mn ? K : M, LB.bm());
  p.b[0] = LB.op(TB, b_mn, 0, b_mn ? K : N, bn);
  p.epi.kind = EPI_STORE_F32;
  p.epi.out[0] = Dp;
  p.epi.out_ld = N;
  p.epi.out_z = (long long)M * N;
  LB.add(p);
  if (!LB.ok()) return -4;
  return LB.launch(stream, PT_SELFTEST) == cudaSuccess ? 0 : -6;
}

}  // namespace ttt
