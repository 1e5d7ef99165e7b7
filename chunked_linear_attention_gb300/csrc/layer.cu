// Host orchestration of the LaCT TTT layer forward ("5.2.1 LaCT and
// TTT-E2E", eqs (2)-(6), (10) and the mask list of section 1.1).
//
// Per (batch, head) the fast weights W1, W3 [m, d] and W2 [d, m] live in fp32
// (the caller's W*_final buffers) with bf16 operand copies in the workspace.
// The chunk scan is a sequence of steps; each step applies the current
// weights to one chunk of queries and/or takes one update from one chunk of
// keys/values, with all (batch, head) pairs batched in every launch:
//
//   APPLY two launches on the apply stream: queries H1q = Q W1^T, H3q = Q W3^T
//                     -> A_q (gated), then the output O = A_q W2^T of the
//                     applied chunk (without an apply stream they join the
//                     PROJ and GRAD launches)
//   PROJ  one launch: keys     H1 = K W1^T, H3 = K W3^T, VW2 = V W2
//                              -> dH1, dH3, P (fused SiLU/SiLU' and eta)
//   GRAD  one launch: g1 = dH1^T K, g3 = dH3^T K, g2 = V^T P (eq 2; K = chunk)
//                     with momentum fused in the epilogue
//   MUON  one fused launch (or 3 launches per Newton-Schulz step) over all
//         matrices (eq 6), ending in W <- L2-Normalize(W - U) (eq 5)
//   NORM  one launch: W <- L2-Normalize(W - U) without Muon (eq 5)
//
// The bf16 operand copies of the weights alternate between two buffers, so
// that the apply side of one step can still read its weights while the
// update writes the next ones.
//
// Matrix slots: 0 = W1 [m, d], 1 = W3 [m, d], 2 = W2 [d, m]; every
// per-matrix buffer is [slot][B*H][rows*cols].
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "builder.h"
#include "layer.h"
#include "exec.h"
#include "ns_cluster.h"
#include "ns_half.h"
#include "ns_products.h"
#include "prof.h"

namespace ttt {

namespace {

// Newton-Schulz kernel for square d x d matrices: the half-panel kernel
// (d % 128 == 0, d <= 512), else the tile-cluster kernel (other square
// d <= 512), else the per-product GEMM launches.
bool use_ns_half(int d) { return ns_half_applicable(d); }

// An integer environment knob, read once (thread-safe: function-local statics
// are initialised exactly once).  `dflt` when unset or empty.
int env_int(const char* name, int dflt) {
  const char* s = std::getenv(name);
  return (s && s[0]) ? std::atoi(s) : dflt;
}

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct LayerWs {
  void* Wb[3];
  void* Wb2[3];        // second bf16 copy: the apply side reads one while the update writes the other
  void* Aq;
  void* dH1;
  void* dH3;
  void* P;
  float* M;
  float* U;
  void* X[2];
  void* G;
  void* Bm;
  float* normsq;       // [3][B*H] squared Frobenius norms of M (per-product paths)
  float* normsq_part;  // [3][B*H][nslot] their partial sums, one per gradient (tile, warp)
  int nslot;
  // static feature map (W1, W3 fixed): phi(q) and the keys' features for every token
  void* PhiQ;          // [B*H][N][m]
  void* PhiK;          // [B*H][N][m]: -eta * phi(k) (recurrent form) or -phi(k) (parallel)
  void* lin;           // parallel form: the chunked linear attention's workspace
};

// The chunked linear attention that the parallel form runs: features of
// width m as keys and queries, values of width d, state W2 [d, m].
LinDims parallel_lin_dims(const LayerDims& D) {
  LinDims L;
  L.B = D.B;
  L.H = D.H;
  L.N = D.N;
  L.dk = D.m;
  L.dv = D.d;
  L.chunk = D.chunk;
  L.bf16 = D.bf16;
  L.mode = D.mode;
  L.mom = D.beta != 0.f ? 1 : 0;
  L.muon_steps = D.muon_steps;
  L.ns[0] = D.ns[0];
  L.ns[1] = D.ns[1];
  L.ns[2] = D.ns[2];
  return L;
}

// Partial-sum slots per matrix for the gradient's squared norm: a bound on
// (output tiles) x (warps per tile) of either GEMM path (tiles at least
// 64 x 64, at most 16 warps).  Slots no tile writes stay zero.
int norm_slots(const LayerDims& D) { return ((D.d + 63) / 64) * ((D.m + 63) / 64) * 16; }

size_t layer_ws_layout(const LayerDims& D, LayerWs* w, char* base) {
  const size_t BH = (size_t)D.B * D.H;
  const size_t dm = (size_t)D.d * D.m;
  const size_t s = (size_t)std::min(D.d, D.m);
  const size_t es = D.bf16 ? 2 : 4;
  size_t off = 0;
  auto take = [&](size_t bytes) -> char* {
    char* p = base ? base + off : nullptr;
    off += align_up(bytes);
    return p;
  };
  LayerWs tmp;
  LayerWs& o = w ? *w : tmp;
  std::memset(&o, 0, sizeof(o));
  if (D.parallel) {
    // bf16 copies of W1, W3 (the feature map), the features, the linear attention
    for (int i = 0; i < 2; ++i) o.Wb[i] = D.bf16 ? take(BH * dm * 2) : nullptr;
    o.PhiQ = take(BH * D.N * D.m * es);
    o.PhiK = take(BH * D.N * D.m * es);
    o.lin = take(linattn_workspace_bytes(parallel_lin_dims(D)));
    return off;
  }
  if (D.last_only) {
    o.PhiQ = take(BH * D.N * D.m * es);
    o.PhiK = take(BH * D.N * D.m * es);
  }
  for (int i = 0; i < 3; ++i) o.Wb[i] = D.bf16 ? take(BH * dm * 2) : nullptr;
  for (int i = 0; i < 3; ++i) o.Wb2[i] = D.bf16 ? take(BH * dm * 2) : nullptr;
  if (!D.last_only) {   // per-chunk activations (the static feature map has them all)
    o.Aq = take(BH * D.chunk * D.m * es);
    o.dH1 = take(BH * D.chunk * D.m * es);
    o.dH3 = take(BH * D.chunk * D.m * es);
    o.P = take(BH * D.chunk * D.m * es);
  }
  o.M = D.beta != 0.f ? reinterpret_cast<float*>(take(3 * BH * dm * 4)) : nullptr;
  o.U = reinterpret_cast<float*>(take(3 * BH * dm * 4));
  if (D.muon_steps > 0) {
    o.X[0] = take(3 * BH * dm * es);
    o.X[1] = take(3 * BH * dm * es);
    o.G = take(3 * BH * s * s * es);
    o.Bm = take(3 * BH * s * s * es);
  } else {
    o.X[0] = o.X[1] = o.G = o.Bm = nullptr;
  }
  o.nslot = norm_slots(D);
  o.normsq = reinterpret_cast<float*>(take(3 * BH * (1 + (size_t)o.nslot) * 4));
  o.normsq_part = o.normsq ? o.normsq + 3 * BH : nullptr;
  return off;
}

// Public W index of each slot: W1 -> 0, W3 -> 2, W2 -> 1.
constexpr int kPub[3] = {0, 2, 1};

EpiDesc epi0() {
  EpiDesc e;
  std::memset(&e, 0, sizeof(e));
  e.z_div = 1;
  return e;
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
  p.epi = epi0();
  return p;
}

}  // namespace

size_t layer_workspace_bytes(const LayerDims& D) { return layer_ws_layout(D, nullptr, nullptr); }

namespace {

uint64_t fbits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return u;
}

// Everything one call enqueues, for a range [h0, h0 + nh) of (batch, head)
// sequences.  All per-(batch, head) buffers are sliced by h0; the tensor maps
// span whole tensors and are shared by every range.
struct LayerPlan {
  const LayerArgs* a;
  const LayerDims* D;
  LayerWs w;
  MatSet ms[3];
  float* mom[3];
  TensorRef Tq, Tk, Tv, TW[2][3], TAq, TdH1, TdH3, TP, TPhiQ, TPhiK;
  void* wb[2][3];   // the two bf16 copies of the weights (both the first when there is one)
  std::vector<std::pair<int, int>> steps;
  int* status;
  unsigned long long wait_ns;
};

#define TTT_CK(x)                      \
  do {                                 \
    if ((x) != cudaSuccess) return -6; \
  } while (0)

// Host-buffer calls: chunk c's inputs are on the device once in_ev[min(c,
// n_in - 1)] has completed (recorded on the host-to-device stream); a range's
// output chunks go back on its own device-to-host stream, each ordered after
// the launch that wrote it.
struct IoHooks {
  const cudaEvent_t* in_ev;
  int n_in;
  cudaStream_t d2h;
  cudaEvent_t out_ev;
};

// CTAs of each apply-side launch for `nh` sequences (TTT_APPLY_CTAS sets the
// CTAs per sequence): the persistent GEMM keeps its CTAs for the whole launch,
// so the apply side is held to a share of the SMs and the update chain finds
// the rest free, while the applies of a step must still finish within about
// one step of the chain.  Measured on the 760M-scale layer with 5 Muon steps
// (four groups of two sequences): 2, 3, 4, 6 CTAs per sequence -> 3.04, 2.90,
// 2.93, 2.95 ms per step; uncapped (152 CTAs) 3.2 ms, and 3.11 ms without the
// split.  The default share grows with the apply work per sequence and chunk
// (b d m, relative to that layer's 2048 x 384 x 384), so that a step's applies
// keep taking about as long, and as 15 / steps with fewer Muon steps, as the
// chain then gets shorter (only that layer and 5 steps measured).
int apply_ctas(int nh, int muon_steps, const LayerDims& D) {
  static const int v = std::max(0, env_int("TTT_APPLY_CTAS", 0));
  const double work = (double)D.chunk * D.d * D.m / (2048.0 * 384.0 * 384.0);
  const double per = v > 0 ? (double)v : 15.0 / muon_steps * (work > 1.0 ? work : 1.0);
  return (int)std::ceil(per * nh);
}

// The chain's GEMM launches rank one priority level below its Newton-Schulz
// launches (TTT_GEMM_PRIORITY_OFFSET=k: k levels; measured on the 760M-scale
// layer: 0, 1, 2 -> 2.92, 2.90, 2.91 ms per step).
int gemm_priority_offset() {
  static const int v = std::max(0, env_int("TTT_GEMM_PRIORITY_OFFSET", 1));
  return v;
}

// TTT_CHAIN_PRIORITY=0 launches the update chain at the streams' own priority.
bool chain_priority_on() {
  static const bool v = env_int("TTT_CHAIN_PRIORITY", 1) != 0;
  return v;
}

// The apply side of a step (query projections and the output GEMM of its
// apply chunk) depends only on that step's weights, and nothing in the scan
// depends on it.  With an apply stream `sa` it runs there, overlapping the
// update chain on `st` (projections of the keys, gradients, Newton-Schulz):
// the update writes the next weights' bf16 copy into the other of the two
// copies, and waits only until the applies that read that copy (one update
// earlier) have finished.  ApplyEvents: ev_w is recorded on `st` whenever new
// weights are complete; ev_a[c] on `sa` after the latest apply that read copy c.
struct ApplyEvents {
  cudaEvent_t ev_w;
  cudaEvent_t ev_a[2];
};

// The static feature map of the last-layer-only forms ("Test-Time Training
// with KV Binding Is Secretly Linear Attention", sec. 6.1 Step 1, App. H):
// phi(x) = SiLU(x W1^T) o (x W3^T) for every token of every sequence, in one
// launch: queries -> PhiQ, keys -> PhiK scaled by -eta per token (recurrent
// form: P of the W2 gradient, g2 = V^T P) or by -1 (parallel form: the
// linear attention's keys, so that its state increment is the gradient).
int enqueue_featurize(const LayerPlan& L, MapCache& cache, bool keys_eta, cudaStream_t st) {
  const LayerArgs& a = *L.a;
  const LayerDims& D = *L.D;
  const int BH = D.B * D.H, N = D.N, d = D.d, m = D.m;
  LaunchBuilder LB(D.bf16, &cache, L.status, L.wait_ns);
  const int BM = LB.bm();
  const int bn = LB.choose_bn(m, 2);
  for (int which = 0; which < 2; ++which) {
    Problem p = prob0(N, m, d, BH, 2, bn);
    p.a[0] = LB.op(which == 0 ? L.Tq : L.Tk, 0, 0, N, BM);
    p.b[0] = LB.op(L.TW[0][0], 0, 0, m, bn);
    p.a[1] = p.a[0];
    p.b[1] = LB.op(L.TW[0][1], 0, 0, m, bn);
    p.a_shared = 1 << 1;
    p.epi.kind = EPI_PROJ_Q;
    p.epi.out[0] = which == 0 ? L.w.PhiQ : L.w.PhiK;
    p.epi.out_ld = m;
    p.epi.out_z = (long long)N * m;
    if (which == 1) {
      if (keys_eta) {
        p.epi.eta = a.eta;
        p.epi.eta_z = N;
      } else {
        p.epi.a = -1.f;
      }
    }
    LB.add(p);
  }
  if (!LB.ok()) return -4;
  return LB.launch(st, PT_FEATURIZE) == cudaSuccess ? 0 : -6;
}

int enqueue_range(const LayerPlan& L, MapCache& cache, int h0, int nh, cudaStream_t st,
                  const IoHooks* io = nullptr,
                  cudaStream_t sa = nullptr, const ApplyEvents* aev = nullptr) {
  const LayerArgs& a = *L.a;
  const LayerDims& D = *L.D;
  const LayerWs& w = L.w;
  const bool tc = D.bf16;
  const int BH = D.B * D.H, d = D.d, m = D.m, b = D.chunk, N = D.N;
  const long long dm = (long long)d * m;
  const int rows_of[3] = {m, m, d}, cols_of[3] = {d, d, m};
  const bool muon = D.muon_steps > 0;
  const bool lo = D.last_only != 0;   // only W2 updates; features precomputed
  const size_t es = tc ? 2 : 4;
  const size_t ios = tc ? 2 : 4;
  auto offs = [&](void* p, long long elems) -> void* {
    return p ? static_cast<char*>(p) + elems * (long long)es : nullptr;
  };
  LaunchBuilder LB(tc, &cache, L.status, L.wait_ns);
  const int BM = LB.bm();
  const long long bm_h = (long long)b * m;   // activation elements per (batch, head)
  const bool split = sa != nullptr && aev != nullptr;
  // the update chain's launches go first; the apply side fills the SMs they leave
  const int prio = split && chain_priority_on() ? high_priority() : 0;
  // the chain's GEMM launches may rank one level below its Newton-Schulz launches
  const int gprio = prio < 0 ? std::min(0, prio + gemm_priority_offset()) : prio;
  int cur = 0;                           // bf16 copy holding the current weights
  bool apply_reads[2] = {false, false};  // an apply that st has not waited for reads copy c

  if (split) {   // the apply stream starts from everything enqueued on st so far
    TTT_CK(cudaEventRecord(aev->ev_w, st));
    TTT_CK(cudaStreamWaitEvent(sa, aev->ev_w, 0));
  }

  // query projections of chunk ap, appended to the launch being built
  auto add_apply_proj = [&](int ap) {
    const int bn = LB.choose_bn(m, 2);
    Problem p = prob0(b, m, d, nh, 2, bn);
    p.a[0] = LB.op(L.Tq, 0, h0 * N + ap * b, N, BM);
    p.b[0] = LB.op(L.TW[cur][0], 0, h0 * m, m, bn);
    p.a[1] = p.a[0];
    p.b[1] = LB.op(L.TW[cur][1], 0, h0 * m, m, bn);
    p.a_shared = 1 << 1;
    p.epi.kind = EPI_PROJ_Q;
    p.epi.out[0] = offs(w.Aq, h0 * bm_h);
    p.epi.out_ld = m;
    p.epi.out_z = bm_h;
    LB.add(p);
  };
  // output O = A_q W2^T of chunk ap, appended to the launch being built
  auto add_apply_out = [&](int ap) {
    const int bn = LB.choose_bn(d, 1);
    Problem p = prob0(b, d, m, nh, 1, bn);
    p.a[0] = lo ? LB.op(L.TPhiQ, 0, h0 * N + ap * b, N, BM) : LB.op(L.TAq, 0, h0 * b, b, BM);
    p.b[0] = LB.op(L.TW[cur][2], 0, h0 * d, d, bn);  // W2 [d, m]: N = d rows, K = m contiguous
    p.kd = (tc && m % 128 == 0) ? 2 : 1;   // same stage size as the gradients
    p.epi.kind = EPI_OUT;
    p.epi.out[0] = static_cast<char*>(a.out) + (long long)h0 * N * d * (long long)ios;
    p.epi.out_ld = d;
    p.epi.out_z = (long long)N * d;
    p.epi.out_row0 = (long long)ap * b;
    LB.add(p);
  };
  // this range's rows of output chunk ap are written (on stream s): copy them back
  auto copy_out = [&](int ap, cudaStream_t s) -> int {
    const size_t row = (size_t)b * d * ios, pitch = (size_t)N * d * ios;
    const size_t off = ((size_t)h0 * N + (size_t)ap * b) * d * ios;
    TTT_CK(cudaEventRecord(io->out_ev, s));
    TTT_CK(cudaStreamWaitEvent(io->d2h, io->out_ev, 0));
    TTT_CK(cudaMemcpy2DAsync(static_cast<char*>(a.host->out) + off, pitch,
                             static_cast<const char*>(a.out) + off, pitch, row, nh,
                             cudaMemcpyDeviceToHost, io->d2h));
    return 0;
  };

  int waited = -1;   // host-buffer calls: last input chunk st waited for
  for (const auto& stp : L.steps) {
    const int ap = stp.first, up = stp.second;
    const int need = split ? up : std::max(ap, up);
    if (io && need > waited) {
      waited = need;
      TTT_CK(cudaStreamWaitEvent(st, io->in_ev[std::min(waited, io->n_in - 1)], 0));
    }
    // ---------------- APPLY (own stream)
    if (split && ap >= 0) {
      TTT_CK(cudaStreamWaitEvent(sa, aev->ev_w, 0));
      if (io) TTT_CK(cudaStreamWaitEvent(sa, io->in_ev[std::min(ap, io->n_in - 1)], 0));
      if (!lo) {
        add_apply_proj(ap);
        if (!LB.ok()) return -4;
        TTT_CK(LB.launch(sa, PT_APPLY_PROJ, 0, apply_ctas(nh, D.muon_steps, D)));
      }
      add_apply_out(ap);
      if (!LB.ok()) return -4;
      TTT_CK(LB.launch(sa, PT_APPLY_OUT, 0, apply_ctas(nh, D.muon_steps, D)));
      if (io) {
        const int rc = copy_out(ap, sa);
        if (rc != 0) return rc;
      }
      TTT_CK(cudaEventRecord(aev->ev_a[cur], sa));
      apply_reads[cur] = true;
    }
    // ---------------- PROJ (not with the static feature map: P is precomputed)
    if (up >= 0 && !lo) {
      const int bn = LB.choose_bn(m, 3);
      Problem p = prob0(b, m, d, nh, 3, bn);
      p.a[0] = LB.op(L.Tk, 0, h0 * N + up * b, N, BM);
      p.b[0] = LB.op(L.TW[cur][0], 0, h0 * m, m, bn);
      p.a[1] = p.a[0];
      p.b[1] = LB.op(L.TW[cur][1], 0, h0 * m, m, bn);
      p.a[2] = LB.op(L.Tv, 0, h0 * N + up * b, N, BM);
      p.b[2] = LB.op(L.TW[cur][2], 1, h0 * d, d, bn);  // W2 [d, m]: K = d rows, N = m contiguous
      p.a_shared = 1 << 1;
      p.epi.kind = EPI_PROJ_K;
      p.epi.out[0] = offs(w.dH1, h0 * bm_h);
      p.epi.out[1] = offs(w.dH3, h0 * bm_h);
      p.epi.out[2] = offs(w.P, h0 * bm_h);
      p.epi.out_ld = m;
      p.epi.out_z = bm_h;
      p.epi.eta = a.eta + (long long)h0 * N;
      p.epi.eta_z = N;
      p.epi.eta_row0 = (long long)up * b;
      LB.add(p);
    }
    if (!split && ap >= 0 && !lo) add_apply_proj(ap);
    if (!lo && (up >= 0 || (!split && ap >= 0))) {
      if (!LB.ok()) return -4;
      TTT_CK(LB.launch(st, PT_PROJ, gprio));
    }

    // ---------------- GRAD (+ OUT)
    if (up >= 0) {
      for (int s = lo ? 2 : 0; s < 3; ++s) {
        const int M = rows_of[s], Nn = cols_of[s];
        const int bn = LB.choose_bn(Nn, 1);
        Problem p = prob0(M, Nn, b, nh, 1, bn);
        // two 64-deep K steps per stage: 16 KB MN-major boxes instead of 8 KB
        const int kdg = (tc && b % 128 == 0) ? 2 : 1;
        if (s < 2) {  // g1 = dH1^T K, g3 = dH3^T K  [m, d]
          p.a[0] = LB.op(s == 0 ? L.TdH1 : L.TdH3, 1, h0 * b, b, 64, 64 * kdg);
          p.b[0] = LB.op(L.Tk, 1, h0 * N + up * b, N, 64, 64 * kdg);
        } else {      // g2 = V^T P  [d, m]
          p.a[0] = LB.op(L.Tv, 1, h0 * N + up * b, N, 64, 64 * kdg);
          p.b[0] = lo ? LB.op(L.TPhiK, 1, h0 * N + up * b, N, 64, 64 * kdg)
                      : LB.op(L.TP, 1, h0 * b, b, 64, 64 * kdg);
        }
        p.kd = kdg;
        p.epi.kind = EPI_GRAD;
        p.epi.out_ld = Nn;
        p.epi.out_z = dm;
        p.epi.mom = L.mom[s] ? L.mom[s] + (long long)h0 * dm : nullptr;
        p.epi.a = D.beta;
        if (muon) {
          p.epi.out[1] = offs(w.X[0], (long long)s * BH * dm + h0 * dm);
          p.epi.normsq_out = w.normsq_part + ((long long)s * BH + h0) * w.nslot;
          p.epi.nslot = w.nslot;
        } else if (!L.mom[s]) {
          p.epi.out[0] = w.U + (long long)s * BH * dm + h0 * dm;
        }
        LB.add(p);
      }
    }
    if (!split && ap >= 0) add_apply_out(ap);
    if (up >= 0 || (!split && ap >= 0)) {
      if (!LB.ok()) return -4;
      TTT_CK(LB.launch(st, PT_GRAD, gprio));
    }
    if (io && !split && ap >= 0) {
      const int rc = copy_out(ap, st);
      if (rc != 0) return rc;
    }

    if (up < 0) continue;

    const int nxt = split ? cur ^ 1 : cur;   // bf16 copy this update writes
    if (split && apply_reads[nxt]) {         // the applies still reading it finish first
      TTT_CK(cudaStreamWaitEvent(st, aev->ev_a[nxt], 0));
      apply_reads[nxt] = false;
    }

    // ---------------- MUON (Newton-Schulz on M, every matrix)
    bool fused_update = false;
    if (muon && tc && d == m) {
      NsArgs na;
      na.X[0] = w.X[0];
      na.X[1] = w.X[1];
      na.G = w.G;
      na.Bm = w.Bm;
      na.U = w.U;
      na.normsq = w.normsq;
      na.normsq_part = w.normsq_part;
      na.nslot = w.nslot;
      for (int s = 0; s < 3; ++s) {
        na.W[s] = L.ms[s].master;
        na.Wb[s] = L.wb[nxt][s];
      }
      na.BH = BH;
      na.h0 = h0;
      na.nh = nh;
      na.d = d;
      na.steps = D.muon_steps;
      na.l2norm = D.l2norm;
      na.ns[0] = D.ns[0];
      na.ns[1] = D.ns[1];
      na.ns[2] = D.ns[2];
      na.priority = prio;
      na.slot0 = lo ? 2 : 0;
      na.nslots = lo ? 1 : 3;
      int rc = 1;
      if (use_ns_half(d)) rc = launch_ns_half(cache, na, L.status, L.wait_ns, st);
      if (rc == 1) {
        TTT_CK(launch_normsq_reduce(w.normsq_part, w.nslot, w.normsq, BH, h0, nh, st));
        rc = launch_ns_cluster(cache, na, L.status, L.wait_ns, st);
      }
      if (rc < 0) return rc;
      fused_update = rc == 0;
    }
    if (muon && !fused_update) {
      if (h0 != 0 || nh != BH) return -4;   // per-product path runs over all sequences
      TTT_CK(launch_normsq_reduce(w.normsq_part, w.nslot, w.normsq, BH, 0, BH, st));
      const int sdim = std::min(d, m);
      const long long ss = (long long)sdim * sdim;
      // groups of equally shaped slots: {0,1,2} if square, else {0,1} and {2}
      NsGroup groups[2];
      int gfirst[2] = {0, 2}, gcount[2] = {d == m ? 3 : 2, 1};
      int ng = d == m ? 1 : 2;
      if (lo) {   // W2 alone
        gfirst[0] = 2;
        gcount[0] = 1;
        ng = 1;
      }
      for (int g = 0; g < ng; ++g) {
        const int s0 = gfirst[g];
        NsGroup& q = groups[g];
        q.X[0] = offs(w.X[0], (long long)s0 * BH * dm);
        q.X[1] = offs(w.X[1], (long long)s0 * BH * dm);
        q.G = offs(w.G, (long long)s0 * BH * ss);
        q.Bm = offs(w.Bm, (long long)s0 * BH * ss);
        q.U = w.U + (long long)s0 * BH * dm;
        q.normsq = w.normsq + (long long)s0 * BH;
        q.Z = gcount[g] * BH;
        q.R = rows_of[s0];
        q.C = cols_of[s0];
      }
      const int rc = enqueue_ns_products(LB, groups, ng, D.muon_steps, D.ns, st);
      if (rc != 0) return rc;
    }

    // ---------------- NORM
    if (!fused_update) {
      MatSet part[3];
      for (int s = 0; s < 3; ++s) {
        const long long rc = (long long)rows_of[s] * cols_of[s];
        part[s] = L.ms[s];
        part[s].master = L.ms[s].master + h0 * rc;
        part[s].work = L.wb[nxt][s] ? static_cast<char*>(L.wb[nxt][s]) + h0 * rc * 2 : nullptr;
        part[s].update = L.ms[s].update + h0 * rc;
      }
      const int s_first = lo ? 2 : 0, ns_ = 3 - s_first;
      ProfScope ps(PT_NORM, st, 0.0, (double)ns_ * nh * dm * (4 + 4 + 4 + (tc ? 2 : 0)));
      TTT_CK(launch_update_normalize(part + s_first, ns_, nh, D.l2norm, st));
    }
    cur = nxt;
    if (split) TTT_CK(cudaEventRecord(aev->ev_w, st));
  }
  if (split) {   // join the apply stream
    TTT_CK(cudaEventRecord(aev->ev_a[0], sa));
    TTT_CK(cudaStreamWaitEvent(st, aev->ev_a[0], 0));
  }
  return 0;
}

// Sequences run one stream each (so that one sequence's latency-bound Muon
// overlaps other sequences' projections) when the whole update of a sequence
// can be enqueued per sequence: the bf16 path with square matrices under the
// cluster Newton-Schulz kernel, or without Muon.
bool per_sequence_streams(const LayerDims& D) {
  if (!D.bf16 || D.B * D.H < 2) return false;
  if (D.muon_steps == 0) return true;
  return D.d == D.m && ((use_ns_half(D.d) && prepare_ns_half(D.d)) || prepare_ns_cluster(D.d));
}

// The apply side of every step runs on its own stream per group (bf16 path);
// TTT_SPLIT_APPLY=0 keeps it in the update chain's launches instead.
bool split_apply_on() {
  static const bool v = env_int("TTT_SPLIT_APPLY", 1) != 0;
  return v;
}

// Number of stream groups the (batch, head) sequences are split into: each
// group's launches cover a contiguous range of sequences on its own stream.
// The default is four groups with the apply side on its own streams, else
// three with Muon and one without (measured on the 760M-scale layer, B*H = 8:
// split, 3 / 4 groups: 2.97 / 2.93 ms per step; unsplit, 1 to 6 groups: 4.41,
// 3.27, 3.19, 3.25, 3.26, 3.29 ms; smaller Newton-Schulz launches pack better
// between the other groups' GEMMs; without Muon 1 / 3 / 4 groups: 1.56 / 1.67
// / 1.76 ms);
// TTT_SEQUENCE_GROUPS (1 .. B*H) overrides it, and 1 runs every launch batched
// over all sequences on the caller's stream.
int sequence_groups(const LayerDims& D, bool split) {
  const int BH = D.B * D.H;
  if (!per_sequence_streams(D)) return 1;
  static const int env = env_int("TTT_SEQUENCE_GROUPS", -1);
  if (env >= 1) return env < BH ? env : BH;
  const int def = split ? 4 : (D.muon_steps > 0 ? 3 : 1);
  return BH < def ? BH : def;
}

// Host-buffer calls: chunks [c, c + n) of q, k, v and eta for every
// sequence, one strided copy per tensor (a row per sequence: n * chunk * width
// contiguous elements, pitch N * width).
int copy_in_chunks(const LayerArgs& a, const LayerDims& D, int c, int n, cudaStream_t s) {
  const HostIO& h = *a.host;
  const int BH = D.B * D.H;
  const size_t ios = D.bf16 ? 2 : 4;
  const size_t row = (size_t)n * D.chunk * D.d * ios, pitch = (size_t)D.N * D.d * ios;
  const size_t off = (size_t)c * D.chunk * D.d * ios;
  const void* src[3] = {h.q, h.k, h.v};
  const void* dst[3] = {a.q, a.k, a.v};
  for (int i = 0; i < 3; ++i) {
    if (i == 1 && h.k == h.q) continue;   // k aliases q
    TTT_CK(cudaMemcpy2DAsync(static_cast<char*>(const_cast<void*>(dst[i])) + off, pitch,
                             static_cast<const char*>(src[i]) + off, pitch, row, BH,
                             cudaMemcpyHostToDevice, s));
  }
  const size_t erow = (size_t)n * D.chunk * 4, epitch = (size_t)D.N * 4;
  TTT_CK(cudaMemcpy2DAsync(const_cast<float*>(a.eta) + (size_t)c * D.chunk, epitch,
                           h.eta + (size_t)c * D.chunk, epitch, erow, BH,
                           cudaMemcpyHostToDevice, s));
  return 0;
}

int enqueue_all(LayerPlan& L, cudaStream_t st) {
  const LayerArgs& a = *L.a;
  const LayerDims& D = *L.D;
  const LayerWs& w = L.w;
  const HostIO* hio = a.host;
  const bool tc = D.bf16;
  const int BH = D.B * D.H;
  const int nc = D.N / D.chunk;
  const long long dm = (long long)D.d * D.m;

  // streams: [0, ng) compute groups when ng > 1, then one apply stream per
  // group (bf16 device-buffer calls), then for host-buffer calls one
  // host-to-device stream and one device-to-host stream per group.  Events per
  // group: ev_w and ev_a[2] (the group's first event is spare).  Host-buffer calls keep the apply side in
  // the chain's launches: with the extra streams their input copies stalled
  // behind queued kernels (8-9 ms per call instead of 4.7 ms).  Without Muon
  // the update chain is short and the capped apply side would set the pace
  // (1.93 ms per step against 1.56 ms unsplit), so only Muon runs split.
  const bool split = tc && !hio && D.muon_steps > 0 && split_apply_on();
  int ng = sequence_groups(D, split);
  auto nstreams = [&](int g) { return (g > 1 ? g : 0) + (split ? g : 0) + (hio ? 1 + g : 0); };
  std::vector<cudaStream_t> pool;
  std::vector<cudaEvent_t> sev;
  if (ng > 1 && !(stream_pool(nstreams(ng), &pool) && stagger_events(4 * ng, &sev))) ng = 1;
  if (ng == 1 && !(stream_pool(nstreams(1), &pool) && stagger_events(4, &sev))) return -6;
  const int ap0 = ng > 1 ? ng : 0;
  const int io0 = ap0 + (split ? ng : 0);
  std::vector<ApplyEvents> aevs(ng);
  for (int g = 0; g < ng; ++g) aevs[g] = ApplyEvents{sev[4 * g + 1], {sev[4 * g + 2], sev[4 * g + 3]}};
  std::vector<IoHooks> hooks(ng);
  std::vector<cudaEvent_t> evs;        // host-buffer calls: input chunks, then one per group
  std::vector<cudaEvent_t> chunk_ev;   // event of each input chunk
  if (hio) {
    std::vector<cudaStream_t> io(pool.begin() + io0, pool.begin() + io0 + 1 + ng);
    TTT_CK(fork_streams(st, io));   // nothing overwrites staging a prior call still reads
    const size_t wrows = (size_t)(a.w_per_batch ? D.B : 1) * D.H;
    for (int s = 0; s < 3; ++s)
      TTT_CK(cudaMemcpyAsync(const_cast<float*>(a.W[s]), hio->W[s], wrows * dm * 4,
                             cudaMemcpyHostToDevice, st));
    if (hio->momentum)
      TTT_CK(cudaMemcpyAsync(a.momentum, hio->momentum, 3 * (size_t)BH * dm * 4,
                             cudaMemcpyHostToDevice, st));
    // every input chunk in order on the host-to-device stream, one event per
    // chunk (the last event also covers any chunks beyond the pool).  One
    // strided copy per tensor and chunk runs at the link's full rate; larger
    // blocks of chunks measured slower overall (the kernels wait longer for
    // the first chunks of each block).
    const int nb = std::min(nc, 4096 - ng);
    if (!io_events(nb + ng, &evs)) return -6;
    chunk_ev.assign(nc, evs[nb - 1]);
    for (int c = 0; c < nc; ++c) {
      const int rc = copy_in_chunks(a, D, c, 1, io[0]);
      if (rc != 0) return rc;
      if (c < nb - 1) {
        TTT_CK(cudaEventRecord(evs[c], io[0]));
        chunk_ev[c] = evs[c];
      }
    }
    TTT_CK(cudaEventRecord(evs[nb - 1], io[0]));
    for (int g = 0; g < ng; ++g)
      hooks[g] = IoHooks{chunk_ev.data(), nc, io[1 + g], evs[nb + g]};
  }

  {
    // weights and their bf16 copies, a zero momentum (when none is passed) and
    // the squared-norm partials, in one launch
    float* mz = (!a.momentum && w.M) ? w.M : nullptr;
    ProfScope ps(PT_INIT, st, 0.0,
                 3.0 * BH * dm * (4 + 4 + (tc ? 2 : 0)) + (mz ? 3.0 * BH * dm * 4 : 0.0) +
                     3.0 * BH * (1 + w.nslot) * 4);
    TTT_CK(launch_init_layer(L.ms, 3, D.B, D.H, mz, 3LL * BH * dm, w.normsq,
                             3LL * BH * (1 + w.nslot), st));
  }
  MapCache cache;
  if (D.last_only) {   // the static feature map's outputs for every token, once
    if (hio) TTT_CK(cudaStreamWaitEvent(st, chunk_ev[nc - 1], 0));
    const int rc = enqueue_featurize(L, cache, true, st);
    if (rc != 0) return rc;
  }
  if (ng > 1) {
    std::vector<cudaStream_t> kids(pool.begin(), pool.begin() + ng);
    TTT_CK(fork_streams(st, kids));
    // Group g covers a contiguous range of sequences on its own stream.
    for (int g = 0; g < ng; ++g) {
      const int h0 = (int)((long long)BH * g / ng), h1 = (int)((long long)BH * (g + 1) / ng);
      const int rc = enqueue_range(L, cache, h0, h1 - h0, kids[g], hio ? &hooks[g] : nullptr,
                                   split ? pool[ap0 + g] : nullptr,
                                   split ? &aevs[g] : nullptr);
      if (rc != 0) return rc;
    }
    TTT_CK(join_streams(st, kids));
  } else {
    const int rc = enqueue_range(L, cache, 0, BH, st, hio ? &hooks[0] : nullptr,
                                 split ? pool[ap0] : nullptr, split ? &aevs[0] : nullptr);
    if (rc != 0) return rc;
  }
  if (hio) {
    for (int s = 0; s < 3; ++s)
      TTT_CK(cudaMemcpyAsync(hio->Wf[s], a.Wf[s], (size_t)BH * dm * 4, cudaMemcpyDeviceToHost,
                             st));
    if (hio->momentum)
      TTT_CK(cudaMemcpyAsync(hio->momentum, a.momentum, 3 * (size_t)BH * dm * 4,
                             cudaMemcpyDeviceToHost, st));
    std::vector<cudaStream_t> io(pool.begin() + io0, pool.begin() + io0 + 1 + ng);
    TTT_CK(join_streams(st, io));
  }
  return 0;
}

// The parallel form ("Test-Time Training with KV Binding Is Secretly Linear
// Attention", sec. 6.2 and App. H; Variant 2): with W1, W3 static and no
// normalisation the W2 update is associative, so the scan becomes
//   1. the features phi(q), phi(k) of every token (one launch),
//   2. chunked linear attention with phi(q) as queries, -phi(k) as keys, v
//      and eta as values and rates, state W2 [d, m]: per updating chunk
//      M <- beta M + G with G = (eta v)^T (-phi(k)) = g2 (the W2 gradient),
//      W2 <- W2 + (-1) Muon(M) (or M), and O = W2 phi(q) in mask order.
// Host-buffer calls copy all inputs in first and the results out after.
int enqueue_parallel(LayerPlan& L, cudaStream_t st) {
  const LayerArgs& a = *L.a;
  const LayerDims& D = *L.D;
  const LayerWs& w = L.w;
  const HostIO* hio = a.host;
  const int BH = D.B * D.H;
  const long long dm = (long long)D.d * D.m;
  const size_t ios = D.bf16 ? 2 : 4;
  const size_t act = (size_t)BH * D.N * D.d * ios;
  float* mom2 = a.momentum ? a.momentum + (long long)BH * dm : nullptr;   // M2 of (M1, M2, M3)
  if (hio) {
    const void* src[3] = {hio->q, hio->k, hio->v};
    const void* dst[3] = {a.q, a.k, a.v};
    for (int i = 0; i < 3; ++i) {
      if (i == 1 && hio->k == hio->q) continue;
      TTT_CK(cudaMemcpyAsync(const_cast<void*>(dst[i]), src[i], act, cudaMemcpyHostToDevice, st));
    }
    TTT_CK(cudaMemcpyAsync(const_cast<float*>(a.eta), hio->eta, (size_t)BH * D.N * 4,
                           cudaMemcpyHostToDevice, st));
    const size_t wrows = (size_t)(a.w_per_batch ? D.B : 1) * D.H;
    for (int s = 0; s < 3; ++s)
      TTT_CK(cudaMemcpyAsync(const_cast<float*>(a.W[s]), hio->W[s], wrows * dm * 4,
                             cudaMemcpyHostToDevice, st));
    if (hio->momentum)
      TTT_CK(cudaMemcpyAsync(a.momentum, hio->momentum, 3 * (size_t)BH * dm * 4,
                             cudaMemcpyHostToDevice, st));
  }
  {
    // final weights = initial ones (W1, W3 stay; W2 is the linear attention's
    // initial state), bf16 copies of W1 and W3 for the feature map
    MatSet ms[3];
    for (int s = 0; s < 3; ++s) {
      ms[s] = L.ms[s];
      ms[s].work = s < 2 ? w.Wb[s] : nullptr;
    }
    ProfScope ps(PT_INIT, st, 0.0, 3.0 * BH * dm * (4 + 4) + 2.0 * BH * dm * (D.bf16 ? 2 : 0));
    TTT_CK(launch_init_layer(ms, 3, D.B, D.H, nullptr, 0, nullptr, 0, st));
  }
  MapCache cache;
  int rc = enqueue_featurize(L, cache, false, st);
  if (rc != 0) return rc;
  LinDims LD = parallel_lin_dims(D);
  LD.mom = (D.beta != 0.f || mom2) ? 1 : 0;
  LinArgs la;
  la.q = w.PhiQ;
  la.k = w.PhiK;
  la.v = a.v;
  la.eta = a.eta;
  la.S0 = a.Wf[1];
  la.update_chunks = a.update_chunks;
  la.out = a.out;
  la.S_final = a.Wf[1];
  la.workspace = w.lin;
  la.stream = st;
  la.M0 = mom2;
  la.M_final = mom2;
  la.alpha_const = D.beta;
  la.lr_const = -1.f;
  rc = linattn_forward(la, LD, L.status, L.wait_ns);
  if (rc != 0) return rc;
  if (hio) {
    TTT_CK(cudaMemcpyAsync(hio->out, a.out, act, cudaMemcpyDeviceToHost, st));
    for (int s = 0; s < 3; ++s)
      TTT_CK(cudaMemcpyAsync(hio->Wf[s], a.Wf[s], (size_t)BH * dm * 4, cudaMemcpyDeviceToHost,
                             st));
    if (hio->momentum)
      TTT_CK(cudaMemcpyAsync(hio->momentum, a.momentum, 3 * (size_t)BH * dm * 4,
                             cudaMemcpyDeviceToHost, st));
  }
  return 0;
}

#undef TTT_CK

}  // namespace

int layer_forward(const LayerArgs& a, const LayerDims& D, int* status,
                  unsigned long long wait_ns) {
  LayerPlan L;
  L.a = &a;
  L.D = &D;
  L.status = status;
  L.wait_ns = wait_ns;
  layer_ws_layout(D, &L.w, static_cast<char*>(a.workspace));
  const LayerWs& w = L.w;
  const bool tc = D.bf16;
  const int BH = D.B * D.H, d = D.d, m = D.m, b = D.chunk, N = D.N;
  const long long dm = (long long)d * m;
  const int nc = N / b;
  const int rows_of[3] = {m, m, d}, cols_of[3] = {d, d, m};
  const bool muon = D.muon_steps > 0;

  for (int s = 0; s < 3; ++s) {
    L.ms[s].init = a.W[kPub[s]];
    L.ms[s].init_per_batch = a.w_per_batch;
    L.ms[s].master = a.Wf[kPub[s]];
    L.ms[s].work = tc ? w.Wb[s] : nullptr;
    L.ms[s].rows = rows_of[s];
    L.ms[s].cols = cols_of[s];
    if (a.momentum)
      L.mom[s] = a.momentum + (long long)kPub[s] * BH * dm;
    else
      L.mom[s] = w.M ? w.M + (long long)s * BH * dm : nullptr;
    float* u_slot = w.U + (long long)s * BH * dm;
    L.ms[s].update = (!muon && L.mom[s]) ? L.mom[s] : u_slot;
  }
  const int wb16 = tc ? 1 : 0;
  L.Tq = TensorRef{a.q, wb16, (long long)BH * N, d};
  L.Tk = TensorRef{a.k, wb16, (long long)BH * N, d};
  L.Tv = TensorRef{a.v, wb16, (long long)BH * N, d};
  for (int s = 0; s < 3; ++s) {
    L.wb[0][s] = tc ? w.Wb[s] : nullptr;
    L.wb[1][s] = tc ? w.Wb2[s] : nullptr;
    for (int c = 0; c < 2; ++c)
      L.TW[c][s] = TensorRef{tc ? L.wb[c][s] : static_cast<const void*>(a.Wf[kPub[s]]), wb16,
                             (long long)BH * rows_of[s], cols_of[s]};
  }
  if (D.last_only) {   // W1, W3 never change: both bf16 copies are the first
    L.wb[1][0] = L.wb[0][0];
    L.wb[1][1] = L.wb[0][1];
    for (int s = 0; s < 2; ++s)
      L.TW[1][s] = L.TW[0][s];
  }
  L.TPhiQ = TensorRef{w.PhiQ, wb16, (long long)BH * N, m};
  L.TPhiK = TensorRef{w.PhiK, wb16, (long long)BH * N, m};
  L.TAq = TensorRef{w.Aq, wb16, (long long)BH * b, m};
  L.TdH1 = TensorRef{w.dH1, wb16, (long long)BH * b, m};
  L.TdH3 = TensorRef{w.dH3, wb16, (long long)BH * b, m};
  L.TP = TensorRef{w.P, wb16, (long long)BH * b, m};

  // step schedule: (apply chunk, update chunk), -1 = none
  std::vector<uint64_t> flagbits((nc + 63) / 64, 0);
  // (inner_steps > 1: the update of a chunk repeated on the same chunk, the
  // apply reading the weights before the first (apply-then-update) or after
  // the last repetition)
  if (D.mode == 0) {
    for (int c = 0; c < nc; ++c) {
      L.steps.push_back({c, c});
      for (int r = 1; r < D.inner_steps; ++r) L.steps.push_back({-1, c});
    }
  } else {
    std::vector<int> pending;
    for (int c = 0; c < nc; ++c) {
      const bool upd = D.mode != 3 || (a.update_chunks && a.update_chunks[c]);
      if (upd) flagbits[c / 64] |= 1ull << (c % 64);
      if (upd) {
        while (pending.size() > 1) {
          L.steps.push_back({pending.front(), -1});
          pending.erase(pending.begin());
        }
        L.steps.push_back({pending.empty() ? -1 : pending.front(), c});
        for (int r = 1; r < D.inner_steps; ++r) L.steps.push_back({-1, c});
        pending.assign(1, c);
      } else {
        pending.push_back(c);
      }
    }
    for (int p : pending) L.steps.push_back({p, -1});
  }

  // every argument the launch sequence depends on
  std::vector<uint64_t> key = {
      0x7474746c61796572ull,  // call kind
      (uint64_t)a.q, (uint64_t)a.k, (uint64_t)a.v, (uint64_t)a.eta,
      (uint64_t)a.W[0], (uint64_t)a.W[1], (uint64_t)a.W[2], (uint64_t)a.w_per_batch,
      (uint64_t)a.out, (uint64_t)a.Wf[0], (uint64_t)a.Wf[1], (uint64_t)a.Wf[2],
      (uint64_t)a.momentum, (uint64_t)a.workspace,
      (uint64_t)D.B, (uint64_t)D.H, (uint64_t)D.N, (uint64_t)D.d, (uint64_t)D.m,
      (uint64_t)D.chunk, (uint64_t)D.bf16, (uint64_t)D.mode, (uint64_t)D.l2norm,
      (uint64_t)D.muon_steps, fbits(D.beta),
      fbits(D.ns[0]), fbits(D.ns[1]),
      fbits(D.ns[2]), (uint64_t)status, (uint64_t)wait_ns, (uint64_t)D.last_only,
      (uint64_t)D.inner_steps, (uint64_t)D.parallel};
  key.insert(key.end(), flagbits.begin(), flagbits.end());
  if (a.host) {   // host-buffer call: the host tensors too
    const HostIO& h = *a.host;
    const void* hp[11] = {h.q, h.k, h.v, h.eta, h.W[0], h.W[1], h.W[2],
                          h.out, h.Wf[0], h.Wf[1], h.Wf[2]};
    key.push_back(0x686f7374ull);
    for (const void* p : hp) key.push_back((uint64_t)p);
    key.push_back((uint64_t)h.momentum);
  }
  // one-time device setup outside any capture
  high_priority();
  if (D.parallel) {   // a few launches; the linear attention's own setup runs on the way
    if (tc && prepare_umma_gemm() != cudaSuccess) return -6;
    return enqueue_parallel(L, a.stream);
  }
  if (tc) {
    if (prepare_umma_gemm() != cudaSuccess) return -6;
    if (muon && d == m) {
      if (use_ns_half(d)) prepare_ns_half(d);
      prepare_ns_cluster(d);
    }
  }
  return run_cached(key, a.stream, [&](cudaStream_t s) { return enqueue_all(L, s); });
}

}  // namespace ttt
