// Host orchestration of the LaCT TTT layer forward ("5.2.1 LaCT and
// TTT-E2E", eqs (2)-(6), (10) and the mask list of section 1.1).
//
// Per (batch, head) the fast weights W1, W3 [m, d] and W2 [d, m] live in fp32
// (the caller's W*_final buffers) with bf16 operand copies in the workspace.
// The chunk scan is a sequence of steps; each step applies the current
// weights to one chunk of queries and/or takes one update from one chunk of
// keys/values, with all (batch, head) pairs batched in every launch:
//
//   PROJ  one launch: queries  H1q = Q W1^T, H3q = Q W3^T -> A_q (gated)
//                     keys     H1 = K W1^T, H3 = K W3^T, VW2 = V W2
//                              -> dH1, dH3, P (fused SiLU/SiLU' and eta)
//   GRAD  one launch: g1 = dH1^T K, g3 = dH3^T K, g2 = V^T P (eq 2; K = chunk)
//                     with momentum fused in the epilogue, and the output
//                     O = A_q W2^T of the applied chunk
//   MUON  3 launches per Newton-Schulz step over all matrices (eq 6)
//   NORM  one launch: W <- L2-Normalize(W - U), refresh bf16 copies (eq 5)
//
// Matrix slots: 0 = W1 [m, d], 1 = W3 [m, d], 2 = W2 [d, m]; every
// per-matrix buffer is [slot][B*H][rows*cols].
#include <algorithm>
#include <cstring>
#include <vector>

#include "builder.h"
#include "layer.h"
#include "ns_cluster.h"
#include "prof.h"

namespace ttt {

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct LayerWs {
  void* Wb[3];
  void* Aq;
  void* dH1;
  void* dH3;
  void* P;
  float* M;
  float* U;
  void* X[2];
  void* G;
  void* Bm;
  float* normsq;
};

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
  for (int i = 0; i < 3; ++i) o.Wb[i] = D.bf16 ? take(BH * dm * 2) : nullptr;
  o.Aq = take(BH * D.chunk * D.m * es);
  o.dH1 = take(BH * D.chunk * D.m * es);
  o.dH3 = take(BH * D.chunk * D.m * es);
  o.P = take(BH * D.chunk * D.m * es);
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
  o.normsq = reinterpret_cast<float*>(take(3 * BH * 4));
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

int layer_forward(const LayerArgs& a, const LayerDims& D, int* status,
                  unsigned long long wait_ns) {
  LayerWs w;
  layer_ws_layout(D, &w, static_cast<char*>(a.workspace));
  cudaStream_t st = a.stream;
  const bool tc = D.bf16;
  const int BH = D.B * D.H, d = D.d, m = D.m, b = D.chunk, N = D.N;
  const long long dm = (long long)d * m;
  const int nc = N / b;
  const int rows_of[3] = {m, m, d}, cols_of[3] = {d, d, m};
  const bool muon = D.muon_steps > 0;
  cudaError_t ce;
#define TTT_CK(x)                   \
  do {                              \
    ce = (x);                       \
    if (ce != cudaSuccess) return -6; \
  } while (0)

  // ---- state init
  MatSet ms[3];
  for (int s = 0; s < 3; ++s) {
    ms[s].init = a.W[kPub[s]];
    ms[s].init_per_batch = a.w_per_batch;
    ms[s].master = a.Wf[kPub[s]];
    ms[s].work = tc ? w.Wb[s] : nullptr;
    ms[s].rows = rows_of[s];
    ms[s].cols = cols_of[s];
    ProfScope ps(PT_INIT, st, 0.0, (double)BH * rows_of[s] * cols_of[s] * (4 + 4 + (tc ? 2 : 0)));
    TTT_CK(launch_init_weights(ms[s], D.B, D.H, st));
  }
  float* mom[3];
  for (int s = 0; s < 3; ++s) {
    if (a.momentum)
      mom[s] = a.momentum + (long long)kPub[s] * BH * dm;
    else
      mom[s] = w.M ? w.M + (long long)s * BH * dm : nullptr;
  }
  if (!a.momentum && w.M) {
    ProfScope ps(PT_INIT, st, 0.0, 3.0 * BH * dm * 4);
    TTT_CK(launch_copy_f32(w.M, nullptr, 3LL * BH * dm, st));
  }
  {
    ProfScope ps(PT_INIT, st, 0.0, 3.0 * BH * 4);
    TTT_CK(launch_copy_f32(w.normsq, nullptr, 3LL * BH, st));
  }
  for (int s = 0; s < 3; ++s) {
    float* u_slot = w.U + (long long)s * BH * dm;
    ms[s].update = (!muon && mom[s]) ? mom[s] : u_slot;
  }

  // ---- tensor views
  const int wb16 = tc ? 1 : 0;
  const size_t es = tc ? 2 : 4;
  TensorRef Tq{a.q, wb16, (long long)BH * N, d};
  TensorRef Tk{a.k, wb16, (long long)BH * N, d};
  TensorRef Tv{a.v, wb16, (long long)BH * N, d};
  TensorRef TW[3];
  for (int s = 0; s < 3; ++s)
    TW[s] = TensorRef{tc ? w.Wb[s] : static_cast<const void*>(a.Wf[kPub[s]]), wb16,
                      (long long)BH * rows_of[s], cols_of[s]};
  TensorRef TAq{w.Aq, wb16, (long long)BH * b, m};
  TensorRef TdH1{w.dH1, wb16, (long long)BH * b, m};
  TensorRef TdH3{w.dH3, wb16, (long long)BH * b, m};
  TensorRef TP{w.P, wb16, (long long)BH * b, m};

  MapCache cache;
  LaunchBuilder LB(tc, &cache, status, wait_ns);
  const int BM = LB.bm();

  // ---- step schedule: (apply chunk, update chunk), -1 = none
  std::vector<std::pair<int, int>> steps;
  if (D.mode == 0) {
    for (int c = 0; c < nc; ++c) steps.push_back({c, c});
  } else {
    std::vector<int> pending;
    for (int c = 0; c < nc; ++c) {
      const bool upd = D.mode != 3 || (a.update_chunks && a.update_chunks[c]);
      if (upd) {
        while (pending.size() > 1) {
          steps.push_back({pending.front(), -1});
          pending.erase(pending.begin());
        }
        steps.push_back({pending.empty() ? -1 : pending.front(), c});
        pending.assign(1, c);
      } else {
        pending.push_back(c);
      }
    }
    for (int p : pending) steps.push_back({p, -1});
  }

  for (const auto& stp : steps) {
    const int ap = stp.first, up = stp.second;
    // ---------------- PROJ
    if (up >= 0) {
      const int bn = LB.choose_bn(m, 3);
      Problem p = prob0(b, m, d, BH, 3, bn);
      p.a[0] = LB.op(Tk, 0, up * b, N, BM);
      p.b[0] = LB.op(TW[0], 0, 0, m, bn);
      p.a[1] = p.a[0];
      p.b[1] = LB.op(TW[1], 0, 0, m, bn);
      p.a[2] = LB.op(Tv, 0, up * b, N, BM);
      p.b[2] = LB.op(TW[2], 1, 0, d, bn);  // W2 [d, m]: K = d rows, N = m contiguous
      p.a_shared = 1 << 1;
      p.epi.kind = EPI_PROJ_K;
      p.epi.out[0] = w.dH1;
      p.epi.out[1] = w.dH3;
      p.epi.out[2] = w.P;
      p.epi.out_ld = m;
      p.epi.out_z = (long long)b * m;
      p.epi.eta = a.eta;
      p.epi.eta_z = N;
      p.epi.eta_row0 = (long long)up * b;
      LB.add(p);
    }
    if (ap >= 0) {
      const int bn = LB.choose_bn(m, 2);
      Problem p = prob0(b, m, d, BH, 2, bn);
      p.a[0] = LB.op(Tq, 0, ap * b, N, BM);
      p.b[0] = LB.op(TW[0], 0, 0, m, bn);
      p.a[1] = p.a[0];
      p.b[1] = LB.op(TW[1], 0, 0, m, bn);
      p.a_shared = 1 << 1;
      p.epi.kind = EPI_PROJ_Q;
      p.epi.out[0] = w.Aq;
      p.epi.out_ld = m;
      p.epi.out_z = (long long)b * m;
      LB.add(p);
    }
    if (!LB.ok()) return -4;
    TTT_CK(LB.launch(st, PT_PROJ));

    // ---------------- GRAD (+ OUT)
    if (up >= 0) {
      for (int s = 0; s < 3; ++s) {
        const int M = rows_of[s], Nn = cols_of[s];
        const int bn = LB.choose_bn(Nn, 1);
        Problem p = prob0(M, Nn, b, BH, 1, bn);
        if (s < 2) {  // g1 = dH1^T K, g3 = dH3^T K  [m, d]
          p.a[0] = LB.op(s == 0 ? TdH1 : TdH3, 1, 0, b, 64);
          p.b[0] = LB.op(Tk, 1, up * b, N, 64);
        } else {      // g2 = V^T P  [d, m]
          p.a[0] = LB.op(Tv, 1, up * b, N, 64);
          p.b[0] = LB.op(TP, 1, 0, b, 64);
        }
        p.epi.kind = EPI_GRAD;
        p.epi.out_ld = Nn;
        p.epi.out_z = dm;
        p.epi.mom = mom[s];
        p.epi.a = D.beta;
        if (muon) {
          p.epi.out[1] = static_cast<char*>(w.X[0]) + (size_t)s * BH * dm * es;
          p.epi.normsq_out = w.normsq + (long long)s * BH;
        } else if (!mom[s]) {
          p.epi.out[0] = w.U + (long long)s * BH * dm;
        }
        LB.add(p);
      }
    }
    if (ap >= 0) {
      const int bn = LB.choose_bn(d, 1);
      Problem p = prob0(b, d, m, BH, 1, bn);
      p.a[0] = LB.op(TAq, 0, 0, b, BM);
      p.b[0] = LB.op(TW[2], 0, 0, d, bn);  // W2 [d, m]: N = d rows, K = m contiguous
      p.epi.kind = EPI_OUT;
      p.epi.out[0] = a.out;
      p.epi.out_ld = d;
      p.epi.out_z = (long long)N * d;
      p.epi.out_row0 = (long long)ap * b;
      LB.add(p);
    }
    if (!LB.ok()) return -4;
    TTT_CK(LB.launch(st, PT_GRAD));

    if (up < 0) continue;

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
      for (int s = 0; s < 3; ++s) {
        na.W[s] = ms[s].master;
        na.Wb[s] = ms[s].work;
      }
      na.BH = BH;
      na.d = d;
      na.steps = D.muon_steps;
      na.l2norm = D.l2norm;
      na.ns[0] = D.ns[0];
      na.ns[1] = D.ns[1];
      na.ns[2] = D.ns[2];
      const int rc = launch_ns_cluster(cache, na, status, wait_ns, st);
      if (rc < 0) return rc;
      fused_update = rc == 0;
    }
    if (muon && !fused_update) {
      const int sdim = std::min(d, m);
      // groups of equally shaped slots: {0,1,2} if square, else {0,1} and {2}
      int groups[2][2];  // first slot, count
      int ng = 0;
      if (d == m) {
        groups[0][0] = 0; groups[0][1] = 3; ng = 1;
      } else {
        groups[0][0] = 0; groups[0][1] = 2; groups[1][0] = 2; groups[1][1] = 1; ng = 2;
      }
      for (int t = 0; t < D.muon_steps; ++t) {
        const int in = t & 1;
        const bool last = t == D.muon_steps - 1;
        // GRAM: G = X X^T (or X^T X for tall slots), scaled on the first step
        for (int g = 0; g < ng; ++g) {
          const int s0 = groups[g][0], cnt = groups[g][1];
          const int R = rows_of[s0], C = cols_of[s0];
          const int Z = cnt * BH;
          TensorRef TX{static_cast<char*>(w.X[in]) + (size_t)s0 * BH * dm * es, wb16,
                       (long long)Z * R, C};
          const int bn = LB.choose_bn(sdim, 1);
          Problem p = prob0(sdim, sdim, std::max(R, C), Z, 1, bn);
          if (R <= C) {
            p.a[0] = LB.op(TX, 0, 0, R, BM);
            p.b[0] = LB.op(TX, 0, 0, R, bn);
          } else {
            p.a[0] = LB.op(TX, 1, 0, R, 64);
            p.b[0] = LB.op(TX, 1, 0, R, 64);
          }
          p.epi.kind = EPI_NS_GRAM;
          p.epi.out[0] = static_cast<char*>(w.G) + (size_t)s0 * BH * sdim * sdim * es;
          p.epi.out_ld = sdim;
          p.epi.out_z = (long long)sdim * sdim;
          p.epi.first = t == 0;
          p.epi.normsq = w.normsq + (long long)s0 * BH;
          p.epi.eps = 1e-7f;
          LB.add(p);
        }
        if (!LB.ok()) return -4;
        TTT_CK(LB.launch(st, PT_NS_GRAM));
        // POLY: Bm = b G + c G G (G symmetric)
        for (int g = 0; g < ng; ++g) {
          const int s0 = groups[g][0], cnt = groups[g][1];
          const int Z = cnt * BH;
          TensorRef TG{static_cast<char*>(w.G) + (size_t)s0 * BH * sdim * sdim * es, wb16,
                       (long long)Z * sdim, sdim};
          const int bn = LB.choose_bn(sdim, 1);
          Problem p = prob0(sdim, sdim, sdim, Z, 1, bn);
          p.a[0] = LB.op(TG, 0, 0, sdim, BM);
          p.b[0] = LB.op(TG, 0, 0, sdim, bn);
          p.epi.kind = EPI_NS_POLY;
          p.epi.in0 = TG.ptr;
          p.epi.out[0] = static_cast<char*>(w.Bm) + (size_t)s0 * BH * sdim * sdim * es;
          p.epi.out_ld = sdim;
          p.epi.out_z = (long long)sdim * sdim;
          p.epi.b = D.ns[1];
          p.epi.c = D.ns[2];
          LB.add(p);
        }
        if (!LB.ok()) return -4;
        TTT_CK(LB.launch(st, PT_NS_POLY));
        // STEP: X' = s (a X + Bm X) (or X Bm for tall slots, in stored orientation)
        for (int g = 0; g < ng; ++g) {
          const int s0 = groups[g][0], cnt = groups[g][1];
          const int R = rows_of[s0], C = cols_of[s0];
          const int Z = cnt * BH;
          TensorRef TX{static_cast<char*>(w.X[in]) + (size_t)s0 * BH * dm * es, wb16,
                       (long long)Z * R, C};
          TensorRef TB{static_cast<char*>(w.Bm) + (size_t)s0 * BH * sdim * sdim * es, wb16,
                       (long long)Z * sdim, sdim};
          const int bn = LB.choose_bn(C, 1);
          Problem p = prob0(R, C, sdim, Z, 1, bn);
          if (R <= C) {
            p.a[0] = LB.op(TB, 0, 0, sdim, BM);
            p.b[0] = LB.op(TX, 1, 0, R, 64);
          } else {
            p.a[0] = LB.op(TX, 0, 0, R, BM);
            p.b[0] = LB.op(TB, 0, 0, sdim, bn);
          }
          p.epi.kind = EPI_NS_STEP;
          p.epi.in0 = TX.ptr;
          if (last)
            p.epi.out[1] = w.U + (long long)s0 * BH * dm;
          else
            p.epi.out[0] = static_cast<char*>(w.X[in ^ 1]) + (size_t)s0 * BH * dm * es;
          p.epi.out_ld = C;
          p.epi.out_z = dm;
          p.epi.a = D.ns[0];
          p.epi.first = t == 0;
          p.epi.normsq = w.normsq + (long long)s0 * BH;
          p.epi.eps = 1e-7f;
          LB.add(p);
        }
        if (!LB.ok()) return -4;
        TTT_CK(LB.launch(st, PT_NS_STEP));
      }
    }

    // ---------------- NORM
    if (!fused_update) {
      ProfScope ps(PT_NORM, st, 0.0, 3.0 * BH * dm * (4 + 4 + 4 + (tc ? 2 : 0)));
      TTT_CK(launch_update_normalize(ms, 3, BH, D.l2norm, muon ? w.normsq : nullptr,
                                     muon ? 3 * BH : 0, st));
    }
  }
#undef TTT_CK
  return 0;
}

}  // namespace ttt
