#include "ns_products.h"

#include <algorithm>
#include <cstring>

#include "prof.h"

namespace ttt {

namespace {

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

int enqueue_ns_products(LaunchBuilder& LB, const NsGroup* groups, int ngroups, int steps,
                        const float ns[3], cudaStream_t st) {
  if (ngroups < 1 || ngroups > 2) return -4;
  const bool tc = LB.tensor_cores();
  const int wb16 = tc ? 1 : 0;
  const int BM = LB.bm();
  for (int t = 0; t < steps; ++t) {
    const int in = t & 1;
    const bool last = t == steps - 1;
    // GRAM: G = X X^T (or X^T X for tall matrices), scaled on the first step
    for (int g = 0; g < ngroups; ++g) {
      const NsGroup& q = groups[g];
      const int R = q.R, C = q.C, s = std::min(R, C);
      TensorRef TX{q.X[in], wb16, (long long)q.Z * R, C};
      const int bn = LB.choose_bn(s, 1);
      Problem p = prob0(s, s, std::max(R, C), q.Z, 1, bn);
      if (R <= C) {
        p.a[0] = LB.op(TX, 0, 0, R, BM);
        p.b[0] = LB.op(TX, 0, 0, R, bn);
      } else {
        p.a[0] = LB.op(TX, 1, 0, R, 64);
        p.b[0] = LB.op(TX, 1, 0, R, 64);
      }
      p.epi.kind = EPI_NS_GRAM;
      p.epi.out[0] = q.G;
      p.epi.out_ld = s;
      p.epi.out_z = (long long)s * s;
      p.epi.first = t == 0;
      p.epi.normsq = const_cast<float*>(q.normsq);
      p.epi.eps = 1e-7f;
      LB.add(p);
    }
    if (!LB.ok()) return -4;
    if (LB.launch(st, PT_NS_GRAM) != cudaSuccess) return -6;
    // POLY: Bm = b G + c G G (G symmetric)
    for (int g = 0; g < ngroups; ++g) {
      const NsGroup& q = groups[g];
      const int s = std::min(q.R, q.C);
      TensorRef TG{q.G, wb16, (long long)q.Z * s, s};
      const int bn = LB.choose_bn(s, 1);
      Problem p = prob0(s, s, s, q.Z, 1, bn);
      p.a[0] = LB.op(TG, 0, 0, s, BM);
      p.b[0] = LB.op(TG, 0, 0, s, bn);
      p.epi.kind = EPI_NS_POLY;
      p.epi.in0 = TG.ptr;
      p.epi.out[0] = q.Bm;
      p.epi.out_ld = s;
      p.epi.out_z = (long long)s * s;
      p.epi.b = ns[1];
      p.epi.c = ns[2];
      LB.add(p);
    }
    if (!LB.ok()) return -4;
    if (LB.launch(st, PT_NS_POLY) != cudaSuccess) return -6;
    // STEP: X' = s (a X + Bm X) (or X Bm for tall matrices, in stored orientation)
    for (int g = 0; g < ngroups; ++g) {
      const NsGroup& q = groups[g];
      const int R = q.R, C = q.C, s = std::min(R, C);
      TensorRef TX{q.X[in], wb16, (long long)q.Z * R, C};
      TensorRef TB{q.Bm, wb16, (long long)q.Z * s, s};
      const int bn = LB.choose_bn(C, 1);
      Problem p = prob0(R, C, s, q.Z, 1, bn);
      if (R <= C) {
        p.a[0] = LB.op(TB, 0, 0, s, BM);
        p.b[0] = LB.op(TX, 1, 0, R, 64);
      } else {
        p.a[0] = LB.op(TX, 0, 0, R, BM);
        p.b[0] = LB.op(TB, 0, 0, s, bn);
      }
      p.epi.kind = EPI_NS_STEP;
      p.epi.in0 = TX.ptr;
      if (last)
        p.epi.out[1] = q.U;
      else
        p.epi.out[0] = q.X[in ^ 1];
      p.epi.out_ld = C;
      p.epi.out_z = (long long)R * C;
      p.epi.a = ns[0];
      p.epi.first = t == 0;
      p.epi.normsq = const_cast<float*>(q.normsq);
      p.epi.eps = 1e-7f;
      LB.add(p);
    }
    if (!LB.ok()) return -4;
    if (LB.launch(st, PT_NS_STEP) != cudaSuccess) return -6;
  }
  return 0;
}

}  // namespace ttt
