#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "ttt_profile.h"
#include "prof.h"

namespace ttt {

namespace {

struct Rec {
  int tag;
  cudaEvent_t a, b;
  double flops, bytes, sm_share;
};

std::atomic<unsigned long long> g_launches{0};
std::mutex g_mu;
bool g_on = false;
std::vector<Rec> g_recs;

const char* kTagName[PT_COUNT] = {
    "init", "gemm.proj", "gemm.grad", "gemm.ns_gram", "gemm.ns_poly", "gemm.ns_step",
    "norm", "lin.scale", "gemm.lin_partial", "lin.prefix", "gemm.lin_out", "gemm.selftest", "muon.cluster",
    "muon.half", "lin.fused", "gemm.apply_proj", "gemm.apply_out", "gemm.featurize"};
const char* kTagKernel[PT_COUNT] = {
    "init_layer_kernel", "umma_gemm_kernel", "umma_gemm_kernel", "umma_gemm_kernel",
    "umma_gemm_kernel", "umma_gemm_kernel", "update_normalize_kernel", "scale_rows_kernel",
    "umma_gemm_kernel", "linattn_prefix_kernel", "umma_gemm_kernel", "umma_gemm_kernel",
    "ns_cluster_kernel", "ns_half_kernel", "linattn_fused_kernel",
    "umma_gemm_kernel", "umma_gemm_kernel", "umma_gemm_kernel"};

}  // namespace

bool prof_recording() {
  std::lock_guard<std::mutex> lk(g_mu);
  return g_on;
}

void prof_count_launches(size_t n) { g_launches.fetch_add(n); }

ProfScope::ProfScope(int tag, cudaStream_t s, double flops, double bytes, double sm_share)
    : idx_(-1), s_(s) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_on) return;
  Rec r;
  r.tag = tag;
  r.flops = flops;
  r.bytes = bytes;
  r.sm_share = sm_share < 1.0 ? sm_share : 1.0;
  if (cudaEventCreate(&r.a) != cudaSuccess) return;
  if (cudaEventCreate(&r.b) != cudaSuccess) {
    cudaEventDestroy(r.a);
    return;
  }
  cudaEventRecord(r.a, s);
  idx_ = (int)g_recs.size();
  g_recs.push_back(r);
}

ProfScope::~ProfScope() {
  g_launches.fetch_add(1);
  if (idx_ < 0) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (idx_ < (int)g_recs.size()) cudaEventRecord(g_recs[idx_].b, s_);
}

}  // namespace ttt

extern "C" {

unsigned long long ttt_launch_count(void) { return ttt::g_launches.load(); }

void ttt_profile_start(void) {
  std::lock_guard<std::mutex> lk(ttt::g_mu);
  for (auto& r : ttt::g_recs) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  ttt::g_recs.clear();
  ttt::g_on = true;
}

int ttt_profile_stop(ttt_profile_entry* entries, int max_entries) {
  std::lock_guard<std::mutex> lk(ttt::g_mu);
  ttt::g_on = false;
  ttt_profile_entry acc[ttt::PT_COUNT];
  std::memset(acc, 0, sizeof(acc));
  int rc = 0;
  for (auto& r : ttt::g_recs) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) rc = -6;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) rc = -6;
    acc[r.tag].launches += 1;
    acc[r.tag].ms += ms;
    acc[r.tag].flops += r.flops;
    acc[r.tag].bytes += r.bytes;
    acc[r.tag].sm_ms += ms * r.sm_share;
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  ttt::g_recs.clear();
  if (rc) return rc;
  int n = 0;
  for (int t = 0; t < ttt::PT_COUNT && n < max_entries; ++t) {
    if (!acc[t].launches) continue;
    std::strncpy(acc[t].name, ttt::kTagName[t], sizeof(acc[t].name) - 1);
    std::strncpy(acc[t].kernel, ttt::kTagKernel[t], sizeof(acc[t].kernel) - 1);
    if (entries) entries[n] = acc[t];
    ++n;
  }
  return n;
}

}  // extern "C"
