// The extern "C" boundary: argument validation (on the host, before anything
// is enqueued), the device status word, and dispatch to the orchestration.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "ttt.h"
#include "ttt_selftest.h"
#include "layer.h"
#include "linattn_fused.h"

namespace {

__device__ int g_ttt_status = 0;

unsigned long long g_wait_limit_ns = 2000000000ull;

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices] = {nullptr};
std::mutex g_status_mu;

// Device address of the status word for the current device (looked up once).
int* status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_status_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_ttt_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  return g_status_ptr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const char* x = static_cast<const char*>(a);
  const char* y = static_cast<const char*>(b);
  return x < y + nb && y < x + na;
}

int check_layer(int B, int H, int N, int d, int m, int chunk, int io, int mode,
                const ttt_update_rule* rule, ttt::LayerDims* D) {
  if (!rule) return TTT_ERR_NULL;
  if (B <= 0 || H <= 0 || N <= 0 || d <= 0 || m <= 0 || chunk <= 0) return TTT_ERR_SHAPE;
  if (N % chunk != 0) return TTT_ERR_SHAPE;
  if (mode < 0 || mode > 3) return TTT_ERR_ARG;
  if (mode == TTT_BIDIRECTIONAL && chunk != N) return TTT_ERR_SHAPE;
  if (io != TTT_F32 && io != TTT_BF16) return TTT_ERR_ARG;
  if (rule->l2norm != 0 && rule->l2norm != 1) return TTT_ERR_ARG;
  if (rule->muon_steps < 0 || rule->muon_steps > 64) return TTT_ERR_ARG;
  if (!std::isfinite(rule->momentum_beta) || !std::isfinite(rule->ns_a) ||
      !std::isfinite(rule->ns_b) || !std::isfinite(rule->ns_c))
    return TTT_ERR_ARG;
  if (rule->last_layer_only != 0 && rule->last_layer_only != 1) return TTT_ERR_ARG;
  if (rule->inner_steps < 0 || rule->inner_steps > 64) return TTT_ERR_ARG;
  if (rule->form < TTT_FORM_AUTO || rule->form > TTT_FORM_PARALLEL) return TTT_ERR_ARG;
  const bool exact_parallel =
      rule->last_layer_only == 1 && rule->l2norm == 0 && rule->inner_steps <= 1;
  if (rule->form == TTT_FORM_PARALLEL && !exact_parallel) return TTT_ERR_ARG;
  if (d > 1024 || m > 1024) return TTT_ERR_UNSUPPORTED;
  if (io == TTT_BF16 && (d % 64 != 0 || m % 64 != 0 || chunk % 128 != 0))
    return TTT_ERR_UNSUPPORTED;
  if ((long long)B * H * N > (1LL << 31) - 1) return TTT_ERR_UNSUPPORTED;
  D->B = B; D->H = H; D->N = N; D->d = d; D->m = m; D->chunk = chunk;
  D->bf16 = io == TTT_BF16;
  D->mode = mode;
  D->l2norm = rule->l2norm;
  D->muon_steps = rule->muon_steps;
  D->beta = rule->momentum_beta;
  D->ns[0] = rule->ns_a; D->ns[1] = rule->ns_b; D->ns[2] = rule->ns_c;
  D->last_only = rule->last_layer_only;
  D->inner_steps = rule->inner_steps < 1 ? 1 : rule->inner_steps;
  D->parallel = exact_parallel && rule->form != TTT_FORM_RECURRENT;
  if (D->parallel && io == TTT_BF16 && (d > 512 || m > 512)) return TTT_ERR_UNSUPPORTED;
  if (D->parallel && mode == TTT_STRIDED && N / chunk > 2048) return TTT_ERR_UNSUPPORTED;
  return TTT_OK;
}

int check_lin(int B, int H, int N, int dk, int dv, int chunk, int io, int mode,
              ttt::LinDims* D) {
  if (B <= 0 || H <= 0 || N <= 0 || dk <= 0 || dv <= 0 || chunk <= 0) return TTT_ERR_SHAPE;
  if (N % chunk != 0) return TTT_ERR_SHAPE;
  if (mode < 0 || mode > 3) return TTT_ERR_ARG;
  if (mode == TTT_BIDIRECTIONAL && chunk != N) return TTT_ERR_SHAPE;
  if (io != TTT_F32 && io != TTT_BF16) return TTT_ERR_ARG;
  if (io == TTT_BF16 && (dk % 64 != 0 || dv % 64 != 0 || dk > 512 || dv > 512 ||
                         chunk % 128 != 0))
    return TTT_ERR_UNSUPPORTED;
  if (io == TTT_F32 && (dk > 1024 || dv > 1024)) return TTT_ERR_UNSUPPORTED;
  if (mode == TTT_STRIDED && N / chunk > 2048) return TTT_ERR_UNSUPPORTED;
  if ((long long)B * H * N > (1LL << 31) - 1) return TTT_ERR_UNSUPPORTED;
  D->B = B; D->H = H; D->N = N; D->dk = dk; D->dv = dv; D->chunk = chunk;
  D->bf16 = io == TTT_BF16;
  D->mode = mode;
  return TTT_OK;
}

// Device staging of a host-buffer layer call, after the layer workspace
// (byte offsets into the workspace, 256-byte aligned; room for a separate k
// and for the momentum whether or not the call uses them).
struct HostStaging {
  size_t q, k, v, eta, W[3], out, Wf[3], mom, total;
};

HostStaging host_staging(const ttt::LayerDims& D, int w_per_batch) {
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t ios = D.bf16 ? 2 : 4, BH = (size_t)D.B * D.H, dm = (size_t)D.d * D.m;
  const size_t act = BH * D.N * D.d * ios;
  HostStaging h;
  size_t off = al(ttt::layer_workspace_bytes(D));
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += al(bytes);
    return o;
  };
  h.q = take(act);
  h.k = take(act);
  h.v = take(act);
  h.eta = take(BH * D.N * 4);
  for (int i = 0; i < 3; ++i) h.W[i] = take((w_per_batch ? BH : (size_t)D.H) * dm * 4);
  h.out = take(act);
  for (int i = 0; i < 3; ++i) h.Wf[i] = take(BH * dm * 4);
  h.mom = take(3 * BH * dm * 4);
  h.total = off;
  return h;
}

// True if p lies in page-locked host memory (allocated or registered with CUDA).
bool host_pinned(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeHost;
}

}  // namespace

extern "C" {

const char* ttt_status_string(int status) {
  switch (status) {
    case TTT_OK: return "ok";
    case TTT_ERR_NULL: return "a required pointer is NULL";
    case TTT_ERR_SHAPE: return "inconsistent sizes";
    case TTT_ERR_ALIGN: return "pointer not 16-byte aligned (workspace: 256-byte)";
    case TTT_ERR_UNSUPPORTED: return "request not supported by this library";
    case TTT_ERR_WORKSPACE: return "workspace missing or too small";
    case TTT_ERR_CUDA: return "CUDA runtime error";
    case TTT_ERR_TIMEOUT: return "a kernel's bounded wait ran out";
    case TTT_ERR_ARG: return "argument value out of range";
    case TTT_ERR_PAGEABLE: return "host buffer not page-locked";
    default: return "unknown status";
  }
}

void ttt_set_wait_limit_ns(unsigned long long ns) { g_wait_limit_ns = ns ? ns : 1; }

size_t ttt_layer_workspace_size(int B, int H, int N, int d_h, int m_h, int chunk, int io_dtype,
                                int mask_mode, const ttt_update_rule* rule) {
  ttt::LayerDims D;
  if (check_layer(B, H, N, d_h, m_h, chunk, io_dtype, mask_mode, rule, &D) != TTT_OK) return 0;
  return ttt::layer_workspace_bytes(D);
}

int ttt_layer_forward(const void* q, const void* k, const void* v, const float* eta,
                      const float* W1, const float* W2, const float* W3, int w_per_batch,
                      int B, int H, int N, int d_h, int m_h, int chunk, int io_dtype,
                      int mask_mode, const unsigned char* update_chunks,
                      const ttt_update_rule* rule, void* out, float* W1_final, float* W2_final,
                      float* W3_final, float* momentum, void* workspace, size_t workspace_bytes,
                      ttt_stream_t stream) {
  if (!q || !k || !v || !eta || !W1 || !W2 || !W3 || !out || !W1_final || !W2_final ||
      !W3_final || !rule)
    return TTT_ERR_NULL;
  ttt::LayerDims D;
  int rc = check_layer(B, H, N, d_h, m_h, chunk, io_dtype, mask_mode, rule, &D);
  if (rc != TTT_OK) return rc;
  if (w_per_batch != 0 && w_per_batch != 1) return TTT_ERR_ARG;
  if (mask_mode == TTT_STRIDED && !update_chunks) return TTT_ERR_NULL;
  const void* ptrs[] = {q, k, v, eta, W1, W2, W3, out, W1_final, W2_final, W3_final, momentum};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return TTT_ERR_ALIGN;
  const size_t need = ttt::layer_workspace_bytes(D);
  if (!workspace || workspace_bytes < need) return TTT_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return TTT_ERR_ALIGN;
  if (!w_per_batch) {
    const size_t wbytes = (size_t)H * d_h * m_h * 4;
    const size_t fbytes = (size_t)B * H * d_h * m_h * 4;
    const float* ins[3] = {W1, W2, W3};
    const float* outs[3] = {W1_final, W2_final, W3_final};
    for (const float* i : ins)
      for (const float* o : outs)
        if (overlap(i, wbytes, o, fbytes)) return TTT_ERR_ARG;
  }
  int* st = status_ptr();
  if (!st) return TTT_ERR_CUDA;
  ttt::LayerArgs a;
  a.q = q; a.k = k; a.v = v; a.eta = eta;
  a.W[0] = W1; a.W[1] = W2; a.W[2] = W3;
  a.w_per_batch = w_per_batch;
  a.update_chunks = update_chunks;
  a.out = out;
  a.Wf[0] = W1_final; a.Wf[1] = W2_final; a.Wf[2] = W3_final;
  a.momentum = momentum;
  a.workspace = workspace;
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  return ttt::layer_forward(a, D, st, g_wait_limit_ns);
}

size_t ttt_layer_host_workspace_size(int B, int H, int N, int d_h, int m_h, int chunk,
                                     int io_dtype, int mask_mode, const ttt_update_rule* rule,
                                     int w_per_batch) {
  ttt::LayerDims D;
  if (check_layer(B, H, N, d_h, m_h, chunk, io_dtype, mask_mode, rule, &D) != TTT_OK) return 0;
  if (w_per_batch != 0 && w_per_batch != 1) return 0;
  return host_staging(D, w_per_batch).total;
}

int ttt_layer_forward_host(const void* q, const void* k, const void* v, const float* eta,
                           const float* W1, const float* W2, const float* W3, int w_per_batch,
                           int B, int H, int N, int d_h, int m_h, int chunk, int io_dtype,
                           int mask_mode, const unsigned char* update_chunks,
                           const ttt_update_rule* rule, void* out, float* W1_final,
                           float* W2_final, float* W3_final, float* momentum, void* workspace,
                           size_t workspace_bytes, ttt_stream_t stream) {
  if (!q || !k || !v || !eta || !W1 || !W2 || !W3 || !out || !W1_final || !W2_final ||
      !W3_final || !rule)
    return TTT_ERR_NULL;
  ttt::LayerDims D;
  int rc = check_layer(B, H, N, d_h, m_h, chunk, io_dtype, mask_mode, rule, &D);
  if (rc != TTT_OK) return rc;
  if (w_per_batch != 0 && w_per_batch != 1) return TTT_ERR_ARG;
  if (mask_mode == TTT_STRIDED && !update_chunks) return TTT_ERR_NULL;
  const void* hptrs[] = {q, k, v, eta, W1, W2, W3, out, W1_final, W2_final, W3_final, momentum};
  for (const void* p : hptrs)
    if (p && !host_pinned(p)) return TTT_ERR_PAGEABLE;
  const HostStaging hs = host_staging(D, w_per_batch);
  if (!workspace || workspace_bytes < hs.total) return TTT_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return TTT_ERR_ALIGN;
  int* st = status_ptr();
  if (!st) return TTT_ERR_CUDA;
  char* ws = static_cast<char*>(workspace);
  ttt::HostIO h;
  h.q = q; h.k = k; h.v = v; h.eta = eta;
  h.W[0] = W1; h.W[1] = W2; h.W[2] = W3;
  h.out = out;
  h.Wf[0] = W1_final; h.Wf[1] = W2_final; h.Wf[2] = W3_final;
  h.momentum = momentum;
  ttt::LayerArgs a;
  a.q = ws + hs.q;
  a.k = k == q ? a.q : ws + hs.k;
  a.v = ws + hs.v;
  a.eta = reinterpret_cast<const float*>(ws + hs.eta);
  for (int i = 0; i < 3; ++i) {
    a.W[i] = reinterpret_cast<const float*>(ws + hs.W[i]);
    a.Wf[i] = reinterpret_cast<float*>(ws + hs.Wf[i]);
  }
  a.w_per_batch = w_per_batch;
  a.update_chunks = update_chunks;
  a.out = ws + hs.out;
  a.momentum = momentum ? reinterpret_cast<float*>(ws + hs.mom) : nullptr;
  a.workspace = workspace;
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  a.host = &h;
  return ttt::layer_forward(a, D, st, g_wait_limit_ns);
}

size_t linattn_workspace_size(int B, int H, int N, int d_k, int d_v, int chunk, int io_dtype,
                              int mask_mode) {
  ttt::LinDims D;
  if (check_lin(B, H, N, d_k, d_v, chunk, io_dtype, mask_mode, &D) != TTT_OK) return 0;
  return ttt::linattn_workspace_bytes(D);
}

int linattn_chunked_forward(const void* q, const void* k, const void* v, const float* eta,
                            const float* S0, int B, int H, int N, int d_k, int d_v, int chunk,
                            int io_dtype, int mask_mode, const unsigned char* update_chunks,
                            void* out, float* S_final, void* workspace, size_t workspace_bytes,
                            ttt_stream_t stream) {
  if (!q || !k || !v || !eta || !out) return TTT_ERR_NULL;
  ttt::LinDims D;
  int rc = check_lin(B, H, N, d_k, d_v, chunk, io_dtype, mask_mode, &D);
  if (rc != TTT_OK) return rc;
  if (mask_mode == TTT_STRIDED && !update_chunks) return TTT_ERR_NULL;
  const void* ptrs[] = {q, k, v, eta, S0, out, S_final};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return TTT_ERR_ALIGN;
  const size_t need = ttt::linattn_workspace_bytes(D);
  if (!workspace || workspace_bytes < need) return TTT_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return TTT_ERR_ALIGN;
  int* st = status_ptr();
  if (!st) return TTT_ERR_CUDA;
  ttt::LinArgs a;
  a.q = q; a.k = k; a.v = v; a.eta = eta; a.S0 = S0;
  a.update_chunks = update_chunks;
  a.out = out;
  a.S_final = S_final;
  a.workspace = workspace;
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  return ttt::linattn_forward(a, D, st, g_wait_limit_ns);
}

}  // extern "C"

namespace {

// Validates a linear-attention rule and fills the dims/args fields it sets.
int apply_lin_rule(const linattn_rule* rule, ttt::LinDims* D, ttt::LinArgs* a) {
  if (!rule) return TTT_OK;
  if (rule->muon_steps < 0 || rule->muon_steps > 64) return TTT_ERR_ARG;
  if (rule->muon_steps > 0 &&
      (!std::isfinite(rule->ns_a) || !std::isfinite(rule->ns_b) || !std::isfinite(rule->ns_c)))
    return TTT_ERR_ARG;
  if ((rule->alpha && (reinterpret_cast<uintptr_t>(rule->alpha) & 3)) ||
      (rule->lr && (reinterpret_cast<uintptr_t>(rule->lr) & 3)) ||
      (rule->M0 && !aligned16(rule->M0)) || (rule->M_final && !aligned16(rule->M_final)))
    return TTT_ERR_ALIGN;
  D->mom = (rule->alpha || rule->M0 || rule->M_final) ? 1 : 0;
  D->muon_steps = rule->muon_steps;
  D->ns[0] = rule->ns_a;
  D->ns[1] = rule->ns_b;
  D->ns[2] = rule->ns_c;
  if (a) {
    a->alpha = rule->alpha;
    a->lr = rule->lr;
    a->M0 = rule->M0;
    a->M_final = rule->M_final;
  }
  return TTT_OK;
}

}  // namespace

extern "C" {

size_t linattn_rule_workspace_size(int B, int H, int N, int d_k, int d_v, int chunk, int io_dtype,
                                   int mask_mode, const linattn_rule* rule) {
  ttt::LinDims D;
  if (check_lin(B, H, N, d_k, d_v, chunk, io_dtype, mask_mode, &D) != TTT_OK) return 0;
  if (apply_lin_rule(rule, &D, nullptr) != TTT_OK) return 0;
  return ttt::linattn_workspace_bytes(D);
}

int linattn_chunked_forward_rule(const void* q, const void* k, const void* v, const float* eta,
                                 const float* S0, int B, int H, int N, int d_k, int d_v,
                                 int chunk, int io_dtype, int mask_mode,
                                 const unsigned char* update_chunks, const linattn_rule* rule,
                                 void* out, float* S_final, void* workspace,
                                 size_t workspace_bytes, ttt_stream_t stream) {
  if (!q || !k || !v || !eta || !out) return TTT_ERR_NULL;
  ttt::LinDims D;
  int rc = check_lin(B, H, N, d_k, d_v, chunk, io_dtype, mask_mode, &D);
  if (rc != TTT_OK) return rc;
  if (mask_mode == TTT_STRIDED && !update_chunks) return TTT_ERR_NULL;
  const void* ptrs[] = {q, k, v, eta, S0, out, S_final};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return TTT_ERR_ALIGN;
  ttt::LinArgs a;
  rc = apply_lin_rule(rule, &D, &a);
  if (rc != TTT_OK) return rc;
  const size_t need = ttt::linattn_workspace_bytes(D);
  if (!workspace || workspace_bytes < need) return TTT_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return TTT_ERR_ALIGN;
  int* st = status_ptr();
  if (!st) return TTT_ERR_CUDA;
  a.q = q; a.k = k; a.v = v; a.eta = eta; a.S0 = S0;
  a.update_chunks = update_chunks;
  a.out = out;
  a.S_final = S_final;
  a.workspace = workspace;
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  return ttt::linattn_forward(a, D, st, g_wait_limit_ns);
}

int ttt_device_status(ttt_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return TTT_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_ttt_status, sizeof(int)) != cudaSuccess) return TTT_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_ttt_status, &zero, sizeof(int)) != cudaSuccess) return TTT_ERR_CUDA;
  return v;
}

int ttt_selftest_gemm(const void* A, const void* B, float* D, int Z, int M, int N, int K,
                      int a_mn_major, int b_mn_major, int dtype, int tile_n,
                      ttt_stream_t stream) {
  if (!A || !B || !D) return TTT_ERR_NULL;
  if (Z <= 0 || M <= 0 || N <= 0 || K <= 0) return TTT_ERR_SHAPE;
  if (dtype != TTT_F32 && dtype != TTT_BF16) return TTT_ERR_ARG;
  if (dtype == TTT_BF16) {
    if (M % 64 || N % 64 || K % 64) return TTT_ERR_UNSUPPORTED;
    if (tile_n != 64 && tile_n != 128 && tile_n != 192 && tile_n != 256) return TTT_ERR_ARG;
    if (!aligned16(A) || !aligned16(B) || !aligned16(D)) return TTT_ERR_ALIGN;
  }
  int* st = status_ptr();
  if (!st) return TTT_ERR_CUDA;
  return ttt::selftest_gemm(A, B, D, Z, M, N, K, a_mn_major ? 1 : 0, b_mn_major ? 1 : 0,
                            dtype == TTT_BF16, tile_n, reinterpret_cast<cudaStream_t>(stream), st,
                            g_wait_limit_ns);
}

void ttt_selftest_withhold_release(int bh) { ttt::linattn_fused_withhold_release(bh); }

}  // extern "C"
