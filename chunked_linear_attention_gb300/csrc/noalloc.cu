// Chunked linear attention for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: a host framework may own the GPU
// memory pool and forbid allocations from outside it, or a latency-critical
// loop cannot afford cudaMalloc's implicit device synchronisation.  This file
// gives them linattn_chunked_forward_noalloc: the same computation as
// linattn_chunked_forward, with its scratch taken from a fixed array that the
// library reserves in device memory when it is loaded, instead of from a
// caller-provided workspace.
//
// Costs and rules of that choice:
//   * Every GPU that loads the library holds kNoAllocScratchBytes (16 MiB) of
//     device memory for this array until the process exits.
//   * Problems whose scratch (linattn_workspace_size) exceeds 16 MiB are
//     rejected with TTT_ERR_WORKSPACE before anything is enqueued.
//   * The host side cannot use the array's name as a device address (in host
//     code it names a host-side stand-in), so the first call on each device
//     looks the address up with cudaGetSymbolAddress, with that device
//     current, and caches it.  That lookup is a runtime call, so make the
//     first call on each device before any stream capture begins.
//   * All calls share the one array and it keeps whatever the last call left
//     there.  No part of it needs to start at zero: every byte a call reads
//     was written earlier in the same call.  Calls that overlap on the GPU
//     (for example on two streams at once) race on the array; serialise them.
#include <mutex>

#include "ttt.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (looked up once
// per device).  Returns NULL if the runtime call fails.
void* scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" int linattn_chunked_forward_noalloc(const void* q, const void* k, const void* v,
                                               const float* eta, const float* S0, int B, int H,
                                               int N, int d_k, int d_v, int chunk, int io_dtype,
                                               int mask_mode, const unsigned char* update_chunks,
                                               void* out, float* S_final, ttt_stream_t stream) {
  const size_t need =
      linattn_workspace_size(B, H, N, d_k, d_v, chunk, io_dtype, mask_mode);
  if (need == 0) {
    // invalid arguments: let the regular entry point report which one
    return linattn_chunked_forward(q, k, v, eta, S0, B, H, N, d_k, d_v, chunk, io_dtype,
                                   mask_mode, update_chunks, out, S_final, nullptr, 0, stream);
  }
  if (need > kNoAllocScratchBytes) return TTT_ERR_WORKSPACE;
  void* scratch = scratch_for_current_device();
  if (!scratch) return TTT_ERR_CUDA;
  return linattn_chunked_forward(q, k, v, eta, S0, B, H, N, d_k, d_v, chunk, io_dtype, mask_mode,
                                 update_chunks, out, S_final, scratch, kNoAllocScratchBytes,
                                 stream);
}
