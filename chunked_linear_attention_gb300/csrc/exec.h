// Execution helpers of the host orchestration: a per-device pool of internal
// streams and events (fork/join of independent (batch, head) sequences), and
// a small cache of instantiated CUDA graphs keyed by the full set of call
// arguments, so that a repeated call replays its whole launch sequence with
// one cudaGraphLaunch.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <functional>
#include <mutex>
#include <vector>

namespace ttt {

// Guards the one-time, per-device setup caches of the kernels (function
// attributes, occupancy checks, SM counts): two host threads making their
// first call at the same time fill each cache once.
std::mutex& setup_mutex();

// Internal non-blocking streams of the current device (created on first use).
// Returns false if the pool cannot provide `n` streams.
bool stream_pool(int n, std::vector<cudaStream_t>* out);

// Fork: `n` pool streams wait for the work enqueued so far on `parent`.
// Join: `parent` waits for everything enqueued on the pool streams.
cudaError_t fork_streams(cudaStream_t parent, const std::vector<cudaStream_t>& kids);
cudaError_t join_streams(cudaStream_t parent, const std::vector<cudaStream_t>& kids);

// `n` events of the current device for ordering between pool streams
// (separate from the fork/join events).  Returns false on failure.
bool stagger_events(int n, std::vector<cudaEvent_t>* out);

// `n` events of the current device for host-transfer ordering (separate from
// the other pools; n <= 4096).  Returns false on failure.
bool io_events(int n, std::vector<cudaEvent_t>* out);

// The highest launch priority of the current device (0 when priorities are
// not supported): launches on the critical path of a call use it so that
// work off that path only fills the SMs it leaves free.
int high_priority();

// Runs `enqueue(stream)` through a cached graph when possible: on the first
// call with a given key the launch sequence is captured on an internal stream
// and instantiated; every call then launches the graph on `stream`.  Falls
// back to enqueueing directly on `stream` when graphs cannot be used (the
// stream is itself being captured, profiling is recording, or capture fails).
// `key` must identify every argument the launch sequence depends on.
// Returns the enqueue status code (0 = ok).
int run_cached(const std::vector<uint64_t>& key, cudaStream_t stream,
               const std::function<int(cudaStream_t)>& enqueue);

}  // namespace ttt
