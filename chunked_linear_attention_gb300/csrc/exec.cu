#include "exec.h"

#include <cstdlib>
#include <list>
#include <mutex>

#include "prof.h"

namespace ttt {

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxPool = 64;
constexpr size_t kMaxGraphs = 8;

struct DevicePool {
  std::vector<cudaStream_t> streams;
  std::vector<cudaEvent_t> events;
  std::vector<cudaEvent_t> order_events;
  std::vector<cudaEvent_t> io_events;
  cudaStream_t capture = nullptr;
};

std::mutex g_pool_mu;
DevicePool g_pools[kMaxDevices];

struct GraphEntry {
  int device;
  std::vector<uint64_t> key;
  cudaGraphExec_t exec;
  size_t nodes;
};

std::mutex g_graph_mu;
std::list<GraphEntry> g_graphs;  // most recently used first

DevicePool* pool_for_current() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  return &g_pools[dev];
}

bool ensure_events(DevicePool* p, size_t n) {
  while (p->events.size() < n) {
    cudaEvent_t e;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return false;
    p->events.push_back(e);
  }
  return true;
}

bool graphs_disabled() {
  static const bool v = [] {
    const char* s = std::getenv("TTT_DISABLE_GRAPHS");
    return s && s[0] && s[0] != '0';
  }();
  return v;
}

}  // namespace

std::mutex& setup_mutex() {
  static std::mutex mu;
  return mu;
}

bool stream_pool(int n, std::vector<cudaStream_t>* out) {
  if (n > kMaxPool) return false;
  std::lock_guard<std::mutex> lk(g_pool_mu);
  DevicePool* p = pool_for_current();
  if (!p) return false;
  while ((int)p->streams.size() < n) {
    cudaStream_t s;
    if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return false;
    p->streams.push_back(s);
  }
  out->assign(p->streams.begin(), p->streams.begin() + n);
  return true;
}

bool stagger_events(int n, std::vector<cudaEvent_t>* out) {
  if (n > kMaxPool) return false;
  std::lock_guard<std::mutex> lk(g_pool_mu);
  DevicePool* p = pool_for_current();
  if (!p) return false;
  while ((int)p->order_events.size() < n) {
    cudaEvent_t e;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return false;
    p->order_events.push_back(e);
  }
  out->assign(p->order_events.begin(), p->order_events.begin() + n);
  return true;
}

int high_priority() {
  static int cached[kMaxDevices];
  static bool done[kMaxDevices] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lk(g_pool_mu);
  if (!done[dev]) {
    int least = 0, greatest = 0;
    cached[dev] = cudaDeviceGetStreamPriorityRange(&least, &greatest) == cudaSuccess ? greatest : 0;
    done[dev] = true;
  }
  return cached[dev];
}

bool io_events(int n, std::vector<cudaEvent_t>* out) {
  if (n > 4096) return false;
  std::lock_guard<std::mutex> lk(g_pool_mu);
  DevicePool* p = pool_for_current();
  if (!p) return false;
  while ((int)p->io_events.size() < n) {
    cudaEvent_t e;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return false;
    p->io_events.push_back(e);
  }
  out->assign(p->io_events.begin(), p->io_events.begin() + n);
  return true;
}

cudaError_t fork_streams(cudaStream_t parent, const std::vector<cudaStream_t>& kids) {
  std::lock_guard<std::mutex> lk(g_pool_mu);
  DevicePool* p = pool_for_current();
  if (!p || !ensure_events(p, 1)) return cudaErrorUnknown;
  cudaError_t e = cudaEventRecord(p->events[0], parent);
  if (e != cudaSuccess) return e;
  for (cudaStream_t k : kids)
    if ((e = cudaStreamWaitEvent(k, p->events[0], 0)) != cudaSuccess) return e;
  return cudaSuccess;
}

cudaError_t join_streams(cudaStream_t parent, const std::vector<cudaStream_t>& kids) {
  std::lock_guard<std::mutex> lk(g_pool_mu);
  DevicePool* p = pool_for_current();
  if (!p || !ensure_events(p, kids.size() + 1)) return cudaErrorUnknown;
  cudaError_t e;
  for (size_t i = 0; i < kids.size(); ++i) {
    if ((e = cudaEventRecord(p->events[i + 1], kids[i])) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(parent, p->events[i + 1], 0)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

int run_cached(const std::vector<uint64_t>& key, cudaStream_t stream,
               const std::function<int(cudaStream_t)>& enqueue) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (graphs_disabled() || prof_recording() ||
      cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
    return enqueue(stream);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return enqueue(stream);

  std::lock_guard<std::mutex> lk(g_graph_mu);
  for (auto it = g_graphs.begin(); it != g_graphs.end(); ++it) {
    if (it->device == dev && it->key == key) {
      g_graphs.splice(g_graphs.begin(), g_graphs, it);
      if (cudaGraphLaunch(it->exec, stream) != cudaSuccess) return -6;
      prof_count_launches(it->nodes);
      return 0;
    }
  }
  // capture the launch sequence on an internal stream
  cudaStream_t cap = nullptr;
  {
    std::lock_guard<std::mutex> plk(g_pool_mu);
    DevicePool* p = pool_for_current();
    if (!p) return enqueue(stream);
    if (!p->capture &&
        cudaStreamCreateWithFlags(&p->capture, cudaStreamNonBlocking) != cudaSuccess)
      return enqueue(stream);
    cap = p->capture;
  }
  if (cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaGetLastError();
    return enqueue(stream);
  }
  const int rc = enqueue(cap);
  cudaGraph_t graph = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(cap, &graph);
  if (rc != 0 || ec != cudaSuccess || !graph) {
    if (graph) cudaGraphDestroy(graph);
    cudaGetLastError();
    return rc != 0 ? rc : enqueue(stream);
  }
  size_t nodes = 0;
  cudaGraphGetNodes(graph, nullptr, &nodes);
  cudaGraphExec_t exec = nullptr;
  const cudaError_t ei = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  if (ei != cudaSuccess || !exec) {
    cudaGetLastError();
    return enqueue(stream);
  }
  if (g_graphs.size() >= kMaxGraphs) {
    cudaGraphExecDestroy(g_graphs.back().exec);
    g_graphs.pop_back();
  }
  g_graphs.push_front(GraphEntry{dev, key, exec, nodes});
  if (cudaGraphLaunch(exec, stream) != cudaSuccess) return -6;
  // the capture counted the launches once already
  return 0;
}

}  // namespace ttt
