// Per-kernel timing of the library's own launches (see trace.h and the
// ringattn_trace_* entry points in include/ringattn.h).
#include "trace.h"

#include <atomic>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "ringattn.h"

namespace ra {

namespace {

struct Record {
  const char* kernel = nullptr;  // static string of the launcher
  int device = 0;
  cudaEvent_t start = nullptr, end = nullptr;
};

std::atomic<bool> g_on{false};
std::mutex g_tmu;
std::vector<Record> g_records;  // launches since the last collect
struct PooledPair {
  int device;
  cudaEvent_t start, end;
};
std::vector<PooledPair> g_pool;  // recycled events, per device
constexpr size_t kMaxRecords = 1 << 16;

bool take_pair(int device, cudaEvent_t* s, cudaEvent_t* e) {
  for (size_t i = 0; i < g_pool.size(); ++i) {
    if (g_pool[i].device == device) {
      *s = g_pool[i].start;
      *e = g_pool[i].end;
      g_pool[i] = g_pool.back();
      g_pool.pop_back();
      return true;
    }
  }
  if (cudaEventCreate(s) != cudaSuccess) return false;
  if (cudaEventCreate(e) != cudaSuccess) {
    cudaEventDestroy(*s);
    return false;
  }
  return true;
}

}  // namespace

bool trace_enabled() { return g_on.load(std::memory_order_relaxed); }

TraceScope::TraceScope(cudaStream_t stream, const char* kernel)
    : stream_(stream), nvtx_(kernel) {
  if (!trace_enabled()) return;
  std::lock_guard<std::mutex> lock(g_tmu);
  if (g_records.size() >= kMaxRecords) return;  // silently stop recording
  Record r;
  r.kernel = kernel;
  if (cudaGetDevice(&r.device) != cudaSuccess) return;
  if (!take_pair(r.device, &r.start, &r.end)) return;
  if (cudaEventRecord(r.start, stream) != cudaSuccess) {
    g_pool.push_back({r.device, r.start, r.end});
    return;
  }
  slot_ = static_cast<int>(g_records.size());
  g_records.push_back(r);
}

TraceScope::~TraceScope() {
  if (slot_ < 0) return;
  std::lock_guard<std::mutex> lock(g_tmu);
  cudaEventRecord(g_records[slot_].end, stream_);
}

}  // namespace ra

using namespace ra;

extern "C" {

ra_status ringattn_trace_enable(int on) {
  g_on.store(on != 0, std::memory_order_relaxed);
  return RA_OK;
}

ra_status ringattn_trace_collect(ra_trace_entry* entries, int max_entries, int* num_entries) {
  if (!num_entries || max_entries < 0 || (max_entries > 0 && !entries)) return RA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_tmu);
  std::vector<ra_trace_entry> agg;
  ra_status st = RA_OK;
  int cur = 0;
  cudaGetDevice(&cur);
  for (const Record& r : g_records) {
    float ms = 0.f;
    if (cudaSetDevice(r.device) != cudaSuccess || cudaEventSynchronize(r.end) != cudaSuccess ||
        cudaEventElapsedTime(&ms, r.start, r.end) != cudaSuccess) {
      st = RA_ERR_CUDA;
    } else {
      size_t i = 0;
      while (i < agg.size() && std::strncmp(agg[i].kernel, r.kernel, sizeof(agg[i].kernel)) != 0) ++i;
      if (i == agg.size()) {
        ra_trace_entry e{};
        std::strncpy(e.kernel, r.kernel, sizeof(e.kernel) - 1);
        agg.push_back(e);
      }
      agg[i].launches += 1;
      agg[i].total_ms += ms;
    }
    g_pool.push_back({r.device, r.start, r.end});
  }
  cudaSetDevice(cur);
  g_records.clear();
  *num_entries = static_cast<int>(agg.size());
  for (int i = 0; i < *num_entries && i < max_entries; ++i) entries[i] = agg[i];
  if (st == RA_OK && *num_entries > max_entries) st = RA_ERR_WORKSPACE;
  return st;
}

}  // extern "C"
