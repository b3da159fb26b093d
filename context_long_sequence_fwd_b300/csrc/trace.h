// Per-kernel timing of the library's own launches (host side).
//
// When tracing is on, every kernel launch is bracketed by two CUDA events
// recorded on the stream it is launched on; ringattn_trace_collect() waits for
// them and reports, per kernel, the number of launches and their summed
// device time.  When tracing is off a launch pays one relaxed atomic load.
#pragma once
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

namespace ra {

bool trace_enabled();

// An NVTX range over one public call (host-side work and launches), for
// profilers that read NVTX (ncu --nvtx --nvtx-include); without one attached
// a push or pop costs a pointer check.
class NvtxRange {
 public:
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Brackets one kernel launch: construct right before it, destroy right after.
// The launch also gets an NVTX range named after the kernel.
class TraceScope {
 public:
  TraceScope(cudaStream_t stream, const char* kernel);
  ~TraceScope();
  TraceScope(const TraceScope&) = delete;
  TraceScope& operator=(const TraceScope&) = delete;

 private:
  cudaStream_t stream_;
  int slot_ = -1;
  NvtxRange nvtx_;
};

}  // namespace ra
