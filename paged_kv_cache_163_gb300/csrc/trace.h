// Named host-side ranges (NVTX) around the library's calls, so a profiler
// that records NVTX (a timeline tool, or ncu's --nvtx filters) can attribute
// host work and launches to them.  The NVTX v3 headers ship with the CUDA
// toolkit and need no library at link time; with no tool attached a range
// costs a few nanoseconds.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace pkv {

class TraceRange {
 public:
  explicit TraceRange(const char *name) { nvtxRangePushA(name); }
  ~TraceRange() { nvtxRangePop(); }
  TraceRange(const TraceRange &) = delete;
  TraceRange &operator=(const TraceRange &) = delete;
};

}  // namespace pkv
