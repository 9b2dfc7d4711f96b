// Host-side NVTX ranges around the library's entry points, so that a profiler
// timeline shows which call issued which kernels (one range per call: the
// decode, its plan, the combine, the append).  NVTX v3 is header-only; with no
// tool attached a range costs a branch.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace mla {

class TraceRange {
 public:
  explicit TraceRange(const char *name) { nvtxRangePushA(name); }
  ~TraceRange() { nvtxRangePop(); }
  TraceRange(const TraceRange &) = delete;
  TraceRange &operator=(const TraceRange &) = delete;
};

}  // namespace mla
