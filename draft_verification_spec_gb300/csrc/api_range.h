// A named NVTX range around one C-ABI call, for profilers (Nsight timelines group the call's
// launches under its name).  NVTX v3 is header-only; without a tool attached each push and pop
// is a check of a null function pointer.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace sv {

struct ApiRange {
  explicit ApiRange(const char* name) { nvtxRangePushA(name); }
  ~ApiRange() { nvtxRangePop(); }
  ApiRange(const ApiRange&) = delete;
  ApiRange& operator=(const ApiRange&) = delete;
};

}  // namespace sv
