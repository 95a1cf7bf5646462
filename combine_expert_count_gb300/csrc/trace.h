// trace.h -- an NVTX range over each C-ABI call of libmoeroute.
//
// A profiler attached to the process (ncu --nvtx, Nsight Systems) sees every
// kernel a call launches inside a range named after the call ("moe_dispatch",
// "moe_combine", ...).  NVTX here is the header-only NVTX3 of the CUDA
// toolkit: with no profiler attached, a push and a pop cost a few
// nanoseconds on the host and nothing on the GPU, and stream capture of the
// calls is unaffected.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace moe {

class CallRange {
  public:
    explicit CallRange(const char *name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
    CallRange(const CallRange &) = delete;
    CallRange &operator=(const CallRange &) = delete;
};

}  // namespace moe

// The range of the enclosing entry point, named after it.
#define MOE_TRACE_CALL() moe::CallRange moe_call_range_(__func__)
