// nvtx_range.h -- a host-side NVTX range around the enqueue of one operation,
// so that profiler timelines (Nsight Systems, ncu's NVTX filters) show which
// kernels each C-ABI call launched.  NVTX v3 is header-only: without a tool
// attached a range costs a check of a function pointer.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace dgrad {

struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

}  // namespace dgrad
