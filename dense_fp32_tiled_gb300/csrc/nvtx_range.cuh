// nvtx_range.cuh -- named ranges around the work each entry point enqueues
// (operand copies, product grids, split tail, host-buffer copies), so that a
// timeline taken with a profiler shows a call's phases by name.  NVTX3 is
// header-only: without a profiler attached each range costs a check of a
// function pointer.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace sg_nvtx {

struct Range {
    explicit Range(const char *name) { nvtxRangePushA(name); }
    ~Range() { nvtxRangePop(); }
    Range(const Range &) = delete;
    Range &operator=(const Range &) = delete;
};

}  // namespace sg_nvtx
