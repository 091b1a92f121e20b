// trace.h -- NVTX ranges around the C-ABI calls, so that a profiler's
// timeline (Nsight Systems, or Nsight Compute's --nvtx filters) shows which
// ck_* call enqueued which kernels.  NVTX 3 is header-only: with no tool
// attached a range costs a predicted branch.  -DCK_NO_NVTX leaves them out.
#pragma once

#ifndef CK_NO_NVTX
#include <nvtx3/nvToolsExt.h>
#endif

namespace ck {

class TraceRange {
  public:
    explicit TraceRange(const char *name) {
#ifndef CK_NO_NVTX
        nvtxRangePushA(name);
#else
        (void)name;
#endif
    }
    ~TraceRange() {
#ifndef CK_NO_NVTX
        nvtxRangePop();
#endif
    }
    TraceRange(const TraceRange &) = delete;
    TraceRange &operator=(const TraceRange &) = delete;
};

}  // namespace ck

// One range over the rest of the enclosing scope, named after the call.
#define CK_TRACE(name) const ::ck::TraceRange ck_trace_range_(name)
