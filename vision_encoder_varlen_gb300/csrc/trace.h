// NVTX ranges around the library's public calls: a profiler (Nsight Systems, or ncu's NVTX
// filters) sees each call's launches under the call's name, in the "vitattn" domain. NVTX 3
// is header-only; with no tool attached a range costs a few nanoseconds, and a tool is found
// the usual NVTX way (the NVTX_INJECTION64_PATH environment variable).
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace vit {

inline nvtxDomainHandle_t trace_domain()
{
    static const nvtxDomainHandle_t domain = nvtxDomainCreateA("vitattn");
    return domain;
}

// One range for the lifetime of the object: pushed on entry to a call, popped on every return.
class TraceRange {
public:
    explicit TraceRange(const char *name)
    {
        nvtxEventAttributes_t a{};
        a.version = NVTX_VERSION;
        a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
        a.messageType = NVTX_MESSAGE_TYPE_ASCII;
        a.message.ascii = name;
        nvtxDomainRangePushEx(trace_domain(), &a);
    }
    ~TraceRange() { nvtxDomainRangePop(trace_domain()); }
    TraceRange(const TraceRange &) = delete;
    TraceRange &operator=(const TraceRange &) = delete;
};

}  // namespace vit
