// NVTX ranges around the public calls, so a profiler timeline (nsys, ncu's
// range filters) shows each ABI call by name with its launches inside it.
// NVTX3 is header-only: without a tool attached a range costs one branch.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace ddt {

// The library's NVTX domain, created on first use.
inline nvtxDomainHandle_t trace_domain() {
    static nvtxDomainHandle_t d = nvtxDomainCreateA("ddtree");
    return d;
}

// One range for the lifetime of the object (the body of an ABI call).
class TraceRange {
  public:
    explicit TraceRange(const char* name) {
        nvtxEventAttributes_t a = {};
        a.version = NVTX_VERSION;
        a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
        a.messageType = NVTX_MESSAGE_TYPE_ASCII;
        a.message.ascii = name;
        nvtxDomainRangePushEx(trace_domain(), &a);
    }
    ~TraceRange() { nvtxDomainRangePop(trace_domain()); }
    TraceRange(const TraceRange&) = delete;
    TraceRange& operator=(const TraceRange&) = delete;
};

}  // namespace ddt
