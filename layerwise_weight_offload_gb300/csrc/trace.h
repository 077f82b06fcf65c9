// trace.h — NVTX ranges in the "dlo" domain around the library's host-side
// work: the hooks of the two-slot schedule, the copies each prefetch
// enqueues, the block forward's launches, the CPU packing of rank-local
// blocks and the CPU flatten / shard split.
//
// NVTX calls go through function pointers that stay empty unless an NVTX
// tool is attached (nsys, `ncu --nvtx`, or any library named by
// NVTX_INJECTION64_PATH), so without one a range costs a load and a branch.
// A tool sees each range's name as an ASCII message and an int64 payload:
// the block index for the hooks and prefetches, the number of rows for a
// forward, the number of parameters for the plan and shard calls, the slot
// bytes for a one-shot reassembly.
#pragma once

#include <nvtx3/nvToolsExt.h>

#include <cstdint>

namespace dlo {

// The "dlo" domain, created on first use (null when no tool is attached).
nvtxDomainHandle_t trace_domain();

// A push/pop range on the calling thread, popped when the scope ends.
class TraceRange {
 public:
  TraceRange(const char* name, int64_t payload) {
    nvtxEventAttributes_t a{};
    a.version = NVTX_VERSION;
    a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
    a.messageType = NVTX_MESSAGE_TYPE_ASCII;
    a.message.ascii = name;
    a.payloadType = NVTX_PAYLOAD_TYPE_INT64;
    a.payload.llValue = payload;
    nvtxDomainRangePushEx(trace_domain(), &a);
  }
  ~TraceRange() { nvtxDomainRangePop(trace_domain()); }
  TraceRange(const TraceRange&) = delete;
  TraceRange& operator=(const TraceRange&) = delete;
};

}  // namespace dlo
