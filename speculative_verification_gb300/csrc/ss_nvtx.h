// ss_nvtx.h -- one NVTX range per public call, named after the call, so that
// a timeline or a profiler's NVTX filter shows which ss_* call issued which
// launches.  NVTX v3 is header-only: with no tool attached a range costs a
// few nanoseconds on the host and nothing on the device.
#pragma once
#include <nvtx3/nvToolsExt.h>

namespace ss {

struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

}  // namespace ss

#define SS_NVTX_RANGE(name) const ::ss::NvtxRange ss_nvtx_range_(name)
