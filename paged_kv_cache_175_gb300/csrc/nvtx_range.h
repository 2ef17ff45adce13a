// NVTX ranges around the entry points that enqueue GPU work, so a profiler's timeline
// shows which library call launched which kernels.  NVTX is header-only: without a
// profiler attached a range costs a few nanoseconds and does nothing.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace pkv {
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
}  // namespace pkv

#define PKV_NVTX(name) ::pkv::NvtxRange pkv_nvtx_range_(name)
