// NVTX ranges around the library's entry points, for timeline tools.
//
// Off by default.  Turned on by CPATTN_NVTX=1 in the environment (read at the
// first call) or by cp_attn_debug(CPATTN_DEBUG_NVTX, 1).  When on, every
// entry point that queues device work pushes a range named after itself for
// the duration of the host call (the range covers the launches it queues,
// not their execution on the GPU).  The NVTX v3 header is header-only: with
// no tool attached its calls do nothing.
#pragma once
#include <atomic>
#include <cstdlib>

#include <nvtx3/nvToolsExt.h>

namespace cpattn {

inline std::atomic<int>& nvtx_flag() {
  static std::atomic<int> flag{[] {
    const char* e = std::getenv("CPATTN_NVTX");
    return (e && *e && *e != '0') ? 1 : 0;
  }()};
  return flag;
}

struct NvtxRange {
  bool on;
  explicit NvtxRange(const char* name) : on(nvtx_flag().load(std::memory_order_relaxed) != 0) {
    if (on) nvtxRangePushA(name);
  }
  ~NvtxRange() {
    if (on) nvtxRangePop();
  }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

}  // namespace cpattn

#define CPATTN_TRACE(name) ::cpattn::NvtxRange cpattn_trace_range_(name)
