// NVTX ranges around the entry points' launches, for profiler timelines.
// Compiled out unless the library is built with -DPKV_NVTX (the build's
// --nvtx flag); then each entry point that enqueues work pushes a range
// named after itself for the host-side time of its checks and launches.
#pragma once

#ifdef PKV_NVTX
#include <nvtx3/nvToolsExt.h>

namespace pkv {
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
}  // namespace pkv

#define PKV_NVTX_RANGE(name) ::pkv::NvtxRange pkv_nvtx_range_(name)
#else
#define PKV_NVTX_RANGE(name) ((void)0)
#endif
