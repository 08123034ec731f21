// pdl.cuh -- chaining the launches of one call with programmatic dependent
// launch (sm_90 and later).
//
// A call whose work does not fit one launch (the tensor and pointer tables
// are passed by value, at most 32 KB per launch) issues several launches of
// the same kernel over disjoint data.  Plain stream order makes each launch
// wait for the previous one to drain completely, leaving SMs idle during
// its last wave.  Chained, launch k+1 (launched with programmatic stream
// serialisation) may start once every CTA of launch k has started
// (launch_dependents is the first thing each CTA does), so its CTAs fill the
// SMs that launch k's last wave frees.  Each CTA of a chained launch waits
// for the previous launch to complete before it exits (griddepcontrol.wait),
// so the last launch completes only after all earlier ones have: to the
// stream, and to the caller, the call still ends when all its work has.
// The wait cannot deadlock: launch k's CTAs have all started before any CTA
// of launch k+1 exists, and none of them waits on anything.  In a launch
// without the attribute griddepcontrol.wait returns at once.
#pragma once

#include <cuda_runtime.h>

namespace cr {

__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait_prerequisites() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Launch `kernel` on `grid` CTAs of `block` threads; `chained` launches it
// as the programmatic dependent of the previous launch on the stream.
template <typename... KArgs, typename... Args>
cudaError_t launch_chained(void (*kernel)(KArgs...), unsigned grid, unsigned block,
                           cudaStream_t s, bool chained, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = chained ? attr : nullptr;
  cfg.numAttrs = chained ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace cr
