// Programmatic dependent launch for the kernels of the expert block's chains.
//
// A kernel launched by launch_pdl(true, ...) may be scheduled while the kernel before it
// on the stream is still finishing: its launch and CTA placement overlap the
// predecessor's tail.  Measured on this GPU, that saves about ten microseconds on a
// decode-size forward (a chain of six short kernels) but costs about thirty on the
// 16384-token forward, whose kernels fill the GPU (chiefly at the requant and
// un-permute boundaries), so the callers ask for it on decode-size batches only;
// launch_pdl(false, ...) is an ordinary launch.
// Every kernel launched this way calls grid_dep_sync() before its first access to global
// memory; griddepcontrol.wait returns once the predecessor grid has completed and its
// memory operations are visible (at once when there is no programmatic predecessor), so
// the stream order of the results is the same as with ordinary launches.
// griddepcontrol.launch_dependents then allows the next such kernel to be scheduled: the
// dependent grid starts only after every CTA of this grid has issued it or exited, i.e.
// after all of this grid's CTAs have been placed, so a waiting dependent never holds
// resources that this grid still needs.
#pragma once
#include <cuda_runtime.h>

#include <utility>

namespace nvfp4 {

__device__ __forceinline__ void grid_dep_sync() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(bool programmatic, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = programmatic ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace nvfp4
