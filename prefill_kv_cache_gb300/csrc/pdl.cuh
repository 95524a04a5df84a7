// Programmatic dependent launch for the decode-path kernels.
//
// A kernel launched with launch_pdl may be scheduled while the kernel before
// it in the stream is still running, so its launch latency overlaps that
// kernel's tail.  Such a kernel calls pdl_wait() before it reads anything an
// earlier kernel wrote: the wait returns once the preceding grid has completed
// and its memory operations are visible.  pdl_trigger() at the top of a kernel
// lets the next one be scheduled as soon as every CTA of this grid is running.
// Launched without the attribute, both instructions are no-ops.
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace snapkv {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... K, typename... A>
cudaError_t launch_pdl(void (*kern)(K...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<A>(args)...);
}

}  // namespace snapkv
