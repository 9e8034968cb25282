// pdl.cuh -- programmatic dependent launch (sm_90 and later): the decode
// split kernel lets the merge kernel be scheduled while it runs, and the
// prefill's V pass lets the attention kernel set up and load Q and K; each
// dependent kernel holds its first access to the previous grid's output until
// that grid has finished and its writes are visible. A kernel launched
// without the attribute passes the wait at once; ordering is never weaker
// than plain stream order for the data the wait guards.
#pragma once
#include <cuda_runtime.h>

#include <utility>

namespace attn {

// Blocks until every grid this one depends on has completed and its memory
// operations are visible.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the next kernel on the stream launch once every CTA of this grid has
// issued this (or exited).
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// <<<grid, block, smem, stream>>> with programmatic stream serialisation.
template <typename... P, typename... A>
cudaError_t launch_pdl(void (*kern)(P...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, A&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<A>(args)...);
}

}  // namespace attn
