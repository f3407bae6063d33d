// pdl.cuh -- programmatic dependent launch for the chains of small kernels
// of the SPEL step.
//
// A kernel launched with launch_chained may be scheduled while the kernel
// before it in the stream is still running.  Every such kernel starts with
// pdl_enter(): it lets the next kernel be scheduled at once, then waits until
// the kernels it depends on have completed and their writes are visible, so
// results are those of plain stream order and only the launch latency is
// hidden.  In a kernel launched without the attribute the wait returns at
// once.
#pragma once
#include <cuda_runtime.h>

namespace mapl {

__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// The two halves of pdl_enter, for a kernel whose setup (barrier init, TMEM
// allocation) touches no memory the earlier kernels write: the setup then
// runs while they finish.
__device__ __forceinline__ void pdl_allow_next() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_prior() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_chained(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                  cudaStream_t s, Args... args) {
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace mapl
