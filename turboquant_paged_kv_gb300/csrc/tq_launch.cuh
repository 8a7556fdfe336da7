// Kernel launch with programmatic dependent launch (CUDA 12+, sm_90+).
//
// A kernel launched this way may be scheduled while the kernel before it in
// the stream is still finishing, which hides the launch gap. Every kernel of
// this library therefore executes grid_dep_wait() before it reads or writes
// any global memory an earlier kernel may touch, and grid_dep_launch() only
// after that wait (so a kernel launched early behind it never starts before
// the kernels that came earlier still have finished).
#ifndef TQ_LAUNCH_CUH_
#define TQ_LAUNCH_CUH_

#include <cuda_runtime.h>

#include <utility>

namespace tq {

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Waits until the kernels this one depends on have completed and their
// memory is visible (a no-op without such dependencies).
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
// Lets the next kernel in the stream be scheduled early.
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

}  // namespace tq

#endif  // TQ_LAUNCH_CUH_
