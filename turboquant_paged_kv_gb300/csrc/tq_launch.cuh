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

// Global loads of anything another kernel may write. Two rules:
//  - They go to L2 (ld.global.cg), never through the non-coherent L1 /
//    read-only path (__ldg, ld.global.nc): a kernel launched early behind
//    another may run on an SM whose L1 still holds lines from before that
//    kernel's writes, and read them (measured on GB300: the LSE reduce read
//    stale partials that way).
//  - They stay after grid_dep_wait() when the data comes from the kernel
//    before: volatile asm statements keep their order, so these loads cannot
//    be moved above the wait (an __ldg may be, since it declares the data
//    constant for the kernel's lifetime).
__device__ __forceinline__ int ld_dep_s32(const int* p) {
  int v;
  asm volatile("ld.global.cg.b32 %0, [%1];\n" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ long long ld_dep_s64(const long long* p) {
  long long v;
  asm volatile("ld.global.cg.b64 %0, [%1];\n" : "=l"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ unsigned short ld_dep_u16(const void* p) {
  unsigned short v;
  asm volatile("ld.global.cg.b16 %0, [%1];\n" : "=h"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ unsigned int ld_dep_u8(const void* p) {
  unsigned int v;
  asm volatile("ld.global.cg.u8 %0, [%1];\n" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ unsigned int ld_dep_u32(const void* p) {
  unsigned int v;
  asm volatile("ld.global.cg.b32 %0, [%1];\n" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ld_dep_u32x2(const void* p) {
  uint2 v;
  asm volatile("ld.global.cg.v2.b32 {%0, %1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 ld_dep_u32x4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.b32 {%0, %1, %2, %3}, [%4];\n" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ float ld_dep_f32(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];\n" : "=f"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ float4 ld_dep_f32x4(const float4* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];\n" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
  return v;
}

}  // namespace tq

#endif  // TQ_LAUNCH_CUH_
