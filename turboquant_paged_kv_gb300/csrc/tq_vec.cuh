// Half-warp vector helpers shared by the store kernels: a half-warp holds the
// d = 128 coordinates of one vector, 8 per lane (coordinate 8 l + j in lane l
// of the half), so a warp works on two vectors at once.
#ifndef TQ_VEC_CUH_
#define TQ_VEC_CUH_

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <type_traits>

#include "tq_launch.cuh"

namespace tq {
namespace {

// 8 consecutive inputs (16 bytes) as floats.
template <typename T>
__device__ __forceinline__ void load8(const void* base, long long elem, float out[8]) {
  const uint4 raw = ld_dep_u32x4(static_cast<const T*>(base) + elem);
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f;
    if constexpr (std::is_same<T, __nv_bfloat16>::value) f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    else f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    out[2 * i] = f.x;
    out[2 * i + 1] = f.y;
  }
}

// Sum, min and max over the 16 lanes of a half-warp (xor 1 .. 8 stay inside
// it). `mask` names the lanes that take part: the whole warp, or one half when
// the two halves run different code.
__device__ __forceinline__ float half_sum(float x, unsigned mask = 0xffffffffu) {
#pragma unroll
  for (int m = 1; m <= 8; m <<= 1) x += __shfl_xor_sync(mask, x, m);
  return x;
}
__device__ __forceinline__ float half_min(float x, unsigned mask = 0xffffffffu) {
#pragma unroll
  for (int m = 1; m <= 8; m <<= 1) x = fminf(x, __shfl_xor_sync(mask, x, m));
  return x;
}
__device__ __forceinline__ float half_max(float x, unsigned mask = 0xffffffffu) {
#pragma unroll
  for (int m = 1; m <= 8; m <<= 1) x = fmaxf(x, __shfl_xor_sync(mask, x, m));
  return x;
}

// Sylvester-order Walsh-Hadamard transform (unnormalised) of the 128
// coordinates of a half-warp, coordinate 8 l + j in lane l: index bits 0-2 in
// the lane, bits 3-6 across lanes l ^ 1 .. l ^ 8. The lane whose stride bit is
// set keeps (partner - own), the other (own + partner).
__device__ __forceinline__ void fwht128_half(float v[8], int l, unsigned mask = 0xffffffffu) {
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j & h) continue;
      const float a = v[j], b = v[j + h];
      v[j] = a + b;
      v[j + h] = a - b;
    }
  }
#pragma unroll
  for (int m = 1; m <= 8; m <<= 1) {
    const float sgn = (l & m) ? -1.f : 1.f;   // one exact fma with +-1 per step
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = fmaf(sgn, v[j], __shfl_xor_sync(mask, v[j], m));
  }
}

}  // namespace
}  // namespace tq

#endif  // TQ_VEC_CUH_
