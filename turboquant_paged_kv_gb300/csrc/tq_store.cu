// tq_store: fused rotate / quantise / pack / write of K and V into the paged
// cache, one warp per (token, KV head).
//
// Method: "vLLM 源码完全拆解(十九):TurboQuant KV Cache 量化" (pinghaoyang.com.cn),
// section "写入内核:store 路径如何旋转、量化与打包":
//   n = ||k||, x = k / (n + 1e-8), y = (H / sqrt(d)) x            ("K 的归一化与旋转")
//   idx_i = #{j : y_i >= mid_j}                                    ("二分查找")
//   stored norm = n / sqrt(sum c[idx]^2 + 1e-16), fp16            ("norm correction 的折叠")
//   LSB-first bit packing of idx                                   ("位打包")
//   V: s = (max-min)/(2^b-1) floored at 1e-8, q = int((v-min)/s+0.5) clamped,
//      fp16 scale and zero                                         ("V 的 min/max 均匀量化")
//   FP8 keys: e4m3(k), no rotation, no norm                       ("FP8 K 路径")
//   slot < 0 writes nothing                                        ("融合 kernel 的骨架")
//
// Differences from the pages' design: the pages run the norm and the rotation
// as a separate cuBLAS GEMM over a materialised fp32 copy of K; here the warp
// holds the 128 coordinates in registers (4 per lane), rotates them with a
// butterfly (2 in-lane stages + 5 xor-shuffle stages) and never writes an
// intermediate. The value-quantisation arithmetic uses explicitly rounded fp32
// operations (no contraction), so V codes are reproducible bit for bit.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "tq_internal.h"
#include "tq_launch.cuh"

namespace tq {
namespace {

constexpr int kStoreWarps = 8;
constexpr int kD = 128;

struct StoreArgs {
  const void* key;
  const void* value;
  const long long* slots;
  uint8_t* cache;
  unsigned int* status;
  long long num_vectors;     // num_tokens * n_kv
  long long num_blocks;
  int n_kv;
  int block_size;
  int log2_bs;               // block_size is a power of two
  int tiles_per_block;
  int tile_bytes;
  int k_off, k_row;
  int v_off, v_row;
  int knorm_off, vscale_off, vzero_off;
  float mid[15];
  float cent[16];
};

enum KeyMode { kMse4 = 4, kMse3 = 3, kFp8 = 8 };

template <typename T>
__device__ __forceinline__ void load4(const void* base, long long elem, float out[4]) {
  const uint2 raw = ld_dep_u32x2(static_cast<const T*>(base) + elem);
  if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
    const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
    float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
    out[0] = a.x; out[1] = a.y; out[2] = b.x; out[3] = b.y;
  } else {
    const __half2 lo = *reinterpret_cast<const __half2*>(&raw.x);
    const __half2 hi = *reinterpret_cast<const __half2*>(&raw.y);
    float2 a = __half22float2(lo), b = __half22float2(hi);
    out[0] = a.x; out[1] = a.y; out[2] = b.x; out[3] = b.y;
  }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
  return x;
}

// Sylvester-order Walsh-Hadamard transform of the 128 coordinates held as
// 4 consecutive values per lane (coordinate 4*lane + j).
__device__ __forceinline__ void fwht128(float v[4], int lane) {
  float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
  v[0] = a0 + a2; v[2] = a0 - a2; v[1] = a1 + a3; v[3] = a1 - a3;
#pragma unroll
  for (int m = 1; m <= 16; m <<= 1) {
    const bool upper = lane & m;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float p = __shfl_xor_sync(0xffffffffu, v[j], m);
      v[j] = upper ? (p - v[j]) : (v[j] + p);
    }
  }
}

__device__ __forceinline__ void flag(unsigned int* status, unsigned int bit) {
  if (status) atomicOr(status, bit);
}

template <int KMODE, typename T>
__global__ void __launch_bounds__(kStoreWarps * 32)
store_kernel(const StoreArgs a) {
  grid_dep_wait();   // inputs and cache may come from the previous kernel
  grid_dep_launch();
  __shared__ float s_cent[16], s_mid[16];
  if (threadIdx.x < 16) {
    s_cent[threadIdx.x] = a.cent[threadIdx.x];
    s_mid[threadIdx.x] = threadIdx.x < 15 ? a.mid[threadIdx.x] : 0.f;
  }
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const long long vec = static_cast<long long>(blockIdx.x) * kStoreWarps + (threadIdx.x >> 5);
  if (vec >= a.num_vectors) return;
  // vec / n_kv in 32 bits whenever the vector count allows
  const long long tok = a.num_vectors < (1ll << 32)
                            ? static_cast<long long>(static_cast<unsigned>(vec) / static_cast<unsigned>(a.n_kv))
                            : vec / a.n_kv;
  const int head = static_cast<int>(vec - tok * a.n_kv);
  const long long slot = ld_dep_s64(a.slots + tok);
  if (slot < 0) return;
  const long long blk = slot >> a.log2_bs;
  const int off = static_cast<int>(slot & (a.block_size - 1));
  if (blk >= a.num_blocks) {
    if (lane == 0) flag(a.status, TQ_DEV_SLOT_OUT_OF_RANGE);
    return;
  }
  uint8_t* tile = a.cache +
      ((blk * a.n_kv + head) * a.tiles_per_block + (off >> 4)) * static_cast<long long>(a.tile_bytes);
  const int r = off & 15;

  float k[4], v[4];
  load4<T>(a.key, vec * kD + lane * 4, k);
  load4<T>(a.value, vec * kD + lane * 4, v);

  // ---------------- keys ----------------
  if constexpr (KMODE == kFp8) {
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(k[0], k[1]), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(k[2], k[3]), __NV_SATFINITE, __NV_E4M3);
    const uint32_t w = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
    *reinterpret_cast<uint32_t*>(tile + a.k_off + r * a.k_row + 4 * lane) = w;
  } else {
    float ss = k[0] * k[0];
    ss = fmaf(k[1], k[1], ss);
    ss = fmaf(k[2], k[2], ss);
    ss = fmaf(k[3], k[3], ss);
    const float n = __fsqrt_rn(warp_sum(ss));
    fwht128(k, lane);
    const float sc = __fdiv_rn(0.088388347648318440f, __fadd_rn(n, 1e-8f));   // 1/sqrt(128) / (n + 1e-8)
    int idx[4];
    float cs = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float y = k[j] * sc;
      // #{m : y >= mid_m} over the ascending midpoints, by binary search
      int c = 0;
#pragma unroll
      for (int step = 1 << (KMODE - 1); step >= 1; step >>= 1) c += (y >= s_mid[c + step - 1]) ? step : 0;
      idx[j] = c;
      const float cv = s_cent[c];
      cs = fmaf(cv, cv, cs);
    }
    cs = warp_sum(cs);
    const float stored = __fdiv_rn(n, __fsqrt_rn(__fadd_rn(cs, 1e-16f)));
    if constexpr (KMODE == kMse4) {
      const uint32_t w = idx[0] | (idx[1] << 4) | (idx[2] << 8) | (idx[3] << 12);
      *reinterpret_cast<uint16_t*>(tile + a.k_off + r * a.k_row + 2 * lane) = static_cast<uint16_t>(w);
    } else {
      const uint32_t w12 = idx[0] | (idx[1] << 3) | (idx[2] << 6) | (idx[3] << 9);
      const uint32_t partner = __shfl_xor_sync(0xffffffffu, w12, 1);
      if ((lane & 1) == 0) {
        const uint32_t w24 = w12 | (partner << 12);
        uint8_t* dst = tile + a.k_off + r * a.k_row + 3 * (lane >> 1);
        dst[0] = static_cast<uint8_t>(w24);
        dst[1] = static_cast<uint8_t>(w24 >> 8);
        dst[2] = static_cast<uint8_t>(w24 >> 16);
      }
    }
    if (lane == 0)
      *reinterpret_cast<uint16_t*>(tile + a.knorm_off + 2 * r) = __half_as_ushort(__float2half_rn(stored));
  }

  // ---------------- values (4-bit) ----------------
  float mn = fminf(fminf(v[0], v[1]), fminf(v[2], v[3]));
  float mx = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
  asm("redux.sync.min.f32 %0, %0, 0xffffffff;" : "+f"(mn));
  asm("redux.sync.max.f32 %0, %0, 0xffffffff;" : "+f"(mx));
  float s = __fdiv_rn(__fsub_rn(mx, mn), 15.0f);
  s = (s > 1e-8f) ? s : 1e-8f;
  // code = trunc(fp32((v - min) / s) + 1/2) with IEEE division, as specified.
  // The product with the correctly rounded reciprocal is within 4e-6 of it
  // (t <= 15), so away from a rounding boundary it gives the same code; within
  // 1e-5 of one the exact quotient is taken.
  const float rs = __frcp_rn(s);
  uint32_t w = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float dv = __fsub_rn(v[j], mn);
    const float u = __fadd_rn(__fmul_rn(dv, rs), 0.5f);
    const float fr = u - floorf(u);
    int q = (fr < 1e-5f || fr > 1.f - 1e-5f) ? __float2int_rz(__fadd_rn(__fdiv_rn(dv, s), 0.5f)) : __float2int_rz(u);
    q = min(max(q, 0), 15);
    w |= static_cast<uint32_t>(q) << (4 * j);
  }
  // pair-interleaved 16-bit words, 16-byte groups swizzled by the pair index:
  // word `lane` of token r = 2p + j
  const int pair = r >> 1;
  const int swz = (a.v_row % 64 == 0) ? 2 * (pair & 3) : 0;
  *reinterpret_cast<uint16_t*>(tile + a.v_off + pair * 2 * a.v_row + 16 * ((lane >> 2) ^ swz) + 4 * (lane & 3) +
                               2 * (r & 1)) = static_cast<uint16_t>(w);
  if (lane == 0) {
    *reinterpret_cast<uint16_t*>(tile + a.vscale_off + 2 * r) = __half_as_ushort(__float2half_rn(s));
    *reinterpret_cast<uint16_t*>(tile + a.vzero_off + 2 * r) = __half_as_ushort(__float2half_rn(mn));
  }
}

template <int KMODE>
cudaError_t launch_store(const StoreArgs& a, int in_dtype, cudaStream_t stream) {
  const long long blocks = (a.num_vectors + kStoreWarps - 1) / kStoreWarps;
  cudaError_t err;
  if (in_dtype == TQ_DTYPE_BF16)
    err = launch_pdl(store_kernel<KMODE, __nv_bfloat16>, dim3(static_cast<unsigned>(blocks)), dim3(kStoreWarps * 32), 0,
                     stream, a);
  else
    err = launch_pdl(store_kernel<KMODE, __half>, dim3(static_cast<unsigned>(blocks)), dim3(kStoreWarps * 32), 0,
                     stream, a);
  return err;
}

}  // namespace
}  // namespace tq

extern "C" tq_status tq_store(const tq_config* cfg, const tq_codebook* cb,
                              const void* key, const void* value, int in_dtype,
                              long long num_tokens, const long long* slot_mapping,
                              void* cache, long long num_blocks,
                              unsigned int* dev_status, tq_stream_t stream) {
  using namespace tq;
  tq_layout L;
  const tq_status st = make_layout(cfg, &L);
  if (st != TQ_OK) return st;
  if (num_tokens < 0 || num_blocks < 0) return TQ_ERR_INVALID_ARG;
  if (in_dtype != TQ_DTYPE_F16 && in_dtype != TQ_DTYPE_BF16) return TQ_ERR_INVALID_ARG;
  if (!L.key_fp8) {
    if (!cb || cb->bits != L.key_bits || cb->head_dim != cfg->head_dim) return TQ_ERR_INVALID_ARG;
  }
  if (num_tokens == 0) return TQ_OK;
  if (!key || !value || !slot_mapping || !cache) return TQ_ERR_INVALID_ARG;
  if (!aligned16(key) || !aligned16(value) || !aligned16(cache) ||
      (reinterpret_cast<unsigned long long>(slot_mapping) & 7ull))
    return TQ_ERR_MISALIGNED;
  if (dev_status && (reinterpret_cast<unsigned long long>(dev_status) & 3ull)) return TQ_ERR_MISALIGNED;
  const long long vectors = num_tokens * cfg->num_kv_heads;
  if (vectors / kStoreWarps + 1 > 0x7fffffffll) return TQ_ERR_INVALID_ARG;

  StoreArgs a;
  a.key = key;
  a.value = value;
  a.slots = slot_mapping;
  a.cache = static_cast<uint8_t*>(cache);
  a.status = dev_status;
  a.num_vectors = vectors;
  a.num_blocks = num_blocks;
  a.n_kv = cfg->num_kv_heads;
  a.block_size = cfg->block_size;
  a.log2_bs = __builtin_ctz(static_cast<unsigned>(cfg->block_size));
  a.tiles_per_block = cfg->block_size / kTileTokens;
  a.tile_bytes = L.tile_bytes;
  a.k_off = L.k_off;
  a.k_row = L.k_row_bytes;
  a.v_off = L.v_off;
  a.v_row = L.v_row_bytes;
  a.knorm_off = L.knorm_off;
  a.vscale_off = L.vscale_off;
  a.vzero_off = L.vzero_off;
  for (int i = 0; i < 15; ++i) a.mid[i] = (!L.key_fp8 && i < cb->num_levels - 1) ? cb->midpoints[i] : 0.f;
  for (int i = 0; i < 16; ++i) a.cent[i] = (!L.key_fp8 && i < cb->num_levels) ? cb->centroids[i] : 0.f;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t err;
  if (L.key_fp8) err = launch_store<kFp8>(a, in_dtype, s);
  else if (L.key_bits == 4) err = launch_store<kMse4>(a, in_dtype, s);
  else err = launch_store<kMse3>(a, in_dtype, s);
  return err == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}
