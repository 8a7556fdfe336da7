// tq_store: fused rotate / quantise / pack / write of K and V into the paged
// cache, one half-warp per (token, KV head).
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
// as a separate cuBLAS GEMM over a materialised fp32 copy of K; here a
// half-warp holds the 128 coordinates in registers (8 per lane: coordinate
// 8 l + j in lane l of the half), rotates them with a butterfly (3 in-lane
// stages + 4 xor-shuffle stages) and never writes an intermediate. Each warp
// quantises two vectors at once, so every shuffle and reduction serves two
// vectors and the per-lane work (bucketize, value codes) runs over 8
// independent coordinates. The value-quantisation arithmetic uses explicitly
// rounded fp32 operations (no contraction), so V codes are reproducible bit
// for bit.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "tq_internal.h"
#include "tq_launch.cuh"
#include "tq_store.cuh"
#include "tq_vec.cuh"

namespace tq {
namespace {

constexpr int kStoreWarps = 8;
constexpr int kVecsPerCta = 2 * kStoreWarps;   // a half-warp per vector
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
  unsigned kv_magic, kv_shift;   // vec / n_kv = umulhi(2 vec, kv_magic) >> kv_shift (vec < 2^31)
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


enum KeyMode { kMse4 = 4, kMse3 = 3, kFp8 = 8 };   // the key codes' bits (8: e4m3)

__device__ __forceinline__ void flag(unsigned int* status, unsigned int bit) {
  if (status) atomicOr(status, bit);
}

// Warp w of the CTA handles vectors 2 w and 2 w + 1 of the CTA's 16, one per
// half-warp. A half whose vector is past the end, or whose slot is negative or
// out of range, computes on zeros and writes nothing (its lanes stay for the
// shuffles).
template <int KMODE, int VBITS, typename T>
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
  const int l = lane & 15;
  const long long vec = static_cast<long long>(blockIdx.x) * kVecsPerCta + (threadIdx.x >> 4);
  bool live = vec < a.num_vectors;
  long long tok = 0, slot = -1;
  int head = 0;
  if (live) {
    // vec / n_kv by multiply and shift whenever the vector count allows
    tok = a.num_vectors < (1ll << 31)
              ? static_cast<long long>(__umulhi(2u * static_cast<unsigned>(vec), a.kv_magic) >> a.kv_shift)
              : vec / a.n_kv;
    head = static_cast<int>(vec - tok * a.n_kv);
    slot = ld_dep_s64(a.slots + tok);
  }
  // the inputs' addresses do not depend on the slot: their loads go out with
  // the slot's, not after it
  float k[8], v[8];
  if (live) {
    load8<T>(a.key, vec * kD + 8 * l, k);
    load8<T>(a.value, vec * kD + 8 * l, v);
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) k[j] = v[j] = 0.f;
  }
  uint8_t* tile = nullptr;
  int r = 0;
  if (live) {
    const long long blk = slot >> a.log2_bs;
    if (slot < 0) {
      live = false;
    } else if (blk >= a.num_blocks) {
      if (l == 0) flag(a.status, TQ_DEV_SLOT_OUT_OF_RANGE);
      live = false;
    } else {
      const int off = static_cast<int>(slot & (a.block_size - 1));
      tile = a.cache + ((blk * a.n_kv + head) * a.tiles_per_block + (off >> 4)) * static_cast<long long>(a.tile_bytes);
      r = off & 15;
    }
  }

  const TileGeom geom = {a.k_off, a.k_row, a.v_off, a.v_row, a.knorm_off, a.vscale_off, a.vzero_off};
  PairBytes o;
  quantize_key<KMODE>(k, l, s_mid, s_cent, o);
  if (live) write_key<KMODE>(tile, r, geom, l, o);
  quantize_value<VBITS>(v, o);
  if (live) write_value<VBITS>(tile, r, geom, l, o);
}

template <int KMODE, int VBITS>
cudaError_t launch_store(const StoreArgs& a, int in_dtype, cudaStream_t stream) {
  const long long blocks = (a.num_vectors + kVecsPerCta - 1) / kVecsPerCta;
  if (in_dtype == TQ_DTYPE_BF16)
    return launch_pdl(store_kernel<KMODE, VBITS, __nv_bfloat16>, dim3(static_cast<unsigned>(blocks)),
                      dim3(kStoreWarps * 32), 0, stream, a);
  return launch_pdl(store_kernel<KMODE, VBITS, __half>, dim3(static_cast<unsigned>(blocks)), dim3(kStoreWarps * 32), 0,
                    stream, a);
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
  if (vectors / kVecsPerCta + 1 > 0x7fffffffll) return TQ_ERR_INVALID_ARG;

  StoreArgs a;
  a.key = key;
  a.value = value;
  a.slots = slot_mapping;
  a.cache = static_cast<uint8_t*>(cache);
  a.status = dev_status;
  a.num_vectors = vectors;
  a.num_blocks = num_blocks;
  a.n_kv = cfg->num_kv_heads;
  // x / n = floor(x magic / 2^(31 + s)) = umulhi(2 x, magic) >> s for every
  // x < 2^31, with s = ceil(log2 n) and magic = ceil(2^(31 + s) / n) < 2^32:
  // the excess magic n - 2^(31 + s) is below n, so x times it stays below
  // 2^(31 + s) and never carries the quotient past the next integer
  {
    unsigned sh = 0;
    while ((1u << sh) < static_cast<unsigned>(a.n_kv)) ++sh;
    a.kv_shift = sh;
    a.kv_magic = static_cast<unsigned>(((1ull << (31 + sh)) + a.n_kv - 1) / a.n_kv);
  }
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
  if (L.key_fp8) err = launch_store<kFp8, 4>(a, in_dtype, s);
  else if (L.key_bits == 4) err = launch_store<kMse4, 4>(a, in_dtype, s);
  else if (L.value_bits == 4) err = launch_store<kMse3, 4>(a, in_dtype, s);
  else err = launch_store<kMse3, 3>(a, in_dtype, s);
  return err == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}
