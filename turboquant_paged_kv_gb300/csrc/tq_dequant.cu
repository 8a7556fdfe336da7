// tq_dequant: the cached keys and values of whole sequences expanded back to
// 16- or 32-bit vectors in the original (unrotated) basis.
//
// Method: "vLLM 源码完全拆解(十九):TurboQuant KV Cache 量化" (pinghaoyang.com.cn),
// section "续写 prefill:小 chunk 走 decode,大 chunk 走反量化", subsection
// "反量化 kernel:_tq_full_dequant_kv": every cached (position, KV head) slot is
// unpacked exactly as the decode unpacks it, with no softmax, and the keys are
// rotated back. The rotation H / sqrt(d) is symmetric and orthonormal (section
// "为什么先旋转"), so it is its own inverse:
//   index-coded keys  k = stored_norm * (H / sqrt(d)) c[idx]
//   FP8 keys          k = e4m3 value (never rotated)
//   values            v = fp16(scale) * code + fp16(zero)
//
// Differences from the pages' design: the pages expand to fp16 in one kernel
// and then rotate back with an fp16 matrix product against a copy of the
// Hadamard matrix; here a half-warp per (position, KV head) holds the 128
// coordinates in registers (8 per lane), applies the inverse rotation as an
// fp32 butterfly (3 in-lane stages + 4 xor-shuffle stages) and rounds once, to
// the caller's output type. Nothing intermediate is written.

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

constexpr int kDequantWarps = 8;
constexpr int kD = 128;

struct DequantArgs {
  const uint8_t* cache;
  const int* block_table;
  const int* seq_lens;
  void* key_out;
  void* value_out;
  unsigned int* status;
  long long num_blocks;
  int n_kv;
  int max_seq_len;
  int len_cap;               // min(max_seq_len, bt_stride * block_size)
  int seq_tiles;             // ceil(max_seq_len / 16): CTAs per (sequence, KV head)
  int bt_stride;
  int log2_bs;
  int tiles_per_block;
  int tile_bytes;
  int k_off, k_row;
  int v_off, v_row;
  int knorm_off, vscale_off, vzero_off;
  float cent[16];
};

enum KeyMode { kMse4 = 4, kMse3 = 3, kFp8 = 8 };

// Sylvester-order Walsh-Hadamard transform of 128 coordinates held by a
// half-warp, 8 consecutive values per lane (coordinate 8 * l + j for lane l of
// the half), unnormalised: coordinate strides 1, 2, 4 inside the lane, then
// 8 .. 64 across lanes l ^ 1 .. l ^ 8. The lane whose stride bit is set keeps
// (partner - own), the other (own + partner); both as one exact fma with +-1.
__device__ __forceinline__ void fwht128_half(float v[8], int l) {
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
    const float sgn = (l & m) ? -1.f : 1.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = fmaf(sgn, v[j], __shfl_xor_sync(0xffffffffu, v[j], m));
  }
}

template <typename T>
__device__ __forceinline__ void store8(void* base, long long elem, const float x[8]) {
  if constexpr (std::is_same<T, float>::value) {
    float4* d = reinterpret_cast<float4*>(static_cast<float*>(base) + elem);
    d[0] = make_float4(x[0], x[1], x[2], x[3]);
    d[1] = make_float4(x[4], x[5], x[6], x[7]);
  } else {
    uint4 w;
    uint32_t* wp = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if constexpr (std::is_same<T, __nv_bfloat16>::value) {
        const __nv_bfloat162 t = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
        wp[i] = *reinterpret_cast<const uint32_t*>(&t);
      } else {
        const __half2 t = __floats2half2_rn(x[2 * i], x[2 * i + 1]);
        wp[i] = *reinterpret_cast<const uint32_t*>(&t);
      }
    }
    *reinterpret_cast<uint4*>(static_cast<T*>(base) + elem) = w;
  }
}

__device__ __forceinline__ float half_bits(const uint8_t* p) {
  return __half2float(__ushort_as_half(ld_dep_u16(p)));
}

// One CTA per (sequence, 16-position tile, KV head): grid (seq_tiles * batch,
// n_kv). Warp w expands positions 2w and 2w + 1 of the tile, one per
// half-warp; lane l of a half holds coordinates 8l .. 8l + 7.
template <int KMODE, int VBITS, typename T>
__global__ void __launch_bounds__(kDequantWarps * 32)
dequant_kernel(const DequantArgs a) {
  grid_dep_wait();   // cache, tables and lengths may come from the previous kernel
  grid_dep_launch();
  __shared__ float s_cent[16];
  if (threadIdx.x < 16) s_cent[threadIdx.x] = a.cent[threadIdx.x];
  __syncthreads();

  const int b = static_cast<int>(blockIdx.x / static_cast<unsigned>(a.seq_tiles));
  const int t = static_cast<int>(blockIdx.x - static_cast<unsigned>(b) * static_cast<unsigned>(a.seq_tiles));
  const int h = blockIdx.y;
  const int lane = threadIdx.x & 31;
  const int l = lane & 15;
  const int r = 2 * (threadIdx.x >> 5) + (lane >> 4);   // row of the tile
  const int p = 16 * t + r;
  // rows past max_seq_len (the last tile) are not in the output; their lanes
  // stay to the end, since the butterfly's shuffles need the whole warp
  const bool in_out = p < a.max_seq_len;
  const long long elem = ((static_cast<long long>(b) * a.max_seq_len + p) * a.n_kv + h) * kD + 8 * l;

  const int raw_len = ld_dep_s32(a.seq_lens + b);
  if (p == 0 && h == 0 && lane == 0 && raw_len > a.len_cap && a.status) atomicOr(a.status, TQ_DEV_SEQ_TOO_LONG);
  const int len = min(max(raw_len, 0), a.len_cap);
  float k[8], v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) k[j] = v[j] = 0.f;
  // the whole tile lies in one cache block; its id is read only if the tile
  // holds a cached position
  int blk = -1;
  if (16 * t < len) {
    blk = ld_dep_s32(a.block_table + static_cast<long long>(b) * a.bt_stride + ((16 * t) >> a.log2_bs));
    if ((blk < 0 || blk >= a.num_blocks) && threadIdx.x == 0 && a.status) atomicOr(a.status, TQ_DEV_BLOCK_OUT_OF_RANGE);
  }
  const bool live = p < len && blk >= 0 && blk < a.num_blocks;
  if (live) {
    const int off = (16 * t) & ((1 << a.log2_bs) - 1);
    const uint8_t* tile = a.cache + ((static_cast<long long>(blk) * a.n_kv + h) * a.tiles_per_block + (off >> 4)) *
                                        static_cast<long long>(a.tile_bytes);
    const uint8_t* krow = tile + a.k_off + r * a.k_row;
    if constexpr (KMODE == kFp8) {
      const uint2 w = ld_dep_u32x2(krow + 8 * l);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t word = i < 2 ? w.x : w.y;
        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(
            static_cast<__nv_fp8x2_storage_t>((word >> (16 * (i & 1))) & 0xFFFFu), __NV_E4M3);
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
        k[2 * i] = f.x;
        k[2 * i + 1] = f.y;
      }
    } else {
      uint32_t w;
      if constexpr (KMODE == kMse4) {
        w = ld_dep_u32(krow + 4 * l);
      } else {
        const uint8_t* g = krow + 3 * l;   // 24 bits, LSB first
        w = ld_dep_u8(g) | (ld_dep_u8(g + 1) << 8) | (ld_dep_u8(g + 2) << 16);
      }
      const float nrm = half_bits(tile + a.knorm_off + 2 * r);
#pragma unroll
      for (int j = 0; j < 8; ++j) k[j] = nrm * s_cent[(w >> (KMODE * j)) & ((1u << KMODE) - 1)];
    }
    const int pair = r >> 1;
    uint32_t codes;   // this lane's codes, LSB-first: coordinate 8 l + j at bit VBITS j
    if constexpr (VBITS == 4) {
      // value words 2l and 2l + 1 of token r = 2 * pair + (r & 1): one 8-byte
      // group holding both words of both tokens of the pair (pair-interleaved,
      // 16-byte groups swizzled by the pair index when rows are 64 bytes)
      const int swz = (a.v_row % 64 == 0) ? 2 * (pair & 3) : 0;
      const uint2 vw = ld_dep_u32x2(tile + a.v_off + pair * 2 * a.v_row + 16 * ((l >> 1) ^ swz) + 8 * (l & 1));
      codes = ((vw.x >> (16 * (r & 1))) & 0xFFFFu) | (((vw.y >> (16 * (r & 1))) & 0xFFFFu) << 16);
    } else {
      // 24 bits from bit 24 l of the token's stream: 16-bit words 3 m and
      // 3 m + 1 (l = 2 m, bits 0-23 of the pair) or 3 m + 1 and 3 m + 2 (l =
      // 2 m + 1, bits 8-31); the pair's 32-bit word i (no swizzle at 48-byte
      // rows) holds word i of both tokens
      const int w0 = 3 * (l >> 1) + (l & 1);
      const uint8_t* pw = tile + a.v_off + pair * 2 * a.v_row + 4 * w0;
      const int sh = 16 * (r & 1);
      const uint32_t lo = (ld_dep_u32(pw) >> sh) & 0xFFFFu, hi = (ld_dep_u32(pw + 4) >> sh) & 0xFFFFu;
      codes = (lo | (hi << 16)) >> (8 * (l & 1));
    }
    const float s = half_bits(tile + a.vscale_off + 2 * r);
    const float z = half_bits(tile + a.vzero_off + 2 * r);
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = fmaf(s, static_cast<float>((codes >> (VBITS * j)) & ((1u << VBITS) - 1)), z);
  }
  if constexpr (KMODE != kFp8) {
    // every half-warp of the warp runs the butterfly (its shuffles need all
    // 32 lanes); rows that hold no key transform zeros
    fwht128_half(k, l);
#pragma unroll
    for (int j = 0; j < 8; ++j) k[j] *= 0.088388347648318440f;   // 1 / sqrt(128)
  }
  if (in_out) {
    store8<T>(a.key_out, elem, k);
    store8<T>(a.value_out, elem, v);
  }
}

template <int KMODE, int VBITS>
cudaError_t launch_dequant(const DequantArgs& a, int batch, int out_dtype, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(static_cast<long long>(a.seq_tiles) * batch), static_cast<unsigned>(a.n_kv));
  const dim3 block(kDequantWarps * 32);
  if (out_dtype == TQ_DTYPE_BF16)
    return launch_pdl(dequant_kernel<KMODE, VBITS, __nv_bfloat16>, grid, block, 0, stream, a);
  if (out_dtype == TQ_DTYPE_F16) return launch_pdl(dequant_kernel<KMODE, VBITS, __half>, grid, block, 0, stream, a);
  return launch_pdl(dequant_kernel<KMODE, VBITS, float>, grid, block, 0, stream, a);
}

}  // namespace
}  // namespace tq

extern "C" tq_status tq_dequant(const tq_config* cfg, const tq_codebook* cb,
                                const void* cache, long long num_blocks,
                                const int* block_table, int bt_stride,
                                const int* seq_lens, int batch, int max_seq_len,
                                void* key_out, void* value_out, int out_dtype,
                                unsigned int* dev_status, tq_stream_t stream) {
  using namespace tq;
  tq_layout L;
  const tq_status st = make_layout(cfg, &L);
  if (st != TQ_OK) return st;
  if (batch < 0 || max_seq_len < 0 || num_blocks < 0 || bt_stride < 1) return TQ_ERR_INVALID_ARG;
  if (out_dtype != TQ_DTYPE_F16 && out_dtype != TQ_DTYPE_BF16 && out_dtype != TQ_DTYPE_F32)
    return TQ_ERR_INVALID_ARG;
  if (!L.key_fp8 && (!cb || cb->bits != L.key_bits || cb->head_dim != cfg->head_dim)) return TQ_ERR_INVALID_ARG;
  if (batch == 0 || max_seq_len == 0) return TQ_OK;
  if (!cache || !block_table || !seq_lens || !key_out || !value_out) return TQ_ERR_INVALID_ARG;
  if (!aligned16(cache) || !aligned16(key_out) || !aligned16(value_out) ||
      (reinterpret_cast<unsigned long long>(block_table) & 3ull) ||
      (reinterpret_cast<unsigned long long>(seq_lens) & 3ull))
    return TQ_ERR_MISALIGNED;
  if (dev_status && (reinterpret_cast<unsigned long long>(dev_status) & 3ull)) return TQ_ERR_MISALIGNED;
  const long long seq_tiles = (static_cast<long long>(max_seq_len) + kTileTokens - 1) / kTileTokens;
  if (seq_tiles * batch > 0x7fffffffll || cfg->num_kv_heads > 65535) return TQ_ERR_INVALID_ARG;

  DequantArgs a;
  a.cache = static_cast<const uint8_t*>(cache);
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.key_out = key_out;
  a.value_out = value_out;
  a.status = dev_status;
  a.num_blocks = num_blocks;
  a.n_kv = cfg->num_kv_heads;
  a.max_seq_len = max_seq_len;
  a.seq_tiles = static_cast<int>(seq_tiles);
  const long long cap = static_cast<long long>(bt_stride) * cfg->block_size;
  a.len_cap = static_cast<int>(cap < max_seq_len ? cap : max_seq_len);
  a.bt_stride = bt_stride;
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
  for (int i = 0; i < 16; ++i) a.cent[i] = (!L.key_fp8 && i < cb->num_levels) ? cb->centroids[i] : 0.f;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t err;
  if (L.key_fp8) err = launch_dequant<kFp8, 4>(a, batch, out_dtype, s);
  else if (L.key_bits == 4) err = launch_dequant<kMse4, 4>(a, batch, out_dtype, s);
  else if (L.value_bits == 4) err = launch_dequant<kMse3, 4>(a, batch, out_dtype, s);
  else err = launch_dequant<kMse3, 3>(a, batch, out_dtype, s);
  return err == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}
