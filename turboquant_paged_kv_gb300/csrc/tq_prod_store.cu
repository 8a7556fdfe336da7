// tq_prod_store: TurboQuant_prod keys — a 2-bit Lloyd-Max code plus a 1-bit
// QJL sign of the residual per coordinate — written into the key-only
// paged cache.
//
// Method: "vLLM 源码完全拆解(十九):TurboQuant KV Cache 量化" (pinghaoyang.com.cn),
// section "Lloyd-Max 量化器" (TurboQuant_prod = the MSE quantizer plus a 1-bit
// QJL layer on its residual, unbiased for inner products), and the page on
// the open-source turboquant project (kwkr.cn/news/555717), subsection
// "最后 1 bit 的巧思": the (b - 1)-bit code of the rotated unit vector gives
// x~; r = x - x~ is projected by a Gaussian matrix S and only the signs are
// kept, with ||r||; <y, x> is estimated as <y, x~> + ||r|| sqrt(pi / 2) / d
// <S y, signs>.
//
// GB300 design:
//   store   one CTA per SM loops over groups of 128 vectors. Each thread
//           issues all of a group's key and slot loads at once (the next
//           group's go out while the current one is projected). A half-warp
//           per vector rotates and quantises (as tq_store does) and leaves the
//           residual r in shared memory; then each warp computes S r for 16
//           vectors on tensor cores (mma.sync TF32, three products of hi/lo
//           splits, so the result carries fp32 accuracy) and packs the signs
//           with warp ballots.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>
#include <type_traits>

#include "tq_internal.h"
#include "tq_launch.cuh"
#include "tq_prod.cuh"
#include "tq_vec.cuh"

namespace tq {
namespace {

constexpr int kGroupVecs = 128;              // vectors per CTA pass of the store

// TF32 (10-bit mantissa) rounding of x, round to nearest, ties away (cvt.rna).
__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(x));
  return r;
}

// x = hi + lo with hi, lo TF32: the three products hi*hi + hi*lo + lo*hi of
// two such pairs give the fp32 product to ~2^-21 relative.
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  hi = to_tf32(x);
  lo = to_tf32(x - __uint_as_float(hi));
}

__device__ __forceinline__ void mma_tf32(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Row stride (floats) of the shared S and R tables: 136 = 8 mod 32, so the
// 8-byte operand loads of a half-warp (rows g, columns 2 t) are conflict-free.
constexpr int kPad = 136;

struct ProdStoreArgs {
  const void* key;
  const long long* slots;
  const float* S;
  uint8_t* cache;
  unsigned int* status;
  long long num_vectors, num_blocks;
  int n_kv, block_size, log2_bs, tiles_per_block;
  unsigned kv_magic, kv_shift;
  float mid[3];
  float cent[4];
};

// Shared memory: S as TF32 hi and lo parts and the group's residuals R, each
// [128][kPad] floats; the tile and row of each vector of the group (null
// tile: nothing to write).
constexpr size_t kStoreSmem = 3 * static_cast<size_t>(kD) * kPad * sizeof(float) +
                              kGroupVecs * (sizeof(uint8_t*) + sizeof(int));

// The inputs of one group for the thread (half-warp h = threadIdx.x / 16,
// lane l of it): the 8 keys' coordinates 8 l .. 8 l + 7 of vectors p 16 + h
// and their tokens' slots, all loads issued at once (slot -1: past the end).
template <typename T>
__device__ __forceinline__ void load_group(const ProdStoreArgs& a, long long grp, int h, int l, uint4 key[8],
                                           long long slot[8]) {
#pragma unroll
  for (int p = 0; p < kGroupVecs / 16; ++p) {
    const long long vec = grp * kGroupVecs + p * 16 + h;
    if (vec < a.num_vectors) {
      const long long tok = a.num_vectors < (1ll << 31)
                                ? static_cast<long long>(__umulhi(2u * static_cast<unsigned>(vec), a.kv_magic) >> a.kv_shift)
                                : vec / a.n_kv;
      slot[p] = ld_dep_s64(a.slots + tok);
      key[p] = ld_dep_u32x4(static_cast<const T*>(a.key) + vec * kD + 8 * l);
    } else {
      slot[p] = -1;
      key[p] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

template <typename T>
__device__ __forceinline__ void unpack8(const uint4 raw, float out[8]) {
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

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) prod_store_kernel(const ProdStoreArgs a) {
  extern __shared__ __align__(16) float s_store[];
  uint32_t* s_hi = reinterpret_cast<uint32_t*>(s_store);   // S[i][j] at i * kPad + j
  uint32_t* s_lo = s_hi + kD * kPad;
  float* R = s_store + 2 * kD * kPad;                       // R[v][j] at v * kPad + j
  uint8_t** tiles = reinterpret_cast<uint8_t**>(R + kGroupVecs * kPad);
  int* trow = reinterpret_cast<int*>(tiles + kGroupVecs);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, l = lane & 15, hv = threadIdx.x >> 4;
  const long long groups = (a.num_vectors + kGroupVecs - 1) / kGroupVecs;
  grid_dep_wait();   // S, keys, slots and cache may come from the previous kernel
  grid_dep_launch();
  // the first group's loads go out before S is staged, so the two wait together
  uint4 key[kGroupVecs / 16];
  long long slot[kGroupVecs / 16];
  long long grp = blockIdx.x;
  if (grp < groups) load_group<T>(a, grp, hv, l, key, slot);
  {
    constexpr int kPer = kD * kD / 4 / kThreads;   // 16 float4 per thread, all in flight
    float4 v[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) v[k] = ld_dep_f32x4(reinterpret_cast<const float4*>(a.S) + threadIdx.x + k * kThreads);
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int e = 4 * (threadIdx.x + k * kThreads), i = e >> 7, j = e & (kD - 1);
      const float x[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) split_tf32(x[q], s_hi[i * kPad + j + q], s_lo[i * kPad + j + q]);
    }
  }
  for (; grp < groups; grp += gridDim.x) {
    // ---- phase 1: a half-warp per vector, 16 vectors per pass
#pragma unroll
    for (int pass = 0; pass < kGroupVecs / 16; ++pass) {
      const int gv = pass * 16 + hv;   // vector of the group
      const long long vec = grp * kGroupVecs + gv;
      bool live = slot[pass] >= 0;
      uint8_t* tile = nullptr;
      int r = 0;
      if (live) {
        const long long blk = slot[pass] >> a.log2_bs;
        if (blk >= a.num_blocks) {
          if (l == 0) flag(a.status, TQ_DEV_SLOT_OUT_OF_RANGE);
          live = false;
        } else {
          const long long tok = a.num_vectors < (1ll << 31)
                                    ? static_cast<long long>(__umulhi(2u * static_cast<unsigned>(vec), a.kv_magic) >> a.kv_shift)
                                    : vec / a.n_kv;
          const int head = static_cast<int>(vec - tok * a.n_kv);
          const int off = static_cast<int>(slot[pass] & (a.block_size - 1));
          tile = a.cache + ((blk * a.n_kv + head) * a.tiles_per_block + (off >> 4)) * static_cast<long long>(kTileBytes);
          r = off & 15;
        }
      }
      float k[8];
      unpack8<T>(key[pass], k);
      if (!live) {
#pragma unroll
        for (int j = 0; j < 8; ++j) k[j] = 0.f;
      }
      float ss = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) ss = fmaf(k[j], k[j], ss);
      ss = half_sum(ss);
      const float n = ss > 0.f ? ss * rsqrtf(ss) : 0.f;
      fwht128_half(k, l);
      const float sc = __fdividef(0.088388347648318440f, n + 1e-8f);   // 1/sqrt(128) / (n + 1e-8)
      uint32_t code = 0;
      float res[8], rr = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float y = k[j] * sc;
        // #{m : y >= mid_m} over the 3 ascending midpoints
        int c = (y >= a.mid[1]) ? 2 : 0;
        c += (y >= (c ? a.mid[2] : a.mid[0])) ? 1 : 0;
        code |= static_cast<uint32_t>(c) << (kMseBits * j);
        const float cv = c == 0 ? a.cent[0] : (c == 1 ? a.cent[1] : (c == 2 ? a.cent[2] : a.cent[3]));
        res[j] = y - cv;
        rr = fmaf(res[j], res[j], rr);
      }
      rr = half_sum(rr);
      float* rrow = R + gv * kPad + 8 * l;
      *reinterpret_cast<float4*>(rrow) = make_float4(res[0], res[1], res[2], res[3]);
      *reinterpret_cast<float4*>(rrow + 4) = make_float4(res[4], res[5], res[6], res[7]);
      if (l == 0) {
        tiles[gv] = live ? tile : nullptr;
        trow[gv] = r;
      }
      if (live) {
        *reinterpret_cast<uint16_t*>(tile + kKOff + r * kKRow + 2 * l) = static_cast<uint16_t>(code);
        if (l == 0) {
          *reinterpret_cast<uint16_t*>(tile + kNormOff + 2 * r) = __half_as_ushort(__float2half_rn(n));
          *reinterpret_cast<uint16_t*>(tile + kRnormOff + 2 * r) =
              __half_as_ushort(__float2half_rn(rr > 0.f ? rr * rsqrtf(rr) : 0.f));
        }
      }
    }
    // the next group's loads are in flight during the projection
    if (grp + gridDim.x < groups) load_group<T>(a, grp + gridDim.x, hv, l, key, slot);
    __syncthreads();
    // ---- phase 2: warp w projects vectors 16 w .. 16 w + 15 on tensor cores:
    // P[v][i] = sum_j R[v][j] S[i][j], mma.sync m16n8k8 TF32 with A = R (rows
    // v), B = S^T, three products per step (hi*hi + hi*lo + lo*hi). The k
    // order inside a step is permuted so a lane's two operand values are
    // adjacent (k slots t and t + 4 hold columns 2 t and 2 t + 1 of the step):
    // A and B use the same order, so the sums are unchanged.
    const int g = lane >> 2, t = lane & 3;
    float acc[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    const float* Rw = R + warp * 16 * kPad;
#pragma unroll 1
    for (int k0 = 0; k0 < kD; k0 += 8) {
      const float2 rg = *reinterpret_cast<const float2*>(Rw + g * kPad + k0 + 2 * t);
      const float2 rh = *reinterpret_cast<const float2*>(Rw + (g + 8) * kPad + k0 + 2 * t);
      uint32_t ah[4], al[4];   // (row g, slot t), (row g + 8, slot t), (row g, slot t + 4), (row g + 8, slot t + 4)
      split_tf32(rg.x, ah[0], al[0]);
      split_tf32(rh.x, ah[1], al[1]);
      split_tf32(rg.y, ah[2], al[2]);
      split_tf32(rh.y, ah[3], al[3]);
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        const int n = 8 * nt + g;   // B column: output row i = n of S
        const uint2 bh = *reinterpret_cast<const uint2*>(s_hi + n * kPad + k0 + 2 * t);
        const uint2 bl = *reinterpret_cast<const uint2*>(s_lo + n * kPad + k0 + 2 * t);
        mma_tf32(acc[nt], ah, bh.x, bh.y);
        mma_tf32(acc[nt], ah, bl.x, bl.y);
        mma_tf32(acc[nt], al, bh.x, bh.y);
      }
    }
    // signs: acc[nt][e] is P[16 w + g + 8 (e >> 1)][8 nt + 2 t + (e & 1)]. The
    // ballot of (nt, e) gives bit 4 g' + t' = the sign of output 8 nt + 2 t' +
    // (e & 1) of vector g' (+ 8): one byte of a vector's stream per (nt, half)
    // from the two parities. Lane (g, t) assembles bytes nt = 4 t .. 4 t + 3 of
    // vectors 16 w + g and 16 w + g + 8, i.e. word t of their 128-bit streams.
    uint32_t word[2] = {0u, 0u};
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const uint32_t m0 = __ballot_sync(0xffffffffu, acc[nt][2 * hf] >= 0.f);
        const uint32_t m1 = __ballot_sync(0xffffffffu, acc[nt][2 * hf + 1] >= 0.f);
        if ((nt >> 2) == t) {
          const uint32_t n0 = (m0 >> (4 * g)) & 0xFu, n1 = (m1 >> (4 * g)) & 0xFu;
          // bit t' of n0 -> bit 2 t', of n1 -> bit 2 t' + 1
          const uint32_t s0 = (n0 & 1u) | ((n0 & 2u) << 1) | ((n0 & 4u) << 2) | ((n0 & 8u) << 3);
          const uint32_t s1 = (n1 & 1u) | ((n1 & 2u) << 1) | ((n1 & 4u) << 2) | ((n1 & 8u) << 3);
          word[hf] |= (s0 | (s1 << 1)) << (8 * (nt & 3));
        }
      }
    }
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int gv = warp * 16 + g + 8 * hf;
      uint8_t* tile = tiles[gv];
      if (tile) *reinterpret_cast<uint32_t*>(tile + kSOff + trow[gv] * kSRow + 4 * t) = word[hf];
    }
    __syncthreads();   // R and tiles are rewritten by the next group
  }
}

void fill_magic(int n, unsigned* magic, unsigned* shift) {
  unsigned sh = 0;
  while ((1u << sh) < static_cast<unsigned>(n)) ++sh;
  *shift = sh;
  *magic = static_cast<unsigned>(((1ull << (31 + sh)) + n - 1) / n);
}

}  // namespace
}  // namespace tq

extern "C" {

tq_status tq_prod_store(const tq_config* cfg, const tq_codebook* cb, const float* S, const void* key, int in_dtype,
                        long long num_tokens, const long long* slot_mapping, void* cache, long long num_blocks,
                        unsigned int* dev_status, tq_stream_t stream) {
  using namespace tq;
  tq_prod_layout L;
  const tq_status st = prod_layout(cfg, &L);
  if (st != TQ_OK) return st;
  if (num_tokens < 0 || num_blocks < 0) return TQ_ERR_INVALID_ARG;
  if (in_dtype != TQ_DTYPE_F16 && in_dtype != TQ_DTYPE_BF16) return TQ_ERR_INVALID_ARG;
  if (!cb || cb->bits != kMseBits || cb->head_dim != cfg->head_dim) return TQ_ERR_INVALID_ARG;
  if (num_tokens == 0) return TQ_OK;
  if (!S || !key || !slot_mapping || !cache) return TQ_ERR_INVALID_ARG;
  if (!aligned16(S) || !aligned16(key) || !aligned16(cache) || (reinterpret_cast<unsigned long long>(slot_mapping) & 7ull))
    return TQ_ERR_MISALIGNED;
  if (dev_status && (reinterpret_cast<unsigned long long>(dev_status) & 3ull)) return TQ_ERR_MISALIGNED;
  const long long vectors = num_tokens * cfg->num_kv_heads;
  ProdStoreArgs a;
  a.key = key;
  a.slots = slot_mapping;
  a.S = S;
  a.cache = static_cast<uint8_t*>(cache);
  a.status = dev_status;
  a.num_vectors = vectors;
  a.num_blocks = num_blocks;
  a.n_kv = cfg->num_kv_heads;
  a.block_size = cfg->block_size;
  a.log2_bs = __builtin_ctz(static_cast<unsigned>(cfg->block_size));
  a.tiles_per_block = cfg->block_size / kTileTokens;
  fill_magic(a.n_kv, &a.kv_magic, &a.kv_shift);
  for (int i = 0; i < 3; ++i) a.mid[i] = cb->midpoints[i];
  for (int i = 0; i < 4; ++i) a.cent[i] = cb->centroids[i];
  const int sms = sm_count();
  if (sms <= 0) return TQ_ERR_CUDA;
  const long long groups = (vectors + kGroupVecs - 1) / kGroupVecs;
  const unsigned grid = static_cast<unsigned>(groups < sms ? groups : sms);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t err;
  if (in_dtype == TQ_DTYPE_BF16) {
    err = cudaFuncSetAttribute(prod_store_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kStoreSmem));
    if (err == cudaSuccess)
      err = launch_pdl(prod_store_kernel<__nv_bfloat16>, dim3(grid), dim3(kThreads), kStoreSmem, s, a);
  } else {
    err = cudaFuncSetAttribute(prod_store_kernel<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kStoreSmem));
    if (err == cudaSuccess) err = launch_pdl(prod_store_kernel<__half>, dim3(grid), dim3(kThreads), kStoreSmem, s, a);
  }
  return err == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // extern "C"
