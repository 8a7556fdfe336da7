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
//   store   two CTAs per SM (105 KB of shared memory, 128 registers each)
//           loop over groups of 64 vectors. Each thread issues all of a
//           group's key and slot loads at once (the next group's go out while
//           the current one is projected). A half-warp per vector rotates and
//           quantises (as tq_store does) and leaves the residual, scaled by
//           2^6, in shared memory as fp16 hi and lo parts; then each warp
//           computes 64 rows of S r for 16 vectors on tensor cores (mma.sync
//           m16n8k16 f16, three products of the hi/lo splits, f32 sums: the
//           result carries fp32 accuracy) and packs the signs with warp
//           ballots.

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

constexpr int kGroupVecs = 64;               // vectors per CTA pass of the store
constexpr int kCtasPerSm = 2;

// x = hi + lo with hi, lo fp16 (hi = fp16(x), lo = fp16(x - hi)): the three
// products hi*hi + hi*lo + lo*hi of two such pairs give the product to about
// 2^-21 relative, fp32's accuracy, as long as the lo parts stay normal (the
// residuals are scaled by 2^6 for that; S is N(0, 1)).
__device__ __forceinline__ void split_h2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
  const __half l0 = __float2half_rn(x0 - __half2float(h0)), l1 = __float2half_rn(x1 - __half2float(h1));
  hi = static_cast<uint32_t>(__half_as_ushort(h0)) | (static_cast<uint32_t>(__half_as_ushort(h1)) << 16);
  lo = static_cast<uint32_t>(__half_as_ushort(l0)) | (static_cast<uint32_t>(__half_as_ushort(l1)) << 16);
}

__device__ __forceinline__ void mma_f16(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Row stride (halves) of the shared S and R tables: 136 halves = 68 words =
// 4 mod 32, so the 4-byte operand loads of a warp (rows g, words t) hit 32
// different banks.
constexpr int kPad = 136;
constexpr float kResidualScale = 64.f;   // exact; scales S r by 2^6, so no sign changes

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

// Shared memory: S as fp16 hi and lo parts, [128][kPad] halves each; the
// group's scaled residuals R as fp16 hi and lo parts, [64][kPad] halves each;
// the tile and row of each vector of the group (null tile: nothing to write).
// 105 KB: two CTAs per SM.
constexpr size_t kStoreSmem = 2 * static_cast<size_t>(kD) * kPad * 2 + 2 * static_cast<size_t>(kGroupVecs) * kPad * 2 +
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
__global__ void __launch_bounds__(kThreads, kCtasPerSm) prod_store_kernel(const ProdStoreArgs a) {
  extern __shared__ __align__(16) uint16_t s_store[];
  uint16_t* s_hi = s_store;                   // S[i][j] at i * kPad + j (halves)
  uint16_t* s_lo = s_hi + kD * kPad;
  uint16_t* r_hi = s_lo + kD * kPad;          // 2^6 R[v][j] at v * kPad + j
  uint16_t* r_lo = r_hi + kGroupVecs * kPad;
  uint8_t** tiles = reinterpret_cast<uint8_t**>(r_lo + kGroupVecs * kPad);
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
      uint32_t h01, l01, h23, l23;
      split_h2(v[k].x, v[k].y, h01, l01);
      split_h2(v[k].z, v[k].w, h23, l23);
      *reinterpret_cast<uint2*>(s_hi + i * kPad + j) = make_uint2(h01, h23);
      *reinterpret_cast<uint2*>(s_lo + i * kPad + j) = make_uint2(l01, l23);
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
      uint32_t rh[4], rl[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) split_h2(kResidualScale * res[2 * q], kResidualScale * res[2 * q + 1], rh[q], rl[q]);
      *reinterpret_cast<uint4*>(r_hi + gv * kPad + 8 * l) = make_uint4(rh[0], rh[1], rh[2], rh[3]);
      *reinterpret_cast<uint4*>(r_lo + gv * kPad + 8 * l) = make_uint4(rl[0], rl[1], rl[2], rl[3]);
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
    // ---- phase 2: warp w projects vectors 16 vb .. 16 vb + 15 (vb = w % 4) onto
    // rows 64 oh .. 64 oh + 63 of S (oh = w / 4) on tensor cores: 2^6 P[v][i] =
    // sum_j 2^6 R[v][j] S[i][j], mma.sync m16n8k16 f16 with A = R (rows v),
    // B = S^T, three products per step (hi*hi + hi*lo + lo*hi), f32 sums.
    const int g = lane >> 2, t = lane & 3, vb = warp & 3, oh = warp >> 2;
    float acc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    const uint16_t* rh0 = r_hi + (16 * vb + g) * kPad + 2 * t;
    const uint16_t* rl0 = r_lo + (16 * vb + g) * kPad + 2 * t;
    const uint16_t* sh0 = s_hi + (64 * oh + g) * kPad + 2 * t;
    const uint16_t* sl0 = s_lo + (64 * oh + g) * kPad + 2 * t;
#pragma unroll 2
    for (int k0 = 0; k0 < kD; k0 += 16) {
      uint32_t ah[4], al[4];   // (row g, k 2t), (row g + 8, k 2t), (row g, k 2t + 8), (row g + 8, k 2t + 8)
      ah[0] = *reinterpret_cast<const uint32_t*>(rh0 + k0);
      ah[1] = *reinterpret_cast<const uint32_t*>(rh0 + 8 * kPad + k0);
      ah[2] = *reinterpret_cast<const uint32_t*>(rh0 + k0 + 8);
      ah[3] = *reinterpret_cast<const uint32_t*>(rh0 + 8 * kPad + k0 + 8);
      al[0] = *reinterpret_cast<const uint32_t*>(rl0 + k0);
      al[1] = *reinterpret_cast<const uint32_t*>(rl0 + 8 * kPad + k0);
      al[2] = *reinterpret_cast<const uint32_t*>(rl0 + k0 + 8);
      al[3] = *reinterpret_cast<const uint32_t*>(rl0 + 8 * kPad + k0 + 8);
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {   // B column n = 64 oh + 8 nt + g: row n of S
        const uint32_t bh0 = *reinterpret_cast<const uint32_t*>(sh0 + 8 * nt * kPad + k0);
        const uint32_t bh1 = *reinterpret_cast<const uint32_t*>(sh0 + 8 * nt * kPad + k0 + 8);
        const uint32_t bl0 = *reinterpret_cast<const uint32_t*>(sl0 + 8 * nt * kPad + k0);
        const uint32_t bl1 = *reinterpret_cast<const uint32_t*>(sl0 + 8 * nt * kPad + k0 + 8);
        mma_f16(acc[nt], ah, bh0, bh1);
        mma_f16(acc[nt], ah, bl0, bl1);
        mma_f16(acc[nt], al, bh0, bh1);
      }
    }
    // signs: acc[nt][e] is 2^6 P[16 vb + g + 8 (e >> 1)][64 oh + 8 nt + 2 t +
    // (e & 1)]. The ballot of (nt, e) gives bit 4 g' + t' = the sign of output
    // 64 oh + 8 nt + 2 t' + (e & 1) of vector g' (+ 8): byte 8 oh + nt of a
    // vector's stream per (nt, half) from the two parities. Lane (g, t < 2)
    // assembles bytes nt = 4 t .. 4 t + 3 of vectors 16 vb + g and 16 vb + g +
    // 8, i.e. word 2 oh + t of their 128-bit streams.
    uint32_t word[2] = {0u, 0u};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
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
    if (t < 2) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int gv = 16 * vb + g + 8 * hf;
        uint8_t* tile = tiles[gv];
        if (tile) *reinterpret_cast<uint32_t*>(tile + kSOff + trow[gv] * kSRow + 4 * (2 * oh + t)) = word[hf];
      }
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
  const long long resident = static_cast<long long>(kCtasPerSm) * sms;
  const unsigned grid = static_cast<unsigned>(groups < resident ? groups : resident);
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
