// tq_prod: TurboQuant_prod keys — a 2-bit Lloyd-Max code plus a 1-bit QJL
// sign of the residual per coordinate — stored into a key-only paged cache,
// and the unbiased inner-product estimates read back from it.
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
//   store   one CTA per SM loops over groups of 128 vectors. A half-warp per
//           vector rotates and quantises (as tq_store does) and leaves the
//           residual r in shared memory; then each warp computes S r for 16
//           vectors as an fp32 register-blocked product (lane l: rows 4 l ..
//           4 l + 3 of S for all 16 vectors, S transposed in shared memory so
//           a lane's four rows are one 16-byte load) and packs the signs with
//           warp ballots.
//   scores  a prep kernel rotates each query head (warp butterfly) and forms
//           S q_r once; the scores kernel gives each warp 16-position tiles
//           of one (sequence, KV head), two lanes per position (64
//           coordinates each), the G query heads' q_r and S q_r staged in
//           shared memory and read as broadcasts.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>
#include <type_traits>

#include "tq_internal.h"
#include "tq_launch.cuh"
#include "tq_vec.cuh"

namespace tq {
namespace {

constexpr int kD = 128;
constexpr int kMseBits = 2;
constexpr int kKRow = kD * kMseBits / 8;     // 32 index bytes per position
constexpr int kSRow = kD / 8;                // 16 sign bytes per position
constexpr int kKOff = 0;
constexpr int kSOff = 16 * kKRow;            // 512
constexpr int kNormOff = kSOff + 16 * kSRow; // 768
constexpr int kRnormOff = kNormOff + 32;     // 800
constexpr int kTileBytes = kRnormOff + 32;   // 832 = 16 x 52
constexpr int kGroupVecs = 128;              // vectors per CTA pass of the store
constexpr int kThreads = 256;
constexpr float kQjlScale = 1.2533141373155003f / kD;   // sqrt(pi / 2) / d

__device__ __forceinline__ void flag(unsigned int* status, unsigned int bit) {
  if (status) atomicOr(status, bit);
}

// Spread the 8 bits of b to bits 0, 4, 8, .., 28.
__device__ __forceinline__ uint32_t spread4(uint32_t b) {
  b = (b | (b << 12)) & 0x000F000Fu;
  b = (b | (b << 6)) & 0x03030303u;
  b = (b | (b << 3)) & 0x11111111u;
  return b;
}

// S^T into shared memory: sT[j * 128 + i] = S[i][j].
__device__ void load_st(float* sT, const float* S) {
  for (int e = threadIdx.x; e < kD * kD; e += blockDim.x) {
    const int j = e >> 7, i = e & (kD - 1);
    sT[e] = ld_dep_f32(S + i * kD + j);
  }
}

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

// Shared memory: S^T (64 KB), residuals R[128][128] (64 KB), the tile and
// row of each vector of the group (null tile: nothing to write).
constexpr size_t kStoreSmem = 2 * kD * kD * sizeof(float) + kGroupVecs * (sizeof(uint8_t*) + sizeof(int));

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) prod_store_kernel(const ProdStoreArgs a) {
  extern __shared__ __align__(16) float s_store[];
  float* sT = s_store;
  float* R = s_store + kD * kD;
  uint8_t** tiles = reinterpret_cast<uint8_t**>(R + kGroupVecs * kD);
  int* trow = reinterpret_cast<int*>(tiles + kGroupVecs);
  grid_dep_wait();   // S, keys, slots and cache may come from the previous kernel
  grid_dep_launch();
  load_st(sT, a.S);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, l = lane & 15;
  const long long groups = (a.num_vectors + kGroupVecs - 1) / kGroupVecs;
  for (long long grp = blockIdx.x; grp < groups; grp += gridDim.x) {
    // ---- phase 1: a half-warp per vector, 16 vectors per pass
    for (int pass = 0; pass < kGroupVecs / 16; ++pass) {
      const int gv = pass * 16 + (threadIdx.x >> 4);   // vector of the group
      const long long vec = grp * kGroupVecs + gv;
      bool live = vec < a.num_vectors;
      uint8_t* tile = nullptr;
      int r = 0;
      if (live) {
        const long long tok = a.num_vectors < (1ll << 31)
                                  ? static_cast<long long>(__umulhi(2u * static_cast<unsigned>(vec), a.kv_magic) >> a.kv_shift)
                                  : vec / a.n_kv;
        const int head = static_cast<int>(vec - tok * a.n_kv);
        const long long slot = ld_dep_s64(a.slots + tok);
        const long long blk = slot >> a.log2_bs;
        if (slot < 0) {
          live = false;
        } else if (blk >= a.num_blocks) {
          if (l == 0) flag(a.status, TQ_DEV_SLOT_OUT_OF_RANGE);
          live = false;
        } else {
          const int off = static_cast<int>(slot & (a.block_size - 1));
          tile = a.cache + ((blk * a.n_kv + head) * a.tiles_per_block + (off >> 4)) * static_cast<long long>(kTileBytes);
          r = off & 15;
        }
      }
      float k[8];
      if (live) {
        load8<T>(a.key, vec * kD + 8 * l, k);
      } else {
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
      float* rrow = R + gv * kD + 8 * l;
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
    __syncthreads();
    // ---- phase 2: warp w projects vectors 16 w .. 16 w + 15; lane l owns rows 4 l .. 4 l + 3
    float acc[16][4];
#pragma unroll
    for (int v = 0; v < 16; ++v) acc[v][0] = acc[v][1] = acc[v][2] = acc[v][3] = 0.f;
    const float* Rw = R + warp * 16 * kD;
#pragma unroll 1
    for (int j4 = 0; j4 < kD / 4; ++j4) {
      float4 s4[4];   // S^T rows 4 j4 .. 4 j4 + 3, columns 4 l .. 4 l + 3
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) s4[jj] = *reinterpret_cast<const float4*>(sT + (4 * j4 + jj) * kD + 4 * lane);
#pragma unroll
      for (int v = 0; v < 16; ++v) {
        const float4 r4 = *reinterpret_cast<const float4*>(Rw + v * kD + 4 * j4);   // broadcast
        const float rj[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          acc[v][0] = fmaf(s4[jj].x, rj[jj], acc[v][0]);
          acc[v][1] = fmaf(s4[jj].y, rj[jj], acc[v][1]);
          acc[v][2] = fmaf(s4[jj].z, rj[jj], acc[v][2]);
          acc[v][3] = fmaf(s4[jj].w, rj[jj], acc[v][3]);
        }
      }
    }
    // signs: bit i of vector v is (S r)_i >= 0; ballot q gives bit l = row 4 l + q.
    // Word w of the 128-bit stream holds rows 32 w .. 32 w + 31, i.e. lanes
    // 8 w .. 8 w + 7 of each ballot; lanes 2 v and 2 v + 1 write vector v's words.
#pragma unroll
    for (int v = 0; v < 16; ++v) {
      uint32_t m[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) m[q] = __ballot_sync(0xffffffffu, acc[v][q] >= 0.f);
      if ((lane >> 1) == v) {
        uint8_t* tile = tiles[warp * 16 + v];
        if (tile) {
          const int w0 = 2 * (lane & 1);
          uint32_t words[2];
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            const int w = w0 + x;
            words[x] = spread4((m[0] >> (8 * w)) & 0xFFu) | (spread4((m[1] >> (8 * w)) & 0xFFu) << 1) |
                       (spread4((m[2] >> (8 * w)) & 0xFFu) << 2) | (spread4((m[3] >> (8 * w)) & 0xFFu) << 3);
          }
          *reinterpret_cast<uint2*>(tile + kSOff + trow[warp * 16 + v] * kSRow + 8 * (lane & 1)) =
              make_uint2(words[0], words[1]);
        }
      }
    }
    __syncthreads();   // R and tiles are rewritten by the next group
  }
}

// ---------------------------------------------------------------- scores

struct ProdScoreArgs {
  const void* q;
  const float* S;
  const uint8_t* cache;
  const int* block_table;
  const int* seq_lens;
  float* scores;
  float* qprep;          // [batch][n_q][2][d]: q_r, then S q_r
  unsigned int* status;
  long long num_blocks;
  int batch, n_q, n_kv, group, bt_stride, max_seq_len, cap, block_size, log2_bs, tiles_per_block;
  float qscale;          // scale / sqrt(d)
  float cent[4];
};

// Sylvester-order Walsh-Hadamard transform of 128 values held as 4
// consecutive coordinates per lane (coordinate 4 lane + j), unnormalised.
__device__ __forceinline__ void fwht128_warp(float v[4], int lane) {
  float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
  v[0] = a0 + a2; v[2] = a0 - a2; v[1] = a1 + a3; v[3] = a1 - a3;
#pragma unroll
  for (int m = 1; m <= 16; m <<= 1) {
    const float sgn = (lane & m) ? -1.f : 1.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = fmaf(sgn, v[j], __shfl_xor_sync(0xffffffffu, v[j], m));
  }
}

// One warp per (sequence, query head): q_r = scale (H / sqrt(d)) q and S q_r.
template <typename TQ>
__global__ void __launch_bounds__(kThreads, 1) prod_query_kernel(const ProdScoreArgs a) {
  extern __shared__ __align__(16) float s_q[];
  float* sT = s_q;
  float* qr = s_q + kD * kD;   // one 128-float row per warp
  grid_dep_wait();
  grid_dep_launch();
  load_st(sT, a.S);
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long row = static_cast<long long>(blockIdx.x) * (kThreads / 32) + warp;   // b * n_q + h
  if (row < static_cast<long long>(a.batch) * a.n_q) {
    const uint2 raw = ld_dep_u32x2(static_cast<const TQ*>(a.q) + row * kD + 4 * lane);
    float x[4];
    const uint32_t w[2] = {raw.x, raw.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float2 f;
      if constexpr (std::is_same<TQ, __nv_bfloat16>::value) f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
      else f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
    fwht128_warp(x, lane);
#pragma unroll
    for (int j = 0; j < 4; ++j) x[j] *= a.qscale;
    float* mine = qr + warp * kD;
    *reinterpret_cast<float4*>(mine + 4 * lane) = make_float4(x[0], x[1], x[2], x[3]);
    __syncwarp();
    float u[4] = {0.f, 0.f, 0.f, 0.f};   // rows 4 lane .. 4 lane + 3
#pragma unroll 4
    for (int j = 0; j < kD; ++j) {
      const float4 s4 = *reinterpret_cast<const float4*>(sT + j * kD + 4 * lane);
      const float qj = mine[j];
      u[0] = fmaf(s4.x, qj, u[0]);
      u[1] = fmaf(s4.y, qj, u[1]);
      u[2] = fmaf(s4.z, qj, u[2]);
      u[3] = fmaf(s4.w, qj, u[3]);
    }
    float* out = a.qprep + row * 2 * kD;
    *reinterpret_cast<float4*>(out + 4 * lane) = make_float4(x[0], x[1], x[2], x[3]);
    *reinterpret_cast<float4*>(out + kD + 4 * lane) = make_float4(u[0], u[1], u[2], u[3]);
  }
}

// Grid (tile groups, n_kv, batch); each warp takes 16-position tiles of its
// (sequence, KV head), lanes l and l + 16 split position l's 128 coordinates.
constexpr int kTilesPerCta = 16;

__global__ void __launch_bounds__(kThreads) prod_scores_kernel(const ProdScoreArgs a) {
  extern __shared__ __align__(16) float s_p[];   // [G][d] pairs (q_r[j], S q_r[j]) as float2
  grid_dep_wait();   // the prep kernel wrote qprep
  grid_dep_launch();
  const int h = blockIdx.y, b = blockIdx.z, G = a.group;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float2* qu = reinterpret_cast<float2*>(s_p);
  for (int e = threadIdx.x; e < G * kD; e += blockDim.x) {
    const int gg = e >> 7, j = e & (kD - 1);
    const float* src = a.qprep + (static_cast<long long>(b) * a.n_q + h * G + gg) * 2 * kD;
    qu[e] = make_float2(ld_dep_f32(src + j), ld_dep_f32(src + kD + j));
  }
  __syncthreads();
  const int raw_len = ld_dep_s32(a.seq_lens + b);
  const int len = min(max(raw_len, 0), min(a.max_seq_len, a.cap));
  if (blockIdx.x == 0 && h == 0 && threadIdx.x == 0 && raw_len > min(a.max_seq_len, a.cap)) flag(a.status, TQ_DEV_SEQ_TOO_LONG);
  const int ntiles_out = (a.max_seq_len + 15) / 16;
  const int p = lane & 15, half = lane >> 4;
  for (int t = blockIdx.x * kTilesPerCta + warp; t < min(ntiles_out, (blockIdx.x + 1) * kTilesPerCta);
       t += kThreads / 32) {
    const int pos = 16 * t + p;
    bool live = pos < len;
    const uint8_t* tile = nullptr;
    if (16 * t < len) {
      const int blk = ld_dep_s32(a.block_table + static_cast<long long>(b) * a.bt_stride + ((16 * t) >> a.log2_bs));
      if (blk < 0 || blk >= a.num_blocks) {
        if (lane == 0) flag(a.status, TQ_DEV_BLOCK_OUT_OF_RANGE);
        live = false;
      } else {
        const int off = (16 * t) & ((1 << a.log2_bs) - 1);
        tile = a.cache + ((static_cast<long long>(blk) * a.n_kv + h) * a.tiles_per_block + (off >> 4)) *
                             static_cast<long long>(kTileBytes);
      }
    } else {
      live = false;
    }
    uint4 codes = make_uint4(0u, 0u, 0u, 0u);   // 64 coordinates x 2 bits
    uint2 sbits = make_uint2(0u, 0u);           // 64 sign bits
    float nrm = 0.f, rnrm = 0.f;
    if (live) {
      codes = ld_dep_u32x4(tile + kKOff + p * kKRow + 16 * half);
      sbits = ld_dep_u32x2(tile + kSOff + p * kSRow + 8 * half);
      nrm = __half2float(__ushort_as_half(ld_dep_u16(tile + kNormOff + 2 * p)));
      rnrm = __half2float(__ushort_as_half(ld_dep_u16(tile + kRnormOff + 2 * p)));
    }
    float mse[8], qjl[8];
#pragma unroll
    for (int gg = 0; gg < 8; ++gg) mse[gg] = qjl[gg] = 0.f;
    const int j0 = 64 * half;
#pragma unroll 4
    for (int jj = 0; jj < 64; ++jj) {
      const uint32_t cw = jj < 16 ? codes.x : (jj < 32 ? codes.y : (jj < 48 ? codes.z : codes.w));
      const uint32_t c = (cw >> (2 * (jj & 15))) & 3u;
      const float cv = c == 0 ? a.cent[0] : (c == 1 ? a.cent[1] : (c == 2 ? a.cent[2] : a.cent[3]));
      const uint32_t sw = jj < 32 ? sbits.x : sbits.y;
      const float sg = ((sw >> (jj & 31)) & 1u) ? 1.f : -1.f;
#pragma unroll
      for (int gg = 0; gg < 8; ++gg) {
        if (gg < G) {
          const float2 v = qu[gg * kD + j0 + jj];   // broadcast within each half
          mse[gg] = fmaf(v.x, cv, mse[gg]);
          qjl[gg] = fmaf(v.y, sg, qjl[gg]);
        }
      }
    }
#pragma unroll
    for (int gg = 0; gg < 8; ++gg) {
      if (gg < G) {
        mse[gg] += __shfl_xor_sync(0xffffffffu, mse[gg], 16);
        qjl[gg] += __shfl_xor_sync(0xffffffffu, qjl[gg], 16);
        if (half == 0 && pos < a.max_seq_len) {
          const float sc = live ? nrm * fmaf(rnrm * kQjlScale, qjl[gg], mse[gg]) : 0.f;
          a.scores[(static_cast<long long>(b) * a.n_q + h * G + gg) * a.max_seq_len + pos] = sc;
        }
      }
    }
  }
}

void fill_magic(int n, unsigned* magic, unsigned* shift) {
  unsigned sh = 0;
  while ((1u << sh) < static_cast<unsigned>(n)) ++sh;
  *shift = sh;
  *magic = static_cast<unsigned>(((1ull << (31 + sh)) + n - 1) / n);
}

tq_status prod_layout(const tq_config* cfg, tq_prod_layout* out) {
  if (!cfg || !out) return TQ_ERR_INVALID_ARG;
  if (cfg->preset != TQ_PRESET_PROD3) return TQ_ERR_INVALID_ARG;
  if (cfg->head_dim <= 0 || cfg->block_size <= 0 || cfg->num_kv_heads <= 0) return TQ_ERR_INVALID_ARG;
  if (cfg->flags & ~TQ_FLAG_INDICES_READY) return TQ_ERR_INVALID_ARG;
  if (cfg->head_dim != kD) return TQ_ERR_UNSUPPORTED;
  const int bs = cfg->block_size;
  if (bs != 16 && bs != 32 && bs != 64 && bs != 128) return TQ_ERR_UNSUPPORTED;
  out->mse_bits = kMseBits;
  out->slot_bytes = kTileBytes / 16;
  out->tile_bytes = kTileBytes;
  out->k_off = kKOff;
  out->k_row_bytes = kKRow;
  out->sign_off = kSOff;
  out->sign_row_bytes = kSRow;
  out->norm_off = kNormOff;
  out->rnorm_off = kRnormOff;
  out->block_bytes = static_cast<long long>(bs) * cfg->num_kv_heads * (kTileBytes / 16);
  return TQ_OK;
}

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

}  // namespace
}  // namespace tq

extern "C" {

tq_status tq_prod_layout_for(const tq_config* cfg, tq_prod_layout* out) { return tq::prod_layout(cfg, out); }

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

size_t tq_prod_scores_workspace_size(const tq_config* cfg, int batch) {
  tq_prod_layout L;
  if (batch < 0 || tq::prod_layout(cfg, &L) != TQ_OK || cfg->num_q_heads <= 0) return 0;
  return static_cast<size_t>(batch) * cfg->num_q_heads * 2 * tq::kD * sizeof(float);
}

tq_status tq_prod_scores(const tq_config* cfg, const tq_codebook* cb, const float* S, const void* q, int q_dtype,
                         const void* cache, long long num_blocks, const int* block_table, int bt_stride,
                         const int* seq_lens, int batch, int max_seq_len, float scale, float* scores,
                         void* workspace, size_t workspace_bytes, unsigned int* dev_status, tq_stream_t stream) {
  using namespace tq;
  tq_prod_layout L;
  const tq_status st = prod_layout(cfg, &L);
  if (st != TQ_OK) return st;
  if (batch < 0 || max_seq_len < 0 || num_blocks < 0 || bt_stride < 1) return TQ_ERR_INVALID_ARG;
  if (cfg->num_q_heads <= 0 || cfg->num_q_heads % cfg->num_kv_heads) return TQ_ERR_INVALID_ARG;
  const int G = cfg->num_q_heads / cfg->num_kv_heads;
  if (G > 8) return TQ_ERR_UNSUPPORTED;
  if (q_dtype != TQ_DTYPE_F16 && q_dtype != TQ_DTYPE_BF16) return TQ_ERR_INVALID_ARG;
  if (!cb || cb->bits != kMseBits || cb->head_dim != cfg->head_dim) return TQ_ERR_INVALID_ARG;
  if (workspace_bytes < tq_prod_scores_workspace_size(cfg, batch)) return TQ_ERR_WORKSPACE_TOO_SMALL;
  if (batch == 0 || max_seq_len == 0) return TQ_OK;
  if (!S || !q || !cache || !block_table || !seq_lens || !scores || !workspace) return TQ_ERR_INVALID_ARG;
  if (!aligned16(S) || !aligned16(q) || !aligned16(cache) || !aligned16(scores) || !aligned16(workspace) ||
      (reinterpret_cast<unsigned long long>(block_table) & 3ull) ||
      (reinterpret_cast<unsigned long long>(seq_lens) & 3ull))
    return TQ_ERR_MISALIGNED;
  if (dev_status && (reinterpret_cast<unsigned long long>(dev_status) & 3ull)) return TQ_ERR_MISALIGNED;
  if (cfg->num_kv_heads > 65535 || batch > 65535) return TQ_ERR_UNSUPPORTED;
  ProdScoreArgs a;
  a.q = q;
  a.S = S;
  a.cache = static_cast<const uint8_t*>(cache);
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.scores = scores;
  a.qprep = static_cast<float*>(workspace);
  a.status = dev_status;
  a.num_blocks = num_blocks;
  a.batch = batch;
  a.n_q = cfg->num_q_heads;
  a.n_kv = cfg->num_kv_heads;
  a.group = G;
  a.bt_stride = bt_stride;
  a.max_seq_len = max_seq_len;
  a.cap = static_cast<int>(static_cast<long long>(bt_stride) * cfg->block_size < max_seq_len
                               ? static_cast<long long>(bt_stride) * cfg->block_size : max_seq_len);
  a.block_size = cfg->block_size;
  a.log2_bs = __builtin_ctz(static_cast<unsigned>(cfg->block_size));
  a.tiles_per_block = cfg->block_size / kTileTokens;
  a.qscale = (scale > 0.f ? scale : 0.088388347648318440f) * 0.088388347648318440f;   // scale / sqrt(d)
  for (int i = 0; i < 4; ++i) a.cent[i] = cb->centroids[i];
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t qsmem = (static_cast<size_t>(kD) * kD + (kThreads / 32) * kD) * sizeof(float);
  const long long rows = static_cast<long long>(batch) * cfg->num_q_heads;
  const dim3 qgrid(static_cast<unsigned>((rows + kThreads / 32 - 1) / (kThreads / 32)));
  cudaError_t err;
  if (q_dtype == TQ_DTYPE_BF16) {
    err = cudaFuncSetAttribute(prod_query_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(qsmem));
    if (err == cudaSuccess) err = launch_pdl(prod_query_kernel<__nv_bfloat16>, qgrid, dim3(kThreads), qsmem, s, a);
  } else {
    err = cudaFuncSetAttribute(prod_query_kernel<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(qsmem));
    if (err == cudaSuccess) err = launch_pdl(prod_query_kernel<__half>, qgrid, dim3(kThreads), qsmem, s, a);
  }
  if (err != cudaSuccess) return TQ_ERR_CUDA;
  const int ntiles = (max_seq_len + 15) / 16;
  const dim3 grid(static_cast<unsigned>((ntiles + kTilesPerCta - 1) / kTilesPerCta),
                  static_cast<unsigned>(cfg->num_kv_heads), static_cast<unsigned>(batch));
  err = launch_pdl(prod_scores_kernel, grid, dim3(kThreads), static_cast<size_t>(G) * kD * sizeof(float2), s, a);
  return err == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // extern "C"
