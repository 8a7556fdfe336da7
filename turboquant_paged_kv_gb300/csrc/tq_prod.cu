// tq_prod: the unbiased inner-product estimates of TurboQuant_prod keys (a
// 2-bit Lloyd-Max code plus a 1-bit QJL sign of the residual per
// coordinate), read back from the key-only paged cache that tq_prod_store.cu
// writes.
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
//   scores  a prep kernel rotates each query head and forms S q_r once,
//           writing each lane's fp16 operand registers; the persistent scores
//           kernel streams 16-position tiles through a cp.async ring and takes
//           the three bit-matrix products on tensor cores (see below).

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

// ---------------------------------------------------------------- scores
//
// Tensor-core form. For a tile of 16 positions and the G (<= 8) query heads
// of one KV head the estimate is three products of a 16 x 128 bit matrix
// with a 128 x G matrix: with the antisymmetric codebook {-A, -B, B, A} the
// Lloyd-Max value of a 2-bit code is c = -A + (A - B) lo + (A + B) hi (lo, hi
// its two bits), and a sign bit s gives the sign 2 s - 1, so
//   <q_r, c[idx]> = -A sum(q_r) + (A - B) <q_r, lo> + (A + B) <q_r, hi>
//   <u, signs>    = 2 <u, s> - sum(u)                    (u = S q_r)
// Each bit goes into an mma.sync.m16n8k16 A operand unchanged: masking a word
// of the cache with 0x00010001 << p leaves, in each 16-bit half, the fp16
// subnormal bit * 2^(p - 24) (p <= 9; bits 10..15 of a half are shifted down
// by 6 first). The query side carries q_r * 2^(e - p) in fp16 (2^e a power of
// two per head that puts max |q_r| just under 2^15), so the only rounding of
// the products is that of q_r and u to fp16 (at most 2^-12 relative per
// coordinate), and sum(q_r), sum(u) are taken over the very same values.
//
// Fragment mapping (lane = 4 g + t): lane t of every group covers
// coordinates 32 t .. 32 t + 31, i.e. Lloyd-Max words 2 t and 2 t + 1 and
// sign word t of a row. In chunk c (k = 16 coordinates) its register pairs
// (k = 2 t, 2 t + 1) and (k = 2 t + 8, 2 t + 9) are the codes (i, i + 8) and
// (i + 1, i + 9) of word 2 t + c / 4 with i = 2 (c % 4) for the Lloyd-Max
// products, and the sign bits (j, j + 16) and (j + 1, j + 17) of word t with
// j = 2 c for the QJL product; the query operand of lane (g, t) holds head
// g's values at the same coordinates.
//
// Kernels: prod_query_kernel, one CTA per (sequence, KV head) with a warp per
// query head, rotates the queries, forms S q_r (S staged in shared memory,
// a warp transpose-reduce for the 128 dot products) and writes each lane's
// fp16 operand registers and epilogue constants to the workspace; the
// persistent prod_scores_kernel splits the flat (sequence, KV head, tile)
// range evenly over its CTAs, a warp taking every 8th tile, reading the block
// table for 32 tiles at once and prefetching the next tile's words.

constexpr int kFragWords = 32;                 // u32 operand registers per lane
constexpr int kConstFloats = 12;               // epilogue constants per lane (10 used)
constexpr int kWsPerKvHead = 32 * (kFragWords * 4 + kConstFloats * 4);   // 5632 bytes
constexpr int kQsRow = 33;                     // 32 coordinates + 1 pad per (head, t)
constexpr size_t kPrepSmem = static_cast<size_t>(kD) * kD * sizeof(float) + 2 * 8 * 4 * kQsRow * sizeof(float);

struct ProdScoreArgs {
  const void* q;
  const float* S;
  const uint8_t* cache;
  const int* block_table;
  const int* seq_lens;
  float* scores;
  uint32_t* frag;        // [batch * n_kv][32 lanes][32] fp16 pairs
  float* consts;         // [batch * n_kv][32 lanes][12]
  unsigned int* status;
  long long num_blocks;
  int batch, n_q, n_kv, group, bt_stride, max_seq_len, cap, block_size, log2_bs, tiles_per_block, ntiles;
  float qscale;          // scale / sqrt(d)
  float cent_a, cent_b;  // the codebook {-A, -B, B, A}
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

// One stage of a warp transpose-reduce: entries k and k + M of every lane
// are summed across lanes l and l ^ M, lane l keeping row k + M * [l & M].
template <int M>
__device__ __forceinline__ void treduce_stage(float (&p)[32], int lane) {
  const bool up = lane & M;
#pragma unroll
  for (int k = 0; k < M; ++k) {
    const float send = up ? p[k] : p[k + M];
    const float keep = up ? p[k + M] : p[k];
    p[k] = keep + __shfl_xor_sync(0xffffffffu, send, M);
  }
}

// Bit position, inside a 16-bit half, of Lloyd-Max pair i (its low bit) and
// of sign pair j once the word is shifted by 6 where needed.
__host__ __device__ constexpr int lo_pos(int i) { return i <= 4 ? 2 * i : 2 * i - 6; }
__host__ __device__ constexpr int sign_pos(int j) { return j <= 9 ? j : j - 6; }

// 2^e as a float for |e| < 127.
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((e + 127) << 23); }

// Exponent of the power-of-two scale that maps max |x| (m) to [2^14, 2^15):
// 15 - e with m < 2^e, clamped to [-100, 111] (m below 2^-96 is scaled as if
// 2^-96; m of 2^115 and more, far outside any query's range, overflows fp16).
__device__ __forceinline__ int scale_exp(float m) {
  const int eb = min(max((__float_as_int(m) >> 23) & 0xFF, 30), 241);   // m < 2^(eb - 126)
  return 141 - eb;
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  return static_cast<uint32_t>(__half_as_ushort(__float2half_rn(lo))) |
         (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(hi))) << 16);
}

__device__ __forceinline__ float h2_sum_scaled(uint32_t v, float w) {   // (lo + hi) * w
  return (__half2float(__ushort_as_half(static_cast<unsigned short>(v & 0xFFFFu))) +
          __half2float(__ushort_as_half(static_cast<unsigned short>(v >> 16)))) * w;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }

// Grid: one CTA per (sequence, KV head), a warp per query head of its group.
template <typename TQ>
__global__ void __launch_bounds__(kThreads) prod_query_kernel(const ProdScoreArgs a) {
  extern __shared__ __align__(16) float s_q[];
  float* sS = s_q;                       // S row-major
  float* qs = s_q + kD * kD;             // [head][t][kQsRow]: q_r of coordinates 32 t + w
  float* us = qs + 8 * 4 * kQsRow;       // same for S q_r
  grid_dep_wait();
  grid_dep_launch();
  const int bh = blockIdx.x, b = bh / a.n_kv, h = bh - b * a.n_kv, G = a.group;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e = threadIdx.x; e < kD * kD / 4; e += blockDim.x)   // all copies in flight at once
    cp_async16(sS + 4 * e, a.S + 4 * e);
  cp_async_commit();
  float x[4];
  {
    const long long row = static_cast<long long>(b) * a.n_q + h * G + warp;
    const uint2 raw = ld_dep_u32x2(static_cast<const TQ*>(a.q) + row * kD + 4 * lane);
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
    for (int j = 0; j < 4; ++j) {
      x[j] *= a.qscale;
      qs[(warp * 4 + (lane >> 3)) * kQsRow + 4 * (lane & 7) + j] = x[j];
    }
  }
  asm volatile("cp.async.wait_all;\n" ::: "memory");
  __syncthreads();   // S staged
#pragma unroll 1
  for (int blk = 0; blk < 4; ++blk) {
    float p[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      const float4 s4 = *reinterpret_cast<const float4*>(sS + (32 * blk + r) * kD + 4 * lane);
      p[r] = fmaf(s4.x, x[0], fmaf(s4.y, x[1], fmaf(s4.z, x[2], s4.w * x[3])));
    }
    treduce_stage<16>(p, lane);
    treduce_stage<8>(p, lane);
    treduce_stage<4>(p, lane);
    treduce_stage<2>(p, lane);
    treduce_stage<1>(p, lane);
    us[(warp * 4 + blk) * kQsRow + lane] = p[0];   // (S q_r)_{32 blk + lane}
  }
  __syncthreads();
  if (warp != 0) return;
  // ---- lane (g, t): operand registers of head g at coordinates 32 t .. 32 t + 31
  const int g = lane >> 2, t = lane & 3;
  float q[32], u[32];
#pragma unroll
  for (int w = 0; w < 32; ++w) {
    q[w] = g < G ? qs[(g * 4 + t) * kQsRow + w] : 0.f;
    u[w] = g < G ? us[(g * 4 + t) * kQsRow + w] : 0.f;
  }
  float mq = 0.f, mu = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    mq = fmaxf(mq, fabsf(q[i]));
    mu = fmaxf(mu, fabsf(u[i]));
  }
#pragma unroll
  for (int m = 1; m <= 2; m <<= 1) {
    mq = fmaxf(mq, __shfl_xor_sync(0xffffffffu, mq, m));
    mu = fmaxf(mu, __shfl_xor_sync(0xffffffffu, mu, m));
  }
  const int eq = scale_exp(mq), eu = scale_exp(mu);
  uint32_t fr[kFragWords];   // per chunk c: Lloyd-Max pairs x = 0, 1, then sign pairs x = 0, 1
  float sq = 0.f, su = 0.f;  // sums of the fp16 values, in units of 2^-e
#pragma unroll
  for (int c = 0; c < 8; ++c) {
#pragma unroll
    for (int x2 = 0; x2 < 2; ++x2) {
      const int i = 2 * (c & 3) + x2, w = 16 * (c >> 2) + i;   // Lloyd-Max pair: local coordinates w, w + 8
      fr[4 * c + x2] = pack_h2(q[w] * exp2i(eq - lo_pos(i)), q[w + 8] * exp2i(eq - lo_pos(i)));
      sq += h2_sum_scaled(fr[4 * c + x2], exp2i(lo_pos(i)));
      const int j = 2 * c + x2;                                  // sign pair: local coordinates j, j + 16
      fr[4 * c + 2 + x2] = pack_h2(u[j] * exp2i(eu - sign_pos(j)), u[j + 16] * exp2i(eu - sign_pos(j)));
      su += h2_sum_scaled(fr[4 * c + 2 + x2], exp2i(sign_pos(j)));
    }
  }
#pragma unroll
  for (int m = 1; m <= 2; m <<= 1) {
    sq += __shfl_xor_sync(0xffffffffu, sq, m);
    su += __shfl_xor_sync(0xffffffffu, su, m);
  }
  // epilogue constants of output columns (heads) 2 t and 2 t + 1, from group g = column
  float k[kConstFloats];
#pragma unroll
  for (int x2 = 0; x2 < 2; ++x2) {
    const int src = 4 * (2 * t + x2);
    const float sqx = __shfl_sync(0xffffffffu, sq, src), sux = __shfl_sync(0xffffffffu, su, src);
    const int eqx = __shfl_sync(0xffffffffu, eq, src), eux = __shfl_sync(0xffffffffu, eu, src);
    k[0 + x2] = -a.cent_a * sqx * exp2i(-eqx);                 // -A sum(q_r)
    k[2 + x2] = (a.cent_a - a.cent_b) * exp2i(24 - eqx);       // per unit of the lo product
    k[4 + x2] = (a.cent_a + a.cent_b) * exp2i(23 - eqx);       // per unit of the hi product
    k[6 + x2] = kQjlScale * exp2i(25 - eux);                   // 2 <u, s> scaled
    k[8 + x2] = -kQjlScale * sux * exp2i(-eux);                // -sum(u) scaled
  }
  k[10] = k[11] = 0.f;
  uint4* fo = reinterpret_cast<uint4*>(a.frag + (static_cast<long long>(bh) * 32 + lane) * kFragWords);
#pragma unroll
  for (int i = 0; i < kFragWords / 4; ++i) fo[i] = make_uint4(fr[4 * i], fr[4 * i + 1], fr[4 * i + 2], fr[4 * i + 3]);
  float4* ko = reinterpret_cast<float4*>(a.consts + (static_cast<long long>(bh) * 32 + lane) * kConstFloats);
#pragma unroll
  for (int i = 0; i < kConstFloats / 4; ++i) ko[i] = make_float4(k[4 * i], k[4 * i + 1], k[4 * i + 2], k[4 * i + 3]);
}

constexpr int kScoreWarps = kThreads / 32;
constexpr int kRing = 4;                                            // tiles in flight per warp
constexpr size_t kScoreSmem = static_cast<size_t>(kScoreWarps) * kRing * kTileBytes;

// Where tile `idx` of the flat (sequence, KV head, tile) range lives. The
// length and block-table entry are loaded by resolve_tile and first used by
// finish_tile many tiles later, so their latency overlaps the work between.
struct TileInfo {
  int bh, T, len;   // len: raw until finish_tile, then clamped to [0, cap]
  int blk;          // raw entry (-2: none read); after finish_tile the tile's index in the cache, -1 if none
};

__device__ __forceinline__ TileInfo resolve_tile(const ProdScoreArgs& a, long long idx, long long hi, int cap) {
  TileInfo r{0, 0, 0, -2};
  if (idx < hi) {
    r.bh = static_cast<int>(idx / a.ntiles);
    r.T = static_cast<int>(idx - static_cast<long long>(r.bh) * a.ntiles);
    const int b = r.bh / a.n_kv;
    r.len = ld_dep_s32(a.seq_lens + b);
    if (16 * r.T < cap)
      r.blk = ld_dep_s32(a.block_table + static_cast<long long>(b) * a.bt_stride + ((16 * r.T) >> a.log2_bs));
  }
  return r;
}

__device__ __forceinline__ void finish_tile(const ProdScoreArgs& a, TileInfo& r, int cap) {
  const int raw = r.len;
  r.len = min(max(raw, 0), cap);
  const int h = r.bh - (r.bh / a.n_kv) * a.n_kv;
  if (raw > cap && h == 0 && r.T == 0) flag(a.status, TQ_DEV_SEQ_TOO_LONG);
  int tile = -1;
  if (16 * r.T < r.len) {
    if (r.blk < 0 || r.blk >= a.num_blocks) {
      flag(a.status, TQ_DEV_BLOCK_OUT_OF_RANGE);
    } else {
      const int off = (16 * r.T) & (a.block_size - 1);
      tile = (r.blk * a.n_kv + h) * a.tiles_per_block + (off >> 4);
    }
  }
  r.blk = tile;
}

__device__ __forceinline__ void cp_async_wait_ring() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(kRing - 1) : "memory");
}

__device__ __forceinline__ void copy_tile(uint8_t* slot, const uint8_t* cache, int tile, int lane) {
  if (tile >= 0) {
    const uint8_t* p = cache + static_cast<long long>(tile) * kTileBytes;
    cp_async16(slot + 16 * lane, p + 16 * lane);
    if (lane < kTileBytes / 16 - 32) cp_async16(slot + 16 * (lane + 32), p + 16 * (lane + 32));
  }
  cp_async_commit();
}

__device__ __forceinline__ void mma_f16(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Persistent: CTA c takes the flat tile range [total c / grid, total (c + 1) / grid),
// warp w every 8th tile from the w-th. Each warp streams its tiles through a
// private ring of kRing shared-memory slots with cp.async (16 bytes a lane,
// one commit group per tile), kRing - 1 tiles ahead of the one it computes;
// lane i resolves the i-th tile of each batch of 32 one batch ahead.
__global__ void __launch_bounds__(kThreads, 2) prod_scores_kernel(const ProdScoreArgs a) {
  extern __shared__ __align__(16) uint8_t s_ring[];
  grid_dep_wait();   // the prep kernel wrote the operands
  grid_dep_launch();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, t = lane & 3;
  const int G = a.group, cap = min(a.max_seq_len, a.cap), L = a.max_seq_len;
  const long long total = static_cast<long long>(a.batch) * a.n_kv * a.ntiles;
  const long long lo = total * blockIdx.x / gridDim.x, hi = total * (blockIdx.x + 1) / gridDim.x;
  const long long first = lo + warp;
  if (first >= hi) return;
  const int cnt = static_cast<int>((hi - first + kScoreWarps - 1) / kScoreWarps);   // tiles of this warp
  uint8_t* ring = s_ring + static_cast<size_t>(warp) * kRing * kTileBytes;
  // output slots of this lane: heads 2 t, 2 t + 1 at rows g, g + 8 of a tile
  const bool h0 = 2 * t < G, h1 = 2 * t + 1 < G;
  const long long o0 = static_cast<long long>(2 * t) * L + g;

  TileInfo cb = resolve_tile(a, first + static_cast<long long>(kScoreWarps) * lane, hi, cap);
  TileInfo nb = resolve_tile(a, first + static_cast<long long>(kScoreWarps) * (32 + lane), hi, cap);
  finish_tile(a, cb, cap);
  bool nb_done = false;

  uint32_t fr[kFragWords];   // per chunk c: Lloyd-Max pairs x = 0, 1, then sign pairs x = 0, 1
  float k[kConstFloats];
  int frag_bh = -1;
  int batch = 0;   // index of the batch cb describes
#pragma unroll
  for (int jj = 0; jj < kRing - 1; ++jj)   // prologue: tiles 0 .. kRing - 2 (all in batch 0)
    copy_tile(ring + jj * kTileBytes, a.cache, jj < cnt ? __shfl_sync(0xffffffffu, cb.blk, jj) : -1, lane);
  for (int j = 0; j < cnt; ++j) {
    if ((j >> 5) != batch) {   // entering the next batch of 32 tiles
      if (!nb_done) finish_tile(a, nb, cap);
      cb = nb;
      batch = j >> 5;
      nb = resolve_tile(a, first + static_cast<long long>(kScoreWarps) * (32 * (batch + 1) + lane), hi, cap);
      nb_done = false;
    }
    {   // copies of tile j + kRing - 1
      const int jj = j + kRing - 1;
      int tile = -1;
      if (jj < cnt) {
        if ((jj >> 5) == batch) {
          tile = __shfl_sync(0xffffffffu, cb.blk, jj & 31);
        } else {
          if (!nb_done) {
            finish_tile(a, nb, cap);
            nb_done = true;
          }
          tile = __shfl_sync(0xffffffffu, nb.blk, jj & 31);
        }
      }
      copy_tile(ring + (jj % kRing) * kTileBytes, a.cache, tile, lane);
    }
    // tile j
    const int src = j & 31;
    const int bh = __shfl_sync(0xffffffffu, cb.bh, src), T = __shfl_sync(0xffffffffu, cb.T, src);
    const int len = __shfl_sync(0xffffffffu, cb.len, src);
    const bool live = __shfl_sync(0xffffffffu, cb.blk, src) >= 0;
    if (bh != frag_bh) {
      const uint4* fi = reinterpret_cast<const uint4*>(a.frag + (static_cast<long long>(bh) * 32 + lane) * kFragWords);
#pragma unroll
      for (int i = 0; i < kFragWords / 4; ++i) {
        const uint4 v = ld_dep_u32x4(fi + i);
        fr[4 * i] = v.x; fr[4 * i + 1] = v.y; fr[4 * i + 2] = v.z; fr[4 * i + 3] = v.w;
      }
      const float4* ki = reinterpret_cast<const float4*>(a.consts + (static_cast<long long>(bh) * 32 + lane) * kConstFloats);
#pragma unroll
      for (int i = 0; i < kConstFloats / 4; ++i) {
        const float4 v = ld_dep_f32x4(ki + i);
        k[4 * i] = v.x; k[4 * i + 1] = v.y; k[4 * i + 2] = v.z; k[4 * i + 3] = v.w;
      }
      frag_bh = bh;
    }
    cp_async_wait_ring();   // this lane's copies of tile j have landed
    __syncwarp();           // .. and every other lane's
    const uint8_t* tile = ring + (j % kRing) * kTileBytes;
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
    if (live) {
      const uint2 k0 = *reinterpret_cast<const uint2*>(tile + kKOff + g * kKRow + 8 * t);
      const uint2 k1 = *reinterpret_cast<const uint2*>(tile + kKOff + (g + 8) * kKRow + 8 * t);
      const uint32_t s0w = *reinterpret_cast<const uint32_t*>(tile + kSOff + g * kSRow + 4 * t);
      const uint32_t s1w = *reinterpret_cast<const uint32_t*>(tile + kSOff + (g + 8) * kSRow + 4 * t);
      const float n0 = __half2float(*reinterpret_cast<const __half*>(tile + kNormOff + 2 * g));
      const float n1 = __half2float(*reinterpret_cast<const __half*>(tile + kNormOff + 2 * (g + 8)));
      const float r0 = __half2float(*reinterpret_cast<const __half*>(tile + kRnormOff + 2 * g));
      const float r1 = __half2float(*reinterpret_cast<const __half*>(tile + kRnormOff + 2 * (g + 8)));
      const uint32_t kw[2][2] = {{k0.x, k0.y}, {k1.x, k1.y}};
      const uint32_t kz[2][2] = {{k0.x >> 6, k0.y >> 6}, {k1.x >> 6, k1.y >> 6}};
      const uint32_t sw[2] = {s0w, s1w}, sz[2] = {s0w >> 6, s1w >> 6};
      // two accumulators per product (even / odd chunks) halve the dependent mma chains
      float dl[2][4] = {}, dh[2][4] = {}, ds[2][4] = {};
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int W = c >> 2, i0 = 2 * (c & 3), i1 = i0 + 1, e = c & 1;
        const uint32_t m0 = 0x00010001u << lo_pos(i0), m1 = 0x00010001u << lo_pos(i1);
        const uint32_t w0g = i0 <= 4 ? kw[0][W] : kz[0][W], w0h = i0 <= 4 ? kw[1][W] : kz[1][W];
        const uint32_t w1g = i1 <= 4 ? kw[0][W] : kz[0][W], w1h = i1 <= 4 ? kw[1][W] : kz[1][W];
        mma_f16(dl[e], w0g & m0, w0h & m0, w1g & m1, w1h & m1, fr[4 * c], fr[4 * c + 1]);
        mma_f16(dh[e], w0g & (m0 << 1), w0h & (m0 << 1), w1g & (m1 << 1), w1h & (m1 << 1), fr[4 * c], fr[4 * c + 1]);
        const int j0 = 2 * c, j1 = j0 + 1;
        const uint32_t q0 = 0x00010001u << sign_pos(j0), q1 = 0x00010001u << sign_pos(j1);
        const uint32_t* s0 = j0 <= 9 ? sw : sz;
        const uint32_t* s1 = j1 <= 9 ? sw : sz;
        mma_f16(ds[e], s0[0] & q0, s0[1] & q0, s1[0] & q1, s1[1] & q1, fr[4 * c + 2], fr[4 * c + 3]);
      }
      // d[0], d[1]: row g, heads 2 t, 2 t + 1; d[2], d[3]: row g + 8
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int x2 = e & 1;
        const float nn = e < 2 ? n0 : n1, rr = e < 2 ? r0 : r1;
        const float mse = fmaf(k[4 + x2], dh[0][e] + dh[1][e], fmaf(k[2 + x2], dl[0][e] + dl[1][e], k[0 + x2]));
        sc[e] = nn * fmaf(rr, fmaf(k[6 + x2], ds[0][e] + ds[1][e], k[8 + x2]), mse);
      }
    }
    __syncwarp();           // every lane has read slot j % kRing before it is refilled
    float* out = a.scores + static_cast<long long>(bh) * G * L + 16 * T + o0;
    const int p0 = 16 * T + g, p1 = p0 + 8;
    if (p0 < L) {
      if (h0) out[0] = p0 < len ? sc[0] : 0.f;
      if (h1) out[L] = p0 < len ? sc[1] : 0.f;
    }
    if (p1 < L) {
      if (h0) out[8] = p1 < len ? sc[2] : 0.f;
      if (h1) out[L + 8] = p1 < len ? sc[3] : 0.f;
    }
  }
  asm volatile("cp.async.wait_all;\n" ::: "memory");   // no copy outlives the CTA
}

}  // namespace
}  // namespace tq

extern "C" {

tq_status tq_prod_layout_for(const tq_config* cfg, tq_prod_layout* out) { return tq::prod_layout(cfg, out); }

size_t tq_prod_scores_workspace_size(const tq_config* cfg, int batch) {
  tq_prod_layout L;
  if (batch < 0 || tq::prod_layout(cfg, &L) != TQ_OK || cfg->num_q_heads <= 0) return 0;
  return static_cast<size_t>(batch) * cfg->num_kv_heads * tq::kWsPerKvHead;
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
  // the tensor-core form needs the antisymmetric codebook {-A, -B, B, A}
  if (cb->centroids[0] != -cb->centroids[3] || cb->centroids[1] != -cb->centroids[2]) return TQ_ERR_INVALID_ARG;
  if (workspace_bytes < tq_prod_scores_workspace_size(cfg, batch)) return TQ_ERR_WORKSPACE_TOO_SMALL;
  if (batch == 0 || max_seq_len == 0) return TQ_OK;
  if (!S || !q || !cache || !block_table || !seq_lens || !scores || !workspace) return TQ_ERR_INVALID_ARG;
  if (!aligned16(S) || !aligned16(q) || !aligned16(cache) || !aligned16(scores) || !aligned16(workspace) ||
      (reinterpret_cast<unsigned long long>(block_table) & 3ull) ||
      (reinterpret_cast<unsigned long long>(seq_lens) & 3ull))
    return TQ_ERR_MISALIGNED;
  if (dev_status && (reinterpret_cast<unsigned long long>(dev_status) & 3ull)) return TQ_ERR_MISALIGNED;
  const long long bh = static_cast<long long>(batch) * cfg->num_kv_heads;
  if (bh * ((max_seq_len + 15) / 16) > (1ll << 40)) return TQ_ERR_UNSUPPORTED;   // flat tile index range
  if (num_blocks * cfg->num_kv_heads * (cfg->block_size / kTileTokens) >= (1ll << 31))
    return TQ_ERR_UNSUPPORTED;   // tiles are indexed in 32 bits (1.7 TiB of cache)
  ProdScoreArgs a;
  a.q = q;
  a.S = S;
  a.cache = static_cast<const uint8_t*>(cache);
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.scores = scores;
  a.frag = static_cast<uint32_t*>(workspace);
  a.consts = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + bh * 32 * kFragWords * 4);
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
  a.ntiles = (max_seq_len + 15) / 16;
  a.qscale = (scale > 0.f ? scale : 0.088388347648318440f) * 0.088388347648318440f;   // scale / sqrt(d)
  a.cent_a = cb->centroids[3];
  a.cent_b = cb->centroids[2];
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t err;
  if (q_dtype == TQ_DTYPE_BF16) {
    err = cudaFuncSetAttribute(prod_query_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kPrepSmem));
    if (err == cudaSuccess)
      err = launch_pdl(prod_query_kernel<__nv_bfloat16>, dim3(static_cast<unsigned>(bh)), dim3(32 * G), kPrepSmem, s, a);
  } else {
    err = cudaFuncSetAttribute(prod_query_kernel<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kPrepSmem));
    if (err == cudaSuccess)
      err = launch_pdl(prod_query_kernel<__half>, dim3(static_cast<unsigned>(bh)), dim3(32 * G), kPrepSmem, s, a);
  }
  if (err != cudaSuccess) return TQ_ERR_CUDA;
  if (cudaFuncSetAttribute(prod_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kScoreSmem)) != cudaSuccess)
    return TQ_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, prod_scores_kernel, kThreads, kScoreSmem) != cudaSuccess ||
      per_sm <= 0)
    return TQ_ERR_CUDA;
  const int sms = sm_count();
  if (sms <= 0) return TQ_ERR_CUDA;
  const long long total = bh * a.ntiles;
  const long long want = (total + kScoreWarps - 1) / kScoreWarps;
  const long long grid = want < static_cast<long long>(per_sm) * sms ? want : static_cast<long long>(per_sm) * sms;
  err = launch_pdl(prod_scores_kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreads), kScoreSmem, s, a);
  return err == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // extern "C"
