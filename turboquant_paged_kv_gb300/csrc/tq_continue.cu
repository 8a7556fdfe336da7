// tq_continue: attention of a prefill chunk's queries against their sequence's
// packed paged cache (the cached history plus the chunk itself, causal), with
// one CTA serving many queries per KV tile.
//
// Method: "vLLM 源码完全拆解(十九):TurboQuant KV Cache 量化" (pinghaoyang.com.cn),
// section "续写 prefill:小 chunk 走 decode,大 chunk 走反量化": a continuation chunk
// of at most 128 new tokens, whose keys and values are already in the cache,
// is served by the decode kernel: query i of the chunk is a decode request of
// length cached + i + 1 over the sequence's block-table row, which makes the
// attention causal. The per-position arithmetic is the decode's (section
// "读取内核": stored_norm * (q_rot . c[idx]) * scale, v = scale * code + zero,
// online softmax per split, LSE merge).
//
// GB300 design. Served one request per query (the pages' way, and what
// tq_decode does with per-query lengths), a chunk of q_len queries reads and
// decodes its whole history q_len times. Here each CTA holds 8 warps, each
// warp 8 (query, head) columns of the mma B operand (G = n_q / n_kv heads of
// 8 / G consecutive queries), so one CTA serves 64 / G queries of one KV head;
// all 8 warps consume every KV tile of the CTA's partition once it is in
// shared memory. A 128-query chunk with G = 4 is then read 8 times instead of
// 128. Per query the columns carry their own causal limit (the query's
// position), so one pass over a tile masks each column where it must.
//   Grid: (n_kv x query groups, partitions, sequences). The tiles of a
//   partition stream through a 4-slot shared-memory ring by cp.async (16 bytes
//   a thread, one commit group per tile, one CTA barrier per tile); the
//   partition's block ids are read into shared memory first. The math per tile
//   and warp is the decode kernel's G > 4 path (tq_decode.cu): K . Q^T on
//   tensor cores from the centroid LUT (hi and lo fp16 parts of the query in
//   two mma), lazy-rescaled online softmax in log2 units, O^T += V^T . P^T
//   from masked value-code operands and movmatrix-transposed probabilities.
//   The LUT here is addressed relative to its base (one add per lookup), so it
//   needs no 64 KB alignment and two CTAs fit on an SM.
//   Each (query, query head, partition) writes one record (normalised
//   accumulator, LSE); a reduce kernel, a warp per (query, query head), merges
//   the partitions. Nothing waits on a spin: the only waits are cp.async group
//   waits and CTA barriers.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>
#include <type_traits>

#include "tq_attn.cuh"
#include "tq_internal.h"
#include "tq_launch.cuh"

namespace tq {
namespace {

constexpr int kD = 128;
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRing = 4;                  // tiles in flight per CTA
constexpr int kMaxPartTiles = 256;        // partition_tokens up to 4096
constexpr int kQRowBytes = kD * 2;        // one fp16 query row
constexpr float kTau = 8.0f;              // lazy rescale threshold, log2 units

struct ContArgs {
  const uint8_t* cache;
  long long num_blocks;
  const void* q;             // [total_q][n_q][d]
  const int* query_start;    // [batch + 1]
  const int* block_table;
  const int* seq_lens;       // total length of each sequence, chunk included
  unsigned int* status;
  float* rec_o;              // [total_q][n_q][n_part][d]
  float* rec_lse;            // [total_q][n_q][n_part], log2 units
  int batch, total_q, n_q, n_kv, group, qpw, qpc, n_part, part_tiles, max_q_len;
  int block_size, log2_bs, tiles_per_block, bt_stride, cap;
  int tile_bytes, k_off, v_off, knorm_off, vscale_off, vzero_off;
  float qscale;              // softmax scale * log2(e) / gamma
  float cent[16];            // gamma * centroids
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_ring() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(kRing - 2) : "memory");
}

template <int KMODE>
__host__ __device__ constexpr uint32_t cont_smem_fixed() {
  return lut_bytes<KMODE>() + kWarps * 8 * kQRowBytes + kMaxPartTiles * 4;
}

// Grid (n_kv * query groups, partitions, batch); see the file comment.
template <int KMODE, int VBITS, typename TQ>
__global__ void __launch_bounds__(kThreads, 2) cont_kernel(const ContArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  constexpr uint32_t kLut = lut_bytes<KMODE>();
  const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  const uint32_t lut = sbase;                                  // LUT, then the query scratch rows,
  const uint32_t qscr = sbase + kLut;                          // the block ids and the ring
  int* bids = reinterpret_cast<int*>(smem + kLut + kWarps * 8 * kQRowBytes);
  const uint32_t ring = sbase + kLut + kWarps * 8 * kQRowBytes + kMaxPartTiles * 4;
  grid_dep_wait();   // q, the cache and the indices may come from the previous kernel
  grid_dep_launch();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, c = lane & 3;
  const int G = a.group;
  const int h = blockIdx.x % a.n_kv, qg = blockIdx.x / a.n_kv, p = blockIdx.y, b = blockIdx.z;
  const int q0 = ld_dep_s32(a.query_start + b);
  const int ql_raw = ld_dep_s32(a.query_start + b + 1) - q0;
  // rows past max_q_len, or outside [0, total_q), are not served (flagged)
  const int ql = q0 < 0 ? 0 : min(min(max(ql_raw, 0), a.max_q_len), max(a.total_q - q0, 0));
  const int i0 = qg * a.qpc;                 // first query of this CTA
  if (qg == 0 && q0 >= 0 && ql_raw > ql) {   // rows not served: empty records, so they come out 0
    const int r_end = q0 + min(ql_raw, a.total_q - q0);
    for (int e = tid; e < (r_end - q0 - ql) * G; e += kThreads) {
      const long long row = q0 + ql + e / G;
      a.rec_lse[(row * a.n_q + h * G + e % G) * a.n_part + p] = -INFINITY;
    }
  }
  if (i0 >= ql) {
    if (ql_raw != ql && qg == 0 && h == 0 && p == 0 && tid == 0) flag(a.status, TQ_DEV_SEQ_TOO_LONG);
    return;
  }
  const int raw_len = ld_dep_s32(a.seq_lens + b);
  const int seq = min(max(raw_len, 0), a.cap);
  if ((raw_len > a.cap || ql_raw != ql) && qg == 0 && h == 0 && p == 0 && tid == 0)
    flag(a.status, TQ_DEV_SEQ_TOO_LONG);
  const int base = seq - max(ql_raw, 0);     // position of query 0 of the chunk (of its true length)
  const int t_lo = p * a.part_tiles;
  const int end = min(seq, base + min(i0 + a.qpc, ql));   // positions the CTA's queries see: [0, end)
  const int t_hi = min((end + 15) >> 4, t_lo + a.part_tiles);

  // this lane's two columns: (query qi, head hd); invalid columns see nothing
  const int qw0 = i0 + warp * a.qpw;
  const int qi0 = qw0 + (2 * c) / G, qi1 = qw0 + (2 * c + 1) / G;
  const int hd0 = (2 * c) % G, hd1 = (2 * c + 1) % G;
  const bool cv0 = qi0 < ql, cv1 = qi1 < ql;
  const int lim0 = cv0 ? base + qi0 : -1, lim1 = cv1 ? base + qi1 : -1;
  const int wlast = qw0 < ql ? base + min(qw0 + a.qpw, ql) - 1 : -1;   // last position this warp sees
  const long long rec0 = (static_cast<long long>(q0 + qi0) * a.n_q + h * G + hd0) * a.n_part + p;
  const long long rec1 = (static_cast<long long>(q0 + qi1) * a.n_q + h * G + hd1) * a.n_part + p;

  if (t_lo >= t_hi) {   // no position of this partition is seen: empty records
    if (g == 0) {
      if (cv0) a.rec_lse[rec0] = -INFINITY;
      if (cv1) a.rec_lse[rec1] = -INFINITY;
    }
    return;
  }
  const int ntl = t_hi - t_lo;
  for (int j = tid; j < ntl; j += kThreads) {
    const int t = t_lo + j;
    const int blk = ld_dep_s32(a.block_table + static_cast<long long>(b) * a.bt_stride + ((16 * t) >> a.log2_bs));
    int tile = -1;
    if (blk < 0 || blk >= a.num_blocks) {
      flag(a.status, TQ_DEV_BLOCK_OUT_OF_RANGE);
    } else {
      tile = (blk * a.n_kv + h) * a.tiles_per_block + (((16 * t) & (a.block_size - 1)) >> 4);
    }
    bids[j] = tile;
  }
  if constexpr (KMODE != kFp8) build_lut<KMODE>(lut, a.cent, tid, kThreads);
  __syncthreads();   // block ids and LUT

  const int chunks = a.tile_bytes >> 4;
  auto copy_tile = [&](int j) {
    if (j < ntl) {
      const int tile = bids[j];
      if (tile >= 0 && tid < chunks)
        cp_async16(ring + static_cast<uint32_t>((j % kRing) * a.tile_bytes) + 16u * tid,
                   a.cache + static_cast<long long>(tile) * a.tile_bytes + 16 * tid);
    }
    cp_async_commit();
  };
#pragma unroll
  for (int j = 0; j < kRing - 1; ++j) copy_tile(j);

  // ---- query operands: column k of this warp is (query qw0 + k / G, head k % G);
  // rotated, scaled, split into fp16 hi and lo parts, and moved into the B
  // layout through this warp's scratch rows (hi parts, then lo parts)
  uint32_t qb[32];   // per k-step: hi parts in qb[0..15], lo parts in qb[16..31]
  {
    const uint32_t rows = qscr + static_cast<uint32_t>(warp) * 8 * kQRowBytes;
    uint32_t lo[8][2];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int qi = qw0 + k / G, hd = k % G;
      float x[4] = {0.f, 0.f, 0.f, 0.f};
      if (qi < ql)
        u2_to_f4<TQ>(ld_dep_u32x2(static_cast<const TQ*>(a.q) +
                                  (static_cast<long long>(q0 + qi) * a.n_q + h * G + hd) * kD + 4 * lane), x);
      float sc = a.qscale;
      if constexpr (KMODE != kFp8) {
        fwht128(x, lane);
        sc *= 0.088388347648318440f;   // 1 / sqrt(128)
      }
      uint32_t h01, h23;
      split_half2(x[0] * sc, x[1] * sc, h01, lo[k][0]);
      split_half2(x[2] * sc, x[3] * sc, h23, lo[k][1]);
      sts64(rows + k * kQRowBytes + 8 * lane, make_uint2(h01, h23));
    }
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      if (part == 1) {
#pragma unroll
        for (int k = 0; k < 8; ++k) sts64(rows + k * kQRowBytes + 8 * lane, make_uint2(lo[k][0], lo[k][1]));
      }
      __syncwarp();
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {   // column g, coordinates 32 c .. 32 c + 31
        const uint4 r = lds128(rows + g * kQRowBytes + 64 * c + 16 * kk);
        qb[16 * part + 4 * kk] = r.x;
        qb[16 * part + 4 * kk + 1] = r.y;
        qb[16 * part + 4 * kk + 2] = r.z;
        qb[16 * part + 4 * kk + 3] = r.w;
      }
      __syncwarp();
    }
  }

  float o[8][4];   // O^T accumulators: rows = coordinates, columns 2 c, 2 c + 1
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  float m0 = -1e30f, m1 = -1e30f, l0 = 0.f, l1 = 0.f, z0 = 0.f, z1 = 0.f;

  for (int j = 0; j < ntl; ++j) {
    cp_async_wait_ring();   // this thread's copies of tile j have landed
    __syncthreads();        // everyone's, and every warp is done with tile j - 1
    copy_tile(j + kRing - 1);
    const int tok0 = 16 * (t_lo + j);
    if (tok0 > wlast) continue;   // no column of this warp sees the tile
    const uint32_t st = ring + static_cast<uint32_t>((j % kRing) * a.tile_bytes);
    const bool tvalid = bids[j] >= 0;

    // ---- S = K . Q^T (rows: tokens g, g + 8; columns 2 c, 2 c + 1)
    float v[4];
    if constexpr (KMODE == kFp8) {
      float va[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t kt = st + a.k_off;
      const uint4 kg0 = lds128(kt + g * 128 + 32 * c), kg1 = lds128(kt + g * 128 + 32 * c + 16);
      const uint4 kh0 = lds128(kt + (g + 8) * 128 + 32 * c), kh1 = lds128(kt + (g + 8) * 128 + 32 * c + 16);
#pragma unroll
      for (int s = 0; s < 8; ++s) {   // coordinates 32 c + 4 s .. + 3
        const uint32_t wg = word_of(s < 4 ? kg0 : kg1, s & 3), wh = word_of(s < 4 ? kh0 : kh1, s & 3);
        const __half2_raw g01 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(wg & 0xFFFFu), __NV_E4M3);
        const __half2_raw g23 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(wg >> 16), __NV_E4M3);
        const __half2_raw h01 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(wh & 0xFFFFu), __NV_E4M3);
        const __half2_raw h23 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(wh >> 16), __NV_E4M3);
        const uint32_t a0 = static_cast<uint32_t>(g01.x) | (static_cast<uint32_t>(g01.y) << 16);
        const uint32_t a1 = static_cast<uint32_t>(h01.x) | (static_cast<uint32_t>(h01.y) << 16);
        const uint32_t a2 = static_cast<uint32_t>(g23.x) | (static_cast<uint32_t>(g23.y) << 16);
        const uint32_t a3 = static_cast<uint32_t>(h23.x) | (static_cast<uint32_t>(h23.y) << 16);
        mma16816(va, a0, a1, a2, a3, qb[2 * s], qb[2 * s + 1]);
        mma16816(va, a0, a1, a2, a3, qb[16 + 2 * s], qb[16 + 2 * s + 1]);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) v[k] = va[k];
    } else {
      const uint32_t kt = st + a.k_off;
      uint4 kg, kh;   // this lane's key slices of tokens g and g + 8
      if constexpr (KMODE == kMse4) {
        kg = lds128(kt + g * 64 + 16 * c);
        kh = lds128(kt + (g + 8) * 64 + 16 * c);
      } else {
        const uint32_t ra = kt + g * 48 + 12 * c, rb = kt + (g + 8) * 48 + 12 * c;
        kg = make_uint4(lds32(ra), lds32(ra + 4), lds32(ra + 8), 0u);
        kh = make_uint4(lds32(rb), lds32(rb + 4), lds32(rb + 8), 0u);
      }
      float va[4] = {0.f, 0.f, 0.f, 0.f}, vb[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t lane4 = 4u * lane;
#pragma unroll
      for (int s2 = 0; s2 < 8; ++s2) {
        const uint32_t g0 = lds32(lut + lut_addr<KMODE>(kg, 2 * s2, lane4));
        const uint32_t g1 = lds32(lut + lut_addr<KMODE>(kg, 2 * s2 + 1, lane4));
        const uint32_t h0 = lds32(lut + lut_addr<KMODE>(kh, 2 * s2, lane4));
        const uint32_t h1 = lds32(lut + lut_addr<KMODE>(kh, 2 * s2 + 1, lane4));
        mma16816(va, g0, h0, g1, h1, qb[2 * s2], qb[2 * s2 + 1]);
        mma16816(vb, g0, h0, g1, h1, qb[16 + 2 * s2], qb[16 + 2 * s2 + 1]);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) v[k] = va[k] + vb[k];
    }

    // ---- value words of the two token pairs this lane's operands need
    uint4 vwa, vwb;
    if constexpr (VBITS == 4) {   // 16-byte group g of each pair, swizzled by 2 c
      const uint32_t vt = st + a.v_off + 16 * (g ^ (2 * c));
      vwa = lds128(vt + 128 * c);
      vwb = lds128(vt + 128 * (c + 4));
    } else {                      // 12 bytes at 12 g of each 96-byte pair
      const uint32_t vt = st + a.v_off + 12 * g;
      vwa = make_uint4(lds32(vt + 96 * c), lds32(vt + 96 * c + 4), lds32(vt + 96 * c + 8), 0u);
      vwb = make_uint4(lds32(vt + 96 * (c + 4)), lds32(vt + 96 * (c + 4) + 4), lds32(vt + 96 * (c + 4) + 8), 0u);
    }

    // ---- scores, masks (length, block, causal limit of each column)
    if constexpr (KMODE != kFp8) {
      const float ng = lds_h2f(st + a.knorm_off + 2 * g), nh = lds_h2f(st + a.knorm_off + 2 * g + 16);
      v[0] *= ng; v[1] *= ng; v[2] *= nh; v[3] *= nh;
    }
    float svg = lds_h2f(st + a.vscale_off + 2 * g), svh = lds_h2f(st + a.vscale_off + 2 * g + 16);
    float szg = lds_h2f(st + a.vzero_off + 2 * g), szh = lds_h2f(st + a.vzero_off + 2 * g + 16);
    const int pg = tok0 + g, ph = tok0 + g + 8;
    if (!tvalid || pg >= seq) { v[0] = v[1] = -INFINITY; svg = 0.f; szg = 0.f; }
    if (!tvalid || ph >= seq) { v[2] = v[3] = -INFINITY; svh = 0.f; szh = 0.f; }
    if (pg > lim0) v[0] = -INFINITY;
    if (pg > lim1) v[1] = -INFINITY;
    if (ph > lim0) v[2] = -INFINITY;
    if (ph > lim1) v[3] = -INFINITY;
    float cm0 = fmaxf(v[0], v[2]), cm1 = fmaxf(v[1], v[3]);
    if (__any_sync(0xffffffffu, cm0 > m0 + kTau || cm1 > m1 + kTau)) {   // rare: move the max, rescale
#pragma unroll
      for (int o_ = 4; o_ < 32; o_ <<= 1) {
        cm0 = fmaxf(cm0, __shfl_xor_sync(0xffffffffu, cm0, o_));
        cm1 = fmaxf(cm1, __shfl_xor_sync(0xffffffffu, cm1, o_));
      }
      float al0 = 1.f, al1 = 1.f;
      if (cm0 > m0 + kTau) { al0 = ex2(m0 - cm0); m0 = cm0; }
      if (cm1 > m1 + kTau) { al1 = ex2(m1 - cm1); m1 = cm1; }
      l0 *= al0; z0 *= al0; l1 *= al1; z1 *= al1;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o[mt][0] *= al0; o[mt][2] *= al0;
        o[mt][1] *= al1; o[mt][3] *= al1;
      }
    }

    // ---- probabilities, P^T operands (movmatrix), O^T += V^T . P^T
    const float p0 = ex2(v[0] - m0), p1 = ex2(v[1] - m1);
    const float p2 = ex2(v[2] - m0), p3 = ex2(v[3] - m1);
    l0 += p0 + p2;
    l1 += p1 + p3;
    z0 = fmaf(p0, szg, fmaf(p2, szh, z0));
    z1 = fmaf(p1, szg, fmaf(p3, szh, z1));
    uint32_t hg, lg, hh, lh;   // hi/lo half2 of (col 2 c, col 2 c + 1) for tokens g and g + 8
    split_half2(p0 * svg, p1 * svg, hg, lg);
    split_half2(p2 * svh, p3 * svh, hh, lh);
    const uint32_t b0 = movmatrix_trans(hg), b1 = movmatrix_trans(hh);
    const uint32_t b0l = movmatrix_trans(lg), b1l = movmatrix_trans(lh);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {   // rows g, g + 8 of tile mt: coordinates 16 g + 2 mt, + 1
      const uint32_t a0 = code_field<VBITS>(vwa, 2 * mt, 0), a1 = code_field<VBITS>(vwa, 2 * mt + 1, 4);
      const uint32_t a2 = code_field<VBITS>(vwb, 2 * mt, 0), a3 = code_field<VBITS>(vwb, 2 * mt + 1, 4);
      mma16816(o[mt], a0, a1, a2, a3, b0, b1);
      mma16816(o[mt], a0, a1, a2, a3, b0l, b1l);
    }
  }
  asm volatile("cp.async.wait_all;\n" ::: "memory");   // no copy outlives the CTA

  // ---- records of this lane's two columns
  float l_[2] = {l0, l1}, z_[2] = {z0, z1};
#pragma unroll
  for (int e = 0; e < 2; ++e)
#pragma unroll
    for (int o_ = 4; o_ < 32; o_ <<= 1) {
      l_[e] += __shfl_xor_sync(0xffffffffu, l_[e], o_);
      z_[e] += __shfl_xor_sync(0xffffffffu, z_[e], o_);
    }
  const float mm[2] = {m0, m1};
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    if (!(e ? cv1 : cv0)) continue;
    const long long rec = e ? rec1 : rec0;
    const float inv = l_[e] > 0.f ? 1.f / l_[e] : 0.f;
    float* dst = a.rec_o + rec * kD + 16 * g;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)   // value operands carried code * 2^-24 (rows g) and code * 2^-20 (rows g + 8)
      *reinterpret_cast<float2*>(dst + 2 * mt) =
          make_float2(fmaf(o[mt][e], 16777216.f, z_[e]) * inv, fmaf(o[mt][2 + e], 1048576.f, z_[e]) * inv);
    if (g == 0) a.rec_lse[rec] = l_[e] > 0.f ? mm[e] + __log2f(l_[e]) : -INFINITY;
  }
}

// ---------------------------------------------------------------- reduce

struct ContReduceArgs {
  const float* rec_o;
  const float* rec_lse;
  void* out;
  long long rows;   // total_q * n_q
  int n_part;
};

template <typename TO>
__device__ __forceinline__ void store4(void* out, long long i, const float v[4]) {
  if constexpr (std::is_same<TO, float>::value) {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + i) = make_float4(v[0], v[1], v[2], v[3]);
  } else if constexpr (std::is_same<TO, __half>::value) {
    const __half2 a = __floats2half2_rn(v[0], v[1]), b = __floats2half2_rn(v[2], v[3]);
    *reinterpret_cast<uint2*>(static_cast<__half*>(out) + i) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
  } else {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + i) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
  }
}

// A warp per (query, query head): out = sum_p 2^lse_p o_p / sum_p 2^lse_p over
// the partitions, lane l holding coordinates 4 l .. 4 l + 3.
template <typename TO>
__global__ void __launch_bounds__(256) cont_reduce_kernel(const ContReduceArgs r) {
  grid_dep_wait();   // the records come from cont_kernel
  grid_dep_launch();
  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (row >= r.rows) return;
  const float* lse = r.rec_lse + row * r.n_part;
  float mx = -INFINITY;
  for (int p = lane; p < r.n_part; p += 32) mx = fmaxf(mx, ld_dep_f32(lse + p));
#pragma unroll
  for (int o_ = 16; o_ >= 1; o_ >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o_));
  float acc[4] = {0.f, 0.f, 0.f, 0.f}, wsum = 0.f;
  if (mx > -INFINITY) {
    for (int p = 0; p < r.n_part; ++p) {
      const float lp = ld_dep_f32(lse + p);
      if (lp == -INFINITY) continue;
      const float w = ex2(lp - mx);
      const float4 ov = ld_dep_f32x4(reinterpret_cast<const float4*>(r.rec_o + (row * r.n_part + p) * kD) + lane);
      acc[0] = fmaf(w, ov.x, acc[0]);
      acc[1] = fmaf(w, ov.y, acc[1]);
      acc[2] = fmaf(w, ov.z, acc[2]);
      acc[3] = fmaf(w, ov.w, acc[3]);
      wsum += w;
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  const float res[4] = {acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv};
  store4<TO>(r.out, row * kD + 4 * lane, res);
}

// ---------------------------------------------------------------- host

struct ContPlan {
  tq_layout L;
  int group, part_tokens, n_part;
  size_t need;
};

tq_status cont_plan(const tq_config* cfg, int total_q, int max_seq_len, ContPlan* P) {
  if (!cfg) return TQ_ERR_INVALID_ARG;
  tq_status st = make_layout(cfg, &P->L);
  if (st != TQ_OK) return st;
  if (total_q < 0 || max_seq_len < 0) return TQ_ERR_INVALID_ARG;
  if (cfg->num_q_heads <= 0 || cfg->num_q_heads % cfg->num_kv_heads) return TQ_ERR_INVALID_ARG;
  P->group = cfg->num_q_heads / cfg->num_kv_heads;
  if (8 % P->group) return TQ_ERR_UNSUPPORTED;   // G in {1, 2, 4, 8}
  const int pt = cfg->partition_tokens;
  if (pt < 0 || pt % kTileTokens) return TQ_ERR_INVALID_ARG;
  P->part_tokens = effective_partition(cfg);
  if (P->part_tokens > kMaxPartTiles * kTileTokens) return TQ_ERR_UNSUPPORTED;
  P->n_part = static_cast<int>((static_cast<long long>(max_seq_len) + P->part_tokens - 1) / P->part_tokens);
  if (P->n_part < 1) P->n_part = 1;
  const long long recs = static_cast<long long>(total_q) * cfg->num_q_heads * P->n_part;
  if (recs > (1ll << 34)) return TQ_ERR_UNSUPPORTED;
  P->need = static_cast<size_t>(((recs * (kD + 1) * 4 + 15) / 16) * 16);
  return TQ_OK;
}

template <int KMODE, int VBITS>
cudaError_t launch_cont(const ContArgs& a, int q_dtype, dim3 grid, cudaStream_t s) {
  const size_t smem = cont_smem_fixed<KMODE>() + static_cast<size_t>(kRing) * a.tile_bytes;
  auto k = q_dtype == TQ_DTYPE_BF16 ? cont_kernel<KMODE, VBITS, __nv_bfloat16> : cont_kernel<KMODE, VBITS, __half>;
  cudaError_t err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  return launch_pdl(k, grid, dim3(kThreads), smem, s, a);
}

}  // namespace
}  // namespace tq

extern "C" {

size_t tq_continue_workspace_size(const tq_config* cfg, int total_q, int max_seq_len) {
  tq::ContPlan P;
  if (tq::cont_plan(cfg, total_q, max_seq_len, &P) != TQ_OK) return 0;
  return P.need;
}

tq_status tq_continue(const tq_config* cfg, const tq_codebook* cb, const void* q, int q_dtype,
                      const int* query_start, int batch, int total_q, int max_q_len, const void* cache,
                      long long num_blocks, const int* block_table, int bt_stride, const int* seq_lens,
                      int max_seq_len, float scale, void* out, int out_dtype, void* workspace,
                      size_t workspace_bytes, unsigned int* dev_status, tq_stream_t stream) {
  using namespace tq;
  ContPlan P;
  tq_status st = cont_plan(cfg, total_q, max_seq_len, &P);
  if (st != TQ_OK) return st;
  if (batch < 0 || max_q_len < 0 || bt_stride < 1 || num_blocks < 0) return TQ_ERR_INVALID_ARG;
  if (batch > 65535) return TQ_ERR_UNSUPPORTED;
  if (q_dtype != TQ_DTYPE_F16 && q_dtype != TQ_DTYPE_BF16) return TQ_ERR_INVALID_ARG;
  if (out_dtype != TQ_DTYPE_F16 && out_dtype != TQ_DTYPE_BF16 && out_dtype != TQ_DTYPE_F32)
    return TQ_ERR_INVALID_ARG;
  if (!P.L.key_fp8 && (!cb || cb->bits != P.L.key_bits || cb->head_dim != cfg->head_dim))
    return TQ_ERR_INVALID_ARG;
  if (workspace_bytes < P.need) return TQ_ERR_WORKSPACE_TOO_SMALL;
  if (batch == 0 || total_q == 0 || max_q_len == 0) return TQ_OK;
  if (!q || !query_start || !cache || !block_table || !seq_lens || !out || !workspace) return TQ_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(cache) || !aligned16(out) || !aligned16(workspace) ||
      (reinterpret_cast<unsigned long long>(query_start) & 3ull) ||
      (reinterpret_cast<unsigned long long>(block_table) & 3ull) ||
      (reinterpret_cast<unsigned long long>(seq_lens) & 3ull))
    return TQ_ERR_MISALIGNED;
  if (dev_status && (reinterpret_cast<unsigned long long>(dev_status) & 3ull)) return TQ_ERR_MISALIGNED;
  if (num_blocks * cfg->num_kv_heads * (cfg->block_size / kTileTokens) >= (1ll << 31))
    return TQ_ERR_UNSUPPORTED;   // tiles are indexed in 32 bits

  ContArgs a;
  a.cache = static_cast<const uint8_t*>(cache);
  a.num_blocks = num_blocks;
  a.q = q;
  a.query_start = query_start;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.status = dev_status;
  const long long recs = static_cast<long long>(total_q) * cfg->num_q_heads * P.n_part;
  a.rec_o = static_cast<float*>(workspace);
  a.rec_lse = a.rec_o + recs * kD;
  a.batch = batch;
  a.total_q = total_q;
  a.n_q = cfg->num_q_heads;
  a.n_kv = cfg->num_kv_heads;
  a.group = P.group;
  a.qpw = 8 / P.group;
  a.qpc = kWarps * a.qpw;
  a.n_part = P.n_part;
  a.part_tiles = P.part_tokens / kTileTokens;
  a.max_q_len = max_q_len;
  a.block_size = cfg->block_size;
  a.log2_bs = __builtin_ctz(static_cast<unsigned>(cfg->block_size));
  a.tiles_per_block = cfg->block_size / kTileTokens;
  a.bt_stride = bt_stride;
  a.cap = static_cast<int>(static_cast<long long>(bt_stride) * cfg->block_size < (1ll << 30)
                               ? static_cast<long long>(bt_stride) * cfg->block_size : (1ll << 30));
  a.tile_bytes = P.L.tile_bytes;
  a.k_off = P.L.k_off;
  a.v_off = P.L.v_off;
  a.knorm_off = P.L.knorm_off;
  a.vscale_off = P.L.vscale_off;
  a.vzero_off = P.L.vzero_off;
  const float sm_scale = scale > 0.f ? scale : 0.088388347648318440f;   // 1/sqrt(128)
  const float gamma = P.L.key_fp8 ? 1.f : centroid_scale(cb->centroids, cb->num_levels);
  a.qscale = sm_scale * 1.4426950408889634f / gamma;                    // log2(e) / gamma
  for (int i = 0; i < 16; ++i)
    a.cent[i] = (!P.L.key_fp8 && i < cb->num_levels) ? static_cast<float>(static_cast<double>(gamma) * cb->centroids[i]) : 0.f;

  const int nqg = (max_q_len + a.qpc - 1) / a.qpc;
  if (static_cast<long long>(nqg) * cfg->num_kv_heads > (1ll << 31) - 1 || P.n_part > 65535) return TQ_ERR_UNSUPPORTED;
  const dim3 grid(static_cast<unsigned>(nqg * cfg->num_kv_heads), static_cast<unsigned>(P.n_part),
                  static_cast<unsigned>(batch));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t err;
  if (P.L.key_fp8) err = launch_cont<kFp8, 4>(a, q_dtype, grid, s);
  else if (P.L.key_bits == 4) err = launch_cont<kMse4, 4>(a, q_dtype, grid, s);
  else if (P.L.value_bits == 4) err = launch_cont<kMse3, 4>(a, q_dtype, grid, s);
  else err = launch_cont<kMse3, 3>(a, q_dtype, grid, s);
  if (err != cudaSuccess) return TQ_ERR_CUDA;

  ContReduceArgs r;
  r.rec_o = a.rec_o;
  r.rec_lse = a.rec_lse;
  r.out = out;
  r.rows = static_cast<long long>(total_q) * cfg->num_q_heads;
  r.n_part = P.n_part;
  const dim3 rgrid(static_cast<unsigned>((r.rows + 7) / 8));
  if (out_dtype == TQ_DTYPE_F32) err = launch_pdl(cont_reduce_kernel<float>, rgrid, dim3(256), 0, s, r);
  else if (out_dtype == TQ_DTYPE_F16) err = launch_pdl(cont_reduce_kernel<__half>, rgrid, dim3(256), 0, s, r);
  else err = launch_pdl(cont_reduce_kernel<__nv_bfloat16>, rgrid, dim3(256), 0, s, r);
  return err == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // extern "C"
