// tq_decode: split-K attention read straight from the packed paged cache,
// plus the LSE reduce.
//
// Method: "vLLM 源码完全拆解(十九):TurboQuant KV Cache 量化" (pinghaoyang.com.cn),
// section "读取内核:decode 如何从 packed slot 还原 K/V 并保持 Softmax 数值稳定":
//   q_rot = (H / sqrt(d)) q once per query head; score = stored_norm *
//   (q_rot . c[idx]) * scale (FP8 keys: (q . k) * scale, q unrotated)
//   ("分数计算:FP8 K 与 MSE K 的两条路径"); v = fp16 scale * code + fp16 zero
//   ("V 的解包"); per split an online softmax in fp32 writing (acc / l, lse)
//   ("在线 softmax"); a second kernel merges the splits by their LSE
//   ("程序入口:split 区间怎么算"; stage 2).
//
// GB300 design (differs from the pages' one-program-per-query-head Triton
// kernel, which reads every KV tile G = n_q / n_kv times):
//   * one warp owns a work item (sequence b, KV head h, partition p) and
//     computes all G <= 8 query heads of that KV head, so each packed byte is
//     read from HBM exactly once;
//   * the two contractions run on the tensor cores with mma.sync.m16n8k16
//     (f16 inputs, f32 accumulate), operands dequantised in registers:
//       S^T[16 x 8 tok] = Q[16 x 16] . K^T: rows g < 8 carry q_hi of query
//         head g and rows 8+g carry q_lo (q = q_hi + q_lo in fp16); the 16-wide
//         k dimension carries 8 coordinates with centroid hi parts and the
//         same 8 coordinates with centroid lo parts, so one 8-byte LUT entry
//         per key byte yields a whole B fragment and the product is accurate to
//         ~2^-22 relative (fp16 alone misses the 2e-3 output tolerance);
//       O^T[16 d x 8] = V^T[16 d x 16 tok] . P^T: the value codes are exact
//         small integers in fp16, columns carry hi and lo parts of p * scale,
//         and sum_p p * zero is accumulated on the side;
//   * values of token pairs are interleaved in 16-bit words by the store, so a
//     32-bit word gives four half2 (token 2c, token 2c+1) operands directly;
//   * a lazy online-softmax rescale (only when the running max grows by more
//     than 2^8) keeps the accumulator rescales off the common path;
//   * the next 16-token tile is loaded into registers while the current one is
//     computed; block ids of a partition are fetched once, 32 at a time.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kD = 128;
constexpr int kDecWarps = 8;
constexpr float kTau = 8.0f;            // lazy rescale threshold, log2 units
constexpr int kLutCopies = 16;          // one copy per lane of a half warp
constexpr int kScratchFloats = 8 * kD;  // per-warp staging: 8 rows of d floats

enum KeyMode { kMse4 = 4, kMse3 = 3, kFp8 = 8 };

struct DecodeArgs {
  const uint8_t* cache;
  long long num_blocks;
  const void* q;
  const int* block_table;
  const int* seq_lens;
  unsigned int* status;
  float* part_o;       // [batch][n_q][num_parts][d]
  float* part_lse;     // [batch][n_q][num_parts], log2 units
  int batch, n_q, n_kv, group;
  int block_size, tiles_per_block, bt_stride;
  int partition_tokens, num_parts, max_seq_len;
  int tile_bytes, k_off, v_off, knorm_off, vscale_off, vzero_off;
  float qscale;        // softmax scale * log2(e)
  float cent[16];
};

struct ReduceArgs {
  const int* seq_lens;
  const float* part_o;
  const float* part_lse;
  void* out;
  int batch, n_q, num_parts, partition_tokens, max_seq_len, cap;
};

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ void mma16816(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ldg128(const uint8_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldg32(const uint8_t* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];\n" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
// (hi, lo) fp16 split of a float pair: x = hi + lo to ~2^-22 relative.
__device__ __forceinline__ void split_half2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(x0, x1);
  const float2 hf = __half22float2(h);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = pack_half2(x0 - hf.x, x1 - hf.y);
}

template <typename T>
__device__ __forceinline__ void load4(const void* base, long long elem, float out[4]) {
  const uint2 raw = __ldg(reinterpret_cast<const uint2*>(static_cast<const T*>(base) + elem));
  if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
    out[0] = a.x; out[1] = a.y; out[2] = b.x; out[3] = b.y;
  } else {
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
    out[0] = a.x; out[1] = a.y; out[2] = b.x; out[3] = b.y;
  }
}

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

// Lazy online-softmax max update (same rule wherever a copy of a row max lives).
__device__ __forceinline__ float lazy_update(float& m, float chunk_max) {
  if (chunk_max > m + kTau) {
    const float a = exp2f(m - chunk_max);
    m = chunk_max;
    return a;
  }
  return 1.f;
}

// value codes (token A in bits 0..15, token B in bits 16..31 of w) -> half2
// (A, B) of nibble j of each 16-bit half, as exact integers.
__device__ __forceinline__ uint32_t vpair(uint32_t w, int j) {
  const uint32_t biased = ((w >> (4 * j)) & 0x000F000Fu) | 0x64006400u;   // 1024 + code
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&biased), __half2half2(__ushort_as_half(0x6400)));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// ---------------------------------------------------------------- chunk data

template <int KMODE>
struct Chunk {
  uint4 k[KMODE == kFp8 ? 4 : 2];   // key bytes of tokens g and g+8 (this lane's slice)
  uint4 va, vb;                     // value words of token pairs (2c,2c+1), (2c+8,2c+9)
  uint32_t kn0, kn1, vs0, vs1, vz0, vz1;
};

template <int KMODE>
__device__ __forceinline__ void load_chunk(Chunk<KMODE>& ch, const uint8_t* tile, const DecodeArgs& a,
                                           int g, int c) {
  if constexpr (KMODE == kMse4) {
    ch.k[0] = ldg128(tile + a.k_off + g * 64 + 16 * c);
    ch.k[1] = ldg128(tile + a.k_off + (g + 8) * 64 + 16 * c);
  } else if constexpr (KMODE == kMse3) {
    const uint8_t* r0 = tile + a.k_off + g * 48 + 12 * c;
    const uint8_t* r1 = tile + a.k_off + (g + 8) * 48 + 12 * c;
    ch.k[0] = make_uint4(ldg32(r0), ldg32(r0 + 4), ldg32(r0 + 8), 0u);
    ch.k[1] = make_uint4(ldg32(r1), ldg32(r1 + 4), ldg32(r1 + 8), 0u);
  } else {
    ch.k[0] = ldg128(tile + a.k_off + g * 128 + 32 * c);
    ch.k[1] = ldg128(tile + a.k_off + g * 128 + 32 * c + 16);
    ch.k[2] = ldg128(tile + a.k_off + (g + 8) * 128 + 32 * c);
    ch.k[3] = ldg128(tile + a.k_off + (g + 8) * 128 + 32 * c + 16);
  }
  ch.va = ldg128(tile + a.v_off + c * 128 + 16 * g);
  ch.vb = ldg128(tile + a.v_off + (c + 4) * 128 + 16 * g);
  if constexpr (KMODE != kFp8) {
    ch.kn0 = ldg32(tile + a.knorm_off + 4 * c);
    ch.kn1 = ldg32(tile + a.knorm_off + 16 + 4 * c);
  } else {
    ch.kn0 = ch.kn1 = 0x3C003C00u;   // fp16 1.0: FP8 keys carry no norm
  }
  ch.vs0 = ldg32(tile + a.vscale_off + 4 * c);
  ch.vs1 = ldg32(tile + a.vscale_off + 16 + 4 * c);
  ch.vz0 = ldg32(tile + a.vzero_off + 4 * c);
  ch.vz1 = ldg32(tile + a.vzero_off + 16 + 4 * c);
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// Shared-memory LUT: entry e (a key byte, or a 6-bit pair of 3-bit indices)
// -> uint2 {half2(c_hi[lo idx], c_hi[hi idx]), half2(c_lo[..], c_lo[..])},
// kLutCopies copies, 8 bytes apart, entry stride 128 bytes.
constexpr int kLutEntries4 = 256;
__shared__ __align__(128) uint2 g_lut[kLutEntries4 * kLutCopies];

template <int KMODE>
__device__ void build_lut(const float* cent) {
  constexpr int kEntries = KMODE == kMse4 ? 256 : 64;
  constexpr int kShift = KMODE == kMse4 ? 4 : 3;
  constexpr int kMask = (1 << kShift) - 1;
  for (int i = threadIdx.x; i < kEntries * kLutCopies; i += blockDim.x) {
    const int e = i / kLutCopies;
    const float c0 = cent[e & kMask], c1 = cent[(e >> kShift) & kMask];
    uint32_t hi, lo;
    split_half2(c0, c1, hi, lo);
    g_lut[i] = make_uint2(hi, lo);
  }
}

// QK for one n-tile (8 tokens): acc += Q . K^T over d = 128.
template <int KMODE>
__device__ __forceinline__ void qk_tile(float acc[4], const uint32_t qa[32], const uint4* kraw,
                                        uint32_t lut_lane) {
  if constexpr (KMODE == kMse4) {
    const uint4 kq = kraw[0];
#pragma unroll
    for (int s = 0; s < 16; ++s) {
      const uint32_t w = word_of(kq, s >> 2);
      const int sh = 8 * (s & 3) - 7;   // byte (s&3) of w -> bits 7..14
      const uint32_t off = (sh < 0 ? (w << 7) : (w >> sh)) & 0x7F80u;
      const uint2 e = lds64(lut_lane + off);
      mma16816(acc, qa[2 * s], qa[2 * s + 1], qa[2 * s], qa[2 * s + 1], e.x, e.y);
    }
  } else if constexpr (KMODE == kMse3) {
    const uint4 kq = kraw[0];
    const uint32_t w[3] = {kq.x, kq.y, kq.z};
#pragma unroll
    for (int s = 0; s < 16; ++s) {
      const int bit = 6 * s, wi = bit >> 5, sh = bit & 31;
      uint32_t f;
      if (sh <= 26) f = w[wi] >> sh;
      else f = __funnelshift_r(w[wi], w[wi + 1], sh);
      const uint32_t off = (f & 63u) << 7;
      const uint2 e = lds64(lut_lane + off);
      mma16816(acc, qa[2 * s], qa[2 * s + 1], qa[2 * s], qa[2 * s + 1], e.x, e.y);
    }
  } else {
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const uint32_t w = word_of(kraw[s >> 2], s & 3);
      const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xFFFFu), __NV_E4M3);
      const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w >> 16), __NV_E4M3);
      const uint32_t b0 = static_cast<uint32_t>(lo.x) | (static_cast<uint32_t>(lo.y) << 16);
      const uint32_t b1 = static_cast<uint32_t>(hi.x) | (static_cast<uint32_t>(hi.y) << 16);
      mma16816(acc, qa[4 * s], qa[4 * s + 1], qa[4 * s + 2], qa[4 * s + 3], b0, b1);
    }
  }
}

__device__ __forceinline__ float h2f_lo(uint32_t w) { return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu))); }
__device__ __forceinline__ float h2f_hi(uint32_t w) { return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16))); }

// ---------------------------------------------------------------- split kernel

template <int KMODE, int GBIG, typename TQ>
__global__ void __launch_bounds__(kDecWarps * 32, 1)
split_kernel(const DecodeArgs a) {
  extern __shared__ __align__(16) float s_scratch[];
  if constexpr (KMODE != kFp8) build_lut<KMODE>(a.cent);
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane >> 2;          // mma groupID: token row of B, query row of A
  const int c = lane & 3;           // thread in group
  const int G = a.group;
  float* scratch = s_scratch + warp * kScratchFloats;
  uint32_t lut_lane = 0;
  if constexpr (KMODE != kFp8) lut_lane = static_cast<uint32_t>(__cvta_generic_to_shared(g_lut)) + 8u * (lane & 15);
  const int cap = a.bt_stride * a.block_size;

  // column n of O^T belongs to query row col_row(n)
  auto col_row = [&](int n) -> int {
    if (GBIG) return n < G ? n : 0;
    return n < G ? n : (n < 2 * G ? n - G : 0);
  };
  const int rc0 = col_row(2 * c), rc1 = col_row(2 * c + 1);

  const long long total = static_cast<long long>(a.batch) * a.n_kv * a.num_parts;
  for (long long it = static_cast<long long>(blockIdx.x) * kDecWarps + warp; it < total;
       it += static_cast<long long>(gridDim.x) * kDecWarps) {
    const int p = static_cast<int>(it % a.num_parts);
    const long long bh = it / a.num_parts;
    const int h = static_cast<int>(bh % a.n_kv);
    const int b = static_cast<int>(bh / a.n_kv);
    int len = a.seq_lens[b];
    if (len > a.max_seq_len || len > cap) {
      if (lane == 0 && p == 0) flag(a.status, TQ_DEV_SEQ_TOO_LONG);
      len = min(len, min(a.max_seq_len, cap));
    }
    const int start = p * a.partition_tokens;
    if (start >= len) continue;
    const int end = min(start + a.partition_tokens, len);

    // ---- query fragments: rotate (index-coded keys), scale, split hi/lo
    for (int gg = 0; gg < G; ++gg) {
      float x[4];
      load4<TQ>(a.q, (static_cast<long long>(b) * a.n_q + h * G + gg) * kD + 4 * lane, x);
      float sc = a.qscale;
      if constexpr (KMODE != kFp8) {
        fwht128(x, lane);
        sc *= 0.088388347648318440f;   // 1 / sqrt(128)
      }
      *reinterpret_cast<float4*>(scratch + gg * kD + 4 * lane) =
          make_float4(x[0] * sc, x[1] * sc, x[2] * sc, x[3] * sc);
    }
    __syncwarp();
    uint32_t qa[32];
    if constexpr (KMODE == kFp8) {
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const int d0 = 32 * c + 4 * s;
        float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
        if (g < G) {
          x0 = scratch[g * kD + d0]; x1 = scratch[g * kD + d0 + 1];
          x2 = scratch[g * kD + d0 + 2]; x3 = scratch[g * kD + d0 + 3];
        }
        split_half2(x0, x1, qa[4 * s], qa[4 * s + 1]);
        split_half2(x2, x3, qa[4 * s + 2], qa[4 * s + 3]);
      }
    } else {
#pragma unroll
      for (int s = 0; s < 16; ++s) {
        const int d0 = 32 * c + 2 * s;
        float x0 = 0.f, x1 = 0.f;
        if (g < G) { x0 = scratch[g * kD + d0]; x1 = scratch[g * kD + d0 + 1]; }
        split_half2(x0, x1, qa[2 * s], qa[2 * s + 1]);
      }
    }
    __syncwarp();

    // ---- state
    float o[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float mrow = -INFINITY, mc0 = -INFINITY, mc1 = -INFINITY, lsum = 0.f, zsum = 0.f;

    // block ids of this partition, 32 at a time (lane j holds block start/bs + j)
    const int first_blk = start / a.block_size;
    int bid_base = first_blk;
    int bid_reg = -1;
    {
      const int j = bid_base + lane;
      if (j * a.block_size < end) bid_reg = a.block_table[static_cast<long long>(b) * a.bt_stride + j];
    }
    auto tile_of = [&](int pos, bool& ok) -> const uint8_t* {
      const int bi = pos / a.block_size;
      if (bi - bid_base >= 32) {   // warp-uniform refill
        bid_base = bi;
        const int j = bid_base + lane;
        bid_reg = (j * a.block_size < end) ? a.block_table[static_cast<long long>(b) * a.bt_stride + j] : -1;
      }
      const int blk = __shfl_sync(0xffffffffu, bid_reg, bi - bid_base);
      ok = blk >= 0 && blk < a.num_blocks;
      if (!ok) return a.cache;
      return a.cache + ((static_cast<long long>(blk) * a.n_kv + h) * a.tiles_per_block +
                        (pos % a.block_size) / kTileTokens) * static_cast<long long>(a.tile_bytes);
    };

    Chunk<KMODE> cur, nxt;
    bool ok_cur, ok_nxt = false;
    const uint8_t* t0 = tile_of(start, ok_cur);
    if (ok_cur) load_chunk<KMODE>(cur, t0, a, g, c);
    for (int pos = start; pos < end; pos += kTileTokens) {
      const int npos = pos + kTileTokens;
      if (npos < end) {
        const uint8_t* t1 = tile_of(npos, ok_nxt);
        if (ok_nxt) load_chunk<KMODE>(nxt, t1, a, g, c);
      }
      if (!ok_cur) {
        if (lane == 0) flag(a.status, TQ_DEV_BLOCK_OUT_OF_RANGE);
      } else {
        const int nvalid = min(kTileTokens, end - pos);
        // ---- scores S^T (rows: query hi/lo, cols: tokens)
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
        qk_tile<KMODE>(s0, qa, &cur.k[0], lut_lane);
        qk_tile<KMODE>(s1, qa, &cur.k[KMODE == kFp8 ? 2 : 1], lut_lane);
        // tokens 2c, 2c+1, 2c+8, 2c+9 of this tile, for query row g
        float sc[4];
        sc[0] = (s0[0] + s0[2]) * h2f_lo(cur.kn0);
        sc[1] = (s0[1] + s0[3]) * h2f_hi(cur.kn0);
        sc[2] = (s1[0] + s1[2]) * h2f_lo(cur.kn1);
        sc[3] = (s1[1] + s1[3]) * h2f_hi(cur.kn1);
        const int tk[4] = {2 * c, 2 * c + 1, 2 * c + 8, 2 * c + 9};
#pragma unroll
        for (int e = 0; e < 4; ++e) if (tk[e] >= nvalid) sc[e] = -INFINITY;
        float cm = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
        cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 1));
        cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 2));
        const float cm0 = __shfl_sync(0xffffffffu, cm, 4 * rc0);
        const float cm1 = __shfl_sync(0xffffffffu, cm, 4 * rc1);
        const float ar = lazy_update(mrow, cm);
        const float a0 = lazy_update(mc0, cm0);
        const float a1 = lazy_update(mc1, cm1);
        if (ar != 1.f) { lsum *= ar; zsum *= ar; }
        if (a0 != 1.f) {
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) { o[mt][0] *= a0; o[mt][2] *= a0; }
        }
        if (a1 != 1.f) {
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) { o[mt][1] *= a1; o[mt][3] *= a1; }
        }
        float ps[4];
        const float vsc[4] = {h2f_lo(cur.vs0), h2f_hi(cur.vs0), h2f_lo(cur.vs1), h2f_hi(cur.vs1)};
        const float vzr[4] = {h2f_lo(cur.vz0), h2f_hi(cur.vz0), h2f_lo(cur.vz1), h2f_hi(cur.vz1)};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const bool valid = tk[e] < nvalid;
          const float pe = valid ? exp2f(sc[e] - mrow) : 0.f;
          lsum += pe;
          ps[e] = valid ? pe * vsc[e] : 0.f;
          zsum = valid ? fmaf(pe, vzr[e], zsum) : zsum;
        }
        uint32_t hi01, lo01, hi23, lo23;
        split_half2(ps[0], ps[1], hi01, lo01);
        split_half2(ps[2], ps[3], hi23, lo23);
        const bool real_row = g < G;
        if (GBIG) {
          const uint32_t b0h = real_row ? hi01 : 0u, b1h = real_row ? hi23 : 0u;
          const uint32_t b0l = real_row ? lo01 : 0u, b1l = real_row ? lo23 : 0u;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            const uint32_t wa = word_of(cur.va, mt >> 1), wb = word_of(cur.vb, mt >> 1);
            const int j0 = 2 * (mt & 1);
            const uint32_t v0 = vpair(wa, j0), v1 = vpair(wa, j0 + 1);
            const uint32_t v2 = vpair(wb, j0), v3 = vpair(wb, j0 + 1);
            mma16816(o[mt], v0, v1, v2, v3, b0h, b1h);
            mma16816(o[mt], v0, v1, v2, v3, b0l, b1l);
          }
        } else {
          const int src = (lane - 4 * G) & 31;
          const uint32_t t01 = __shfl_sync(0xffffffffu, lo01, src);
          const uint32_t t23 = __shfl_sync(0xffffffffu, lo23, src);
          const uint32_t b0 = real_row ? hi01 : (g < 2 * G ? t01 : 0u);
          const uint32_t b1 = real_row ? hi23 : (g < 2 * G ? t23 : 0u);
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            const uint32_t wa = word_of(cur.va, mt >> 1), wb = word_of(cur.vb, mt >> 1);
            const int j0 = 2 * (mt & 1);
            mma16816(o[mt], vpair(wa, j0), vpair(wa, j0 + 1), vpair(wb, j0), vpair(wb, j0 + 1), b0, b1);
          }
        }
      }
      cur = nxt;
      ok_cur = ok_nxt;
    }

    // ---- finalize: combine hi/lo columns, add sum p*zero, normalise, store
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
    zsum += __shfl_xor_sync(0xffffffffu, zsum, 1);
    zsum += __shfl_xor_sync(0xffffffffu, zsum, 2);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int d0 = 16 * g + 2 * mt;
      scratch[(2 * c) * kD + d0] = o[mt][0];
      scratch[(2 * c + 1) * kD + d0] = o[mt][1];
      scratch[(2 * c) * kD + d0 + 1] = o[mt][2];
      scratch[(2 * c + 1) * kD + d0 + 1] = o[mt][3];
    }
    __syncwarp();
    for (int gg = 0; gg < G; ++gg) {
      const float l = __shfl_sync(0xffffffffu, lsum, 4 * gg);
      const float z = __shfl_sync(0xffffffffu, zsum, 4 * gg);
      const float m = __shfl_sync(0xffffffffu, mrow, 4 * gg);
      float4 v = *reinterpret_cast<const float4*>(scratch + gg * kD + 4 * lane);
      if (!GBIG) {
        const float4 w = *reinterpret_cast<const float4*>(scratch + (G + gg) * kD + 4 * lane);
        v.x += w.x; v.y += w.y; v.z += w.z; v.w += w.w;
      }
      // l == 0 only when every tile of the partition was skipped (bad block ids)
      const float inv = l > 0.f ? 1.f / l : 0.f;
      v.x = (v.x + z) * inv; v.y = (v.y + z) * inv; v.z = (v.z + z) * inv; v.w = (v.w + z) * inv;
      const long long row = (static_cast<long long>(b) * a.n_q + h * G + gg) * a.num_parts + p;
      *reinterpret_cast<float4*>(a.part_o + row * kD + 4 * lane) = v;
      if (lane == 0) a.part_lse[row] = l > 0.f ? m + __log2f(l) : -INFINITY;
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------- reduce

template <typename TO>
__device__ __forceinline__ void store_out(void* out, long long i, float v) {
  if constexpr (std::is_same<TO, float>::value) static_cast<float*>(out)[i] = v;
  else if constexpr (std::is_same<TO, __half>::value) static_cast<__half*>(out)[i] = __float2half_rn(v);
  else static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
}

template <typename TO>
__global__ void __launch_bounds__(kD) reduce_kernel(const ReduceArgs a) {
  const int hq = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
  int len = a.seq_lens[b];
  len = min(len, min(a.max_seq_len, a.cap));
  const long long orow = static_cast<long long>(b) * a.n_q + hq;
  if (len <= 0) { store_out<TO>(a.out, orow * kD + d, 0.f); return; }
  const int parts = (len + a.partition_tokens - 1) / a.partition_tokens;
  const long long base = orow * a.num_parts;
  float mx = -INFINITY;
  for (int p = 0; p < parts; ++p) mx = fmaxf(mx, a.part_lse[base + p]);
  if (mx == -INFINITY) { store_out<TO>(a.out, orow * kD + d, 0.f); return; }
  float acc = 0.f, den = 0.f;
  for (int p = 0; p < parts; ++p) {
    const float w = exp2f(a.part_lse[base + p] - mx);
    den += w;
    acc = fmaf(w, a.part_o[(base + p) * kD + d], acc);
  }
  store_out<TO>(a.out, orow * kD + d, acc / den);
}

// ---------------------------------------------------------------- host glue

struct Prepared {
  tq_layout L;
  int pt, num_parts, cap;
  size_t need;
};

tq_status prepare(const tq_config* cfg, int batch, int max_seq_len, int bt_stride, size_t ws_bytes,
                  const void* workspace, Prepared* out) {
  tq_status st = make_layout(cfg, &out->L);
  if (st != TQ_OK) return st;
  if (batch < 0 || max_seq_len < 0 || bt_stride < 0) return TQ_ERR_INVALID_ARG;
  if (cfg->num_q_heads <= 0 || cfg->num_q_heads % cfg->num_kv_heads) return TQ_ERR_INVALID_ARG;
  if (cfg->num_q_heads / cfg->num_kv_heads > 8) return TQ_ERR_UNSUPPORTED;
  out->pt = effective_partition(cfg);
  if (out->pt % kTileTokens || out->pt < 16 || out->pt > 65536) return TQ_ERR_INVALID_ARG;
  out->num_parts = static_cast<int>((static_cast<long long>(max_seq_len) + out->pt - 1) / out->pt);
  if (out->num_parts < 1) out->num_parts = 1;
  out->cap = bt_stride * cfg->block_size;
  out->need = tq_decode_workspace_size(cfg, batch, max_seq_len);
  if (ws_bytes < out->need) return TQ_ERR_WORKSPACE_TOO_SMALL;
  if (batch > 0 && !aligned16(workspace)) return TQ_ERR_MISALIGNED;
  return TQ_OK;
}

template <int KMODE, int GBIG>
cudaError_t launch_split_typed(const DecodeArgs& a, int q_dtype, cudaStream_t s, int sms) {
  const size_t dyn = static_cast<size_t>(kDecWarps) * kScratchFloats * sizeof(float);
  const long long items = static_cast<long long>(a.batch) * a.n_kv * a.num_parts;
  long long blocks = (items + kDecWarps - 1) / kDecWarps;
  const long long cap_blocks = static_cast<long long>(sms);
  if (blocks > cap_blocks) blocks = cap_blocks;
  if (blocks < 1) blocks = 1;
  if (q_dtype == TQ_DTYPE_BF16) {
    auto k = split_kernel<KMODE, GBIG, __nv_bfloat16>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(dyn));
    k<<<static_cast<unsigned>(blocks), kDecWarps * 32, dyn, s>>>(a);
  } else {
    auto k = split_kernel<KMODE, GBIG, __half>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(dyn));
    k<<<static_cast<unsigned>(blocks), kDecWarps * 32, dyn, s>>>(a);
  }
  return cudaGetLastError();
}

template <int KMODE>
cudaError_t launch_split(const DecodeArgs& a, int q_dtype, cudaStream_t s, int sms) {
  return a.group > 4 ? launch_split_typed<KMODE, 1>(a, q_dtype, s, sms)
                     : launch_split_typed<KMODE, 0>(a, q_dtype, s, sms);
}

tq_status run_partials(const tq_config* cfg, const tq_codebook* cb, const void* q, int q_dtype,
                       const void* cache, long long num_blocks, const int* block_table, int bt_stride,
                       const int* seq_lens, int batch, int max_seq_len, float scale, void* workspace,
                       size_t ws_bytes, unsigned int* dev_status, cudaStream_t stream) {
  Prepared P;
  tq_status st = prepare(cfg, batch, max_seq_len, bt_stride, ws_bytes, workspace, &P);
  if (st != TQ_OK) return st;
  if (q_dtype != TQ_DTYPE_F16 && q_dtype != TQ_DTYPE_BF16) return TQ_ERR_INVALID_ARG;
  if (!P.L.key_fp8 && (!cb || cb->bits != P.L.key_bits || cb->head_dim != cfg->head_dim))
    return TQ_ERR_INVALID_ARG;
  if (batch == 0) return TQ_OK;
  if (!q || !cache || !block_table || !seq_lens || !workspace) return TQ_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(cache) || (reinterpret_cast<unsigned long long>(block_table) & 3ull) ||
      (reinterpret_cast<unsigned long long>(seq_lens) & 3ull))
    return TQ_ERR_MISALIGNED;
  if (num_blocks < 0 || bt_stride < 1) return TQ_ERR_INVALID_ARG;

  DecodeArgs a;
  a.cache = static_cast<const uint8_t*>(cache);
  a.num_blocks = num_blocks;
  a.q = q;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.status = dev_status;
  const long long rows = static_cast<long long>(batch) * cfg->num_q_heads * P.num_parts;
  a.part_o = static_cast<float*>(workspace);
  a.part_lse = a.part_o + rows * kD;
  a.batch = batch;
  a.n_q = cfg->num_q_heads;
  a.n_kv = cfg->num_kv_heads;
  a.group = cfg->num_q_heads / cfg->num_kv_heads;
  a.block_size = cfg->block_size;
  a.tiles_per_block = cfg->block_size / kTileTokens;
  a.bt_stride = bt_stride;
  a.partition_tokens = P.pt;
  a.num_parts = P.num_parts;
  a.max_seq_len = max_seq_len;
  a.tile_bytes = P.L.tile_bytes;
  a.k_off = P.L.k_off;
  a.v_off = P.L.v_off;
  a.knorm_off = P.L.knorm_off;
  a.vscale_off = P.L.vscale_off;
  a.vzero_off = P.L.vzero_off;
  const float sm_scale = scale > 0.f ? scale : 0.088388347648318440f;   // 1/sqrt(128)
  a.qscale = sm_scale * 1.4426950408889634f;                              // log2(e)
  for (int i = 0; i < 16; ++i) a.cent[i] = (!P.L.key_fp8 && i < cb->num_levels) ? cb->centroids[i] : 0.f;

  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaError_t err;
  if (P.L.key_fp8) err = launch_split<kFp8>(a, q_dtype, stream, sms);
  else if (P.L.key_bits == 4) err = launch_split<kMse4>(a, q_dtype, stream, sms);
  else err = launch_split<kMse3>(a, q_dtype, stream, sms);
  return err == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

tq_status run_reduce(const tq_config* cfg, const int* seq_lens, int batch, int max_seq_len, int bt_stride,
                     void* out, int out_dtype, const void* workspace, size_t ws_bytes, cudaStream_t stream) {
  Prepared P;
  tq_status st = prepare(cfg, batch, max_seq_len, bt_stride, ws_bytes, workspace, &P);
  if (st != TQ_OK) return st;
  if (out_dtype != TQ_DTYPE_F16 && out_dtype != TQ_DTYPE_BF16 && out_dtype != TQ_DTYPE_F32)
    return TQ_ERR_INVALID_ARG;
  if (batch == 0) return TQ_OK;
  if (!seq_lens || !out || !workspace) return TQ_ERR_INVALID_ARG;
  if (!aligned16(out)) return TQ_ERR_MISALIGNED;
  if (bt_stride < 1) return TQ_ERR_INVALID_ARG;
  ReduceArgs r;
  r.seq_lens = seq_lens;
  const long long rows = static_cast<long long>(batch) * cfg->num_q_heads * P.num_parts;
  r.part_o = static_cast<const float*>(workspace);
  r.part_lse = r.part_o + rows * kD;
  r.out = out;
  r.batch = batch;
  r.n_q = cfg->num_q_heads;
  r.num_parts = P.num_parts;
  r.partition_tokens = P.pt;
  r.max_seq_len = max_seq_len;
  r.cap = P.cap;
  const dim3 grid(static_cast<unsigned>(cfg->num_q_heads), static_cast<unsigned>(batch));
  if (out_dtype == TQ_DTYPE_F32) reduce_kernel<float><<<grid, kD, 0, stream>>>(r);
  else if (out_dtype == TQ_DTYPE_F16) reduce_kernel<__half><<<grid, kD, 0, stream>>>(r);
  else reduce_kernel<__nv_bfloat16><<<grid, kD, 0, stream>>>(r);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // namespace
}  // namespace tq

extern "C" {

tq_status tq_decode_partials(const tq_config* cfg, const tq_codebook* cb, const void* q, int q_dtype,
                             const void* cache, long long num_blocks, const int* block_table, int bt_stride,
                             const int* seq_lens, int batch, int max_seq_len, float scale, void* workspace,
                             size_t workspace_bytes, unsigned int* dev_status, tq_stream_t stream) {
  return tq::run_partials(cfg, cb, q, q_dtype, cache, num_blocks, block_table, bt_stride, seq_lens, batch,
                          max_seq_len, scale, workspace, workspace_bytes, dev_status,
                          reinterpret_cast<cudaStream_t>(stream));
}

tq_status tq_decode_reduce(const tq_config* cfg, const int* seq_lens, int batch, int max_seq_len, int bt_stride,
                           void* out, int out_dtype, const void* workspace, size_t workspace_bytes,
                           tq_stream_t stream) {
  return tq::run_reduce(cfg, seq_lens, batch, max_seq_len, bt_stride, out, out_dtype, workspace,
                        workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

tq_status tq_decode(const tq_config* cfg, const tq_codebook* cb, const void* q, int q_dtype, const void* cache,
                    long long num_blocks, const int* block_table, int bt_stride, const int* seq_lens, int batch,
                    int max_seq_len, float scale, void* out, int out_dtype, void* workspace,
                    size_t workspace_bytes, unsigned int* dev_status, tq_stream_t stream) {
  if (out_dtype != TQ_DTYPE_F16 && out_dtype != TQ_DTYPE_BF16 && out_dtype != TQ_DTYPE_F32)
    return TQ_ERR_INVALID_ARG;
  if (batch > 0 && !out) return TQ_ERR_INVALID_ARG;
  if (batch > 0 && !tq::aligned16(out)) return TQ_ERR_MISALIGNED;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  tq_status st = tq::run_partials(cfg, cb, q, q_dtype, cache, num_blocks, block_table, bt_stride, seq_lens,
                                  batch, max_seq_len, scale, workspace, workspace_bytes, dev_status, s);
  if (st != TQ_OK) return st;
  return tq::run_reduce(cfg, seq_lens, batch, max_seq_len, bt_stride, out, out_dtype, workspace,
                        workspace_bytes, s);
}

}  // extern "C"
