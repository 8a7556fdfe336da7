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
// GB300 design (the pages' Triton kernel runs one program per QUERY head and a
// fixed split count, so every KV tile is read G = n_q / n_kv times):
//
//  Work split. The cache positions are cut into 16-token tiles; the tiles of
//  all (sequence, KV head) pairs, in (b, h, t) order, form one line of T tiles
//  that is cut into equal contiguous ranges, one per warp of a persistent grid
//  (stream-K). A warp's range crosses (b, h) "segments" (optionally also cut at
//  every partition_tokens positions); for every segment it touches the warp
//  writes one partial record (acc / l, lse for all G query heads) at index
//  segment + warp, which is unique because both sequences are monotone. Every
//  warp does the same amount of work whatever the sequence lengths are.
//
//  Data movement. Each warp owns a ring of 4 tile buffers in shared memory fed
//  by cp.async.bulk (one 2144-byte copy per tile at 4bit_nc, completion on an
//  mbarrier) and two query buffers fed the same way; the ring runs ahead across
//  segment boundaries. Block ids are read 32 at a time into a lane-indexed
//  register window. Every mbarrier wait is bounded: on expiry the warp flags
//  TQ_DEV_TIMEOUT, drains its own copies (bounded again) and stops.
//
//  Math. Both contractions run on tensor cores with mma.sync.m16n8k16 (f16 in,
//  f32 accumulate), operands dequantised in registers:
//    S^T[16 x 8 tok] = Q[16 x 16] . K^T. Rows g < 8 carry q_hi of query head g
//      and rows 8 + g carry q_lo (q = q_hi + q_lo in fp16). The 16-wide k
//      dimension holds 8 coordinates with centroid hi parts and the same 8
//      with centroid lo parts: one 8-byte LUT entry per key byte (32 copies,
//      one per lane, so lookups never conflict; the table is aligned so one
//      PRMT forms the address) yields a whole B fragment, and the product is
//      accurate to ~2^-22 relative (fp16 operands alone miss the 2e-3 gate).
//    O^T[16 d x 8] = V^T[16 d x 16 tok] . P^T. Value codes are exact fp16
//      integers; the store interleaves the 16-bit words of token pairs so one
//      32-bit word gives four (token 2c, token 2c+1) operand pairs. Columns
//      carry hi and lo parts of p * scale; sum_p p * zero is kept on the side.
//  Softmax in log2 units with a lazy rescale (the running max only moves when
//  it grows by more than 2^8).

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
constexpr int kWarps = 12;              // warps per CTA, one CTA per SM
constexpr int kStages = 4;              // tile buffers per warp
constexpr float kTau = 8.0f;            // lazy rescale threshold, log2 units
constexpr uint32_t kWaitLimit = 1u << 21;
constexpr int kQBufBytes = 8 * kD * 2;  // G <= 8 rows of 16-bit q
constexpr int kMaxCtas = 256;           // grid cap; sizes the workspace without a device query

enum KeyMode { kMse4 = 4, kMse3 = 3, kFp8 = 8 };

struct DecodeArgs {
  const uint8_t* cache;
  long long num_blocks;
  const void* q;
  const int* block_table;
  const int* seq_lens;
  unsigned int* status;
  float* rec_o;        // [num_records][G][d]
  float* rec_lse;      // [num_records][G], log2 units
  int batch, n_q, n_kv, group;
  int block_size, log2_bs, tiles_per_block, bt_stride;
  int part_tiles;      // tiles per partition (0: whole sequence)
  int num_parts;       // partitions per (b, h) in the record index
  int max_seq_len, cap;
  int tile_bytes, tile_stride, k_off, v_off, knorm_off, vscale_off, vzero_off;
  int warp_bytes;      // per-warp shared buffer
  int dyn_bytes;
  float qscale;        // softmax scale * log2(e)
  float cent[16];
};

struct ReduceArgs {
  const int* seq_lens;
  const float* rec_o;
  const float* rec_lse;
  void* out;
  int batch, n_q, n_kv, group, part_tiles, num_parts, max_seq_len, cap, num_warps;
};

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ void mma16816(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];\n" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts64(uint32_t a, uint2 v) {
  asm volatile("st.shared.v2.u32 [%0], {%1,%2};\n" ::"r"(a), "r"(v.x), "r"(v.y));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait; returns false when the limit expired.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitLimit; ++i)
    if (mbar_try(bar, parity)) return true;
  return false;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;\n" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void bulk_g2s_plain(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(p));
  return p;
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
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
__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

template <typename T>
__device__ __forceinline__ void u2_to_f4(uint2 raw, float out[4]) {
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

// Sylvester-order Walsh-Hadamard transform of 128 values held as 4
// consecutive coordinates per lane (coordinate 4 * lane + j).
__device__ __forceinline__ void fwht128(float v[4], int lane) {
  float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
  v[0] = a0 + a2; v[2] = a0 - a2; v[1] = a1 + a3; v[3] = a1 - a3;
#pragma unroll
  for (int m = 1; m <= 16; m <<= 1) {
    const float sgn = (lane & m) ? -1.f : 1.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float p = __shfl_xor_sync(0xffffffffu, v[j], m);
      v[j] = fmaf(sgn, v[j], p);   // lower index: v + p, upper: p - v
    }
  }
}

__device__ __forceinline__ void flag(unsigned int* status, unsigned int bit) {
  if (status) atomicOr(status, bit);
}

__device__ __forceinline__ float lazy_update(float& m, float chunk_max) {
  if (chunk_max > m + kTau) {
    const float a = ex2(m - chunk_max);
    m = chunk_max;
    return a;
  }
  return 1.f;
}

// value codes -> half2 operands: token A in bits 0..15, token B in bits 16..31
// of w; nibble j of each half, as exact integers (1024 + code, minus 1024).
__device__ __forceinline__ uint32_t vpair(uint32_t w, int j) {
  const uint32_t biased = ((w >> (4 * j)) & 0x000F000Fu) | 0x64006400u;
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&biased), __half2half2(__ushort_as_half(0x6400)));
  return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// ---------------------------------------------------------------- LUT

// Entry e (a key byte, or a 6-bit pair of 3-bit indices) holds, for each of 32
// lanes, uint2 {half2(c_hi[lo idx], c_hi[hi idx]), half2(c_lo[..], c_lo[..])};
// entry stride 256 bytes. The table is aligned to its own size, so the address
// of (entry, lane) is the entry number OR-ed into bits 8.. of the lane's base:
// for 4-bit keys a single byte permute of the key word.
template <int KMODE>
__host__ __device__ constexpr uint32_t lut_bytes() { return KMODE == kMse4 ? 65536u : (KMODE == kMse3 ? 16384u : 0u); }

template <int KMODE>
__device__ void build_lut(uint32_t lut, const float* cent) {
  constexpr int kEntries = KMODE == kMse4 ? 256 : 64;
  constexpr int kShift = KMODE == kMse4 ? 4 : 3;
  constexpr int kMask = (1 << kShift) - 1;
  for (int i = threadIdx.x; i < kEntries * 32; i += blockDim.x) {
    const int e = i >> 5;
    uint32_t hi, lo;
    split_half2(cent[e & kMask], cent[(e >> kShift) & kMask], hi, lo);
    sts64(lut + 8u * i, make_uint2(hi, lo));
  }
}

// S^T for one n-tile of 8 tokens, two independent accumulator chains.
template <int KMODE>
__device__ __forceinline__ void qk_tile(float acc[2][4], const uint32_t qa[32], const uint4* kraw,
                                        uint32_t lut_lane) {
  if constexpr (KMODE == kMse4) {
    const uint4 kq = kraw[0];
#pragma unroll
    for (int s = 0; s < 16; ++s) {
      const uint32_t w = word_of(kq, s >> 2);
      const uint32_t addr = __byte_perm(w, lut_lane, 0x7604u | ((s & 3) << 4));
      const uint2 e = lds64(addr);
      mma16816(acc[s & 1], qa[2 * s], qa[2 * s + 1], qa[2 * s], qa[2 * s + 1], e.x, e.y);
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
      const uint32_t addr = ((f << 8) & 0x3F00u) | lut_lane;
      const uint2 e = lds64(addr);
      mma16816(acc[s & 1], qa[2 * s], qa[2 * s + 1], qa[2 * s], qa[2 * s + 1], e.x, e.y);
    }
  } else {
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const uint32_t w = word_of(kraw[s >> 2], s & 3);
      const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xFFFFu), __NV_E4M3);
      const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w >> 16), __NV_E4M3);
      const uint32_t b0 = static_cast<uint32_t>(lo.x) | (static_cast<uint32_t>(lo.y) << 16);
      const uint32_t b1 = static_cast<uint32_t>(hi.x) | (static_cast<uint32_t>(hi.y) << 16);
      mma16816(acc[s & 1], qa[4 * s], qa[4 * s + 1], qa[4 * s + 2], qa[4 * s + 3], b0, b1);
    }
  }
}

// ---------------------------------------------------------------- tile walker

// Position in the (b, h, t) tile line. All fields are warp-uniform.
struct Walk {
  int b, h, t;      // sequence, KV head, tile within the sequence
  int nt;           // tiles of sequence b
  int len;          // clamped length of sequence b
  int lens_base;    // first sequence of the lane-cached length window
  int lens_reg;     // lane j: clamped length of sequence lens_base + j
};

__device__ __forceinline__ int clamp_len(const DecodeArgs& a, int len) {
  return min(max(len, 0), min(a.max_seq_len, a.cap));
}

__device__ __forceinline__ void lens_fill(Walk& w, const DecodeArgs& a, int base, int lane) {
  w.lens_base = base;
  const int j = base + lane;
  w.lens_reg = j < a.batch ? clamp_len(a, __ldg(a.seq_lens + j)) : 0;
}

__device__ __forceinline__ int lens_get(Walk& w, const DecodeArgs& a, int b, int lane) {
  if (b - w.lens_base >= 32 || b < w.lens_base) lens_fill(w, a, b, lane);
  return __shfl_sync(0xffffffffu, w.lens_reg, b - w.lens_base);
}

// Move to the next tile; skips empty sequences. Returns false past the end.
__device__ __forceinline__ bool walk_next(Walk& w, const DecodeArgs& a, int lane) {
  if (++w.t < w.nt) return true;
  w.t = 0;
  if (++w.h < a.n_kv) return true;
  w.h = 0;
  while (++w.b < a.batch) {
    w.len = lens_get(w, a, w.b, lane);
    w.nt = (w.len + kTileTokens - 1) / kTileTokens;
    if (w.nt > 0) return true;
  }
  return false;
}

__device__ __forceinline__ long long segment_of(const Walk& w, const DecodeArgs& a) {
  const int p = a.part_tiles > 0 ? w.t / a.part_tiles : 0;
  return (static_cast<long long>(w.b) * a.n_kv + w.h) * a.num_parts + p;
}

// ---------------------------------------------------------------- split kernel

template <int KMODE, int GBIG, typename TQ>
__global__ void __launch_bounds__(kWarps * 32, 1)
split_kernel(const DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t s_dyn[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane >> 2;          // mma groupID: token row of B, query row of A
  const int c = lane & 3;           // thread in group
  const int G = a.group;

  // ---- shared-memory plan: LUT at an address aligned to its size, warp
  // buffers packed around it (identical in every thread)
  const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(s_dyn));
  const uint32_t end = base + static_cast<uint32_t>(a.dyn_bytes);
  constexpr uint32_t kLut = lut_bytes<KMODE>();
  const uint32_t lut = kLut ? ((base + kLut - 1) & ~(kLut - 1)) : end;
  uint32_t wbase = base, my_base = 0;
  for (int w = 0; w <= warp; ++w) {
    if (kLut && wbase < lut + kLut && wbase + a.warp_bytes > lut) wbase = lut + kLut;
    if (w == warp) my_base = wbase;
    wbase += a.warp_bytes;
  }
  const bool fits = my_base + a.warp_bytes <= end && (!kLut || lut + kLut <= end);
  if (!__syncthreads_and(fits)) {   // launch misconfigured: flag and leave
    if (threadIdx.x == 0) flag(a.status, TQ_DEV_TIMEOUT);
    return;
  }
  if constexpr (kLut != 0) build_lut<KMODE>(lut, a.cent);

  const uint32_t ring = my_base;                                  // kStages tiles
  const uint32_t qbuf = ring + kStages * a.tile_stride;           // 2 query buffers
  const uint32_t bars = qbuf + 2 * kQBufBytes;                    // kStages + 2 mbarriers
  if (lane == 0) {
    for (int i = 0; i < kStages + 2; ++i) mbar_init(bars + 8 * i, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();   // LUT built, barriers initialised

  uint32_t lut_lane = 0;
  if constexpr (kLut != 0) lut_lane = lut + 8u * lane;
  const uint64_t policy = evict_first_policy();

  // ---- this warp's range of the tile line
  const long long nwarps = static_cast<long long>(gridDim.x) * kWarps;
  const long long wid = static_cast<long long>(blockIdx.x) * kWarps + warp;
  // total tiles: n_kv * sum_b ceil(len_b / 16)
  long long total = 0;
  bool too_long = false;
  for (int b0 = 0; b0 < a.batch; b0 += 32) {
    const int j = b0 + lane;
    int nt = 0;
    if (j < a.batch) {
      const int raw = __ldg(a.seq_lens + j);
      too_long |= raw > min(a.max_seq_len, a.cap);
      nt = (clamp_len(a, raw) + kTileTokens - 1) / kTileTokens;
    }
    for (int o = 1; o < 32; o <<= 1) nt += __shfl_xor_sync(0xffffffffu, nt, o);
    total += nt;
  }
  if (wid == 0 && __any_sync(0xffffffffu, too_long) && lane == 0) flag(a.status, TQ_DEV_SEQ_TOO_LONG);
  total *= a.n_kv;
  const long long r0 = total * wid / nwarps, r1 = total * (wid + 1) / nwarps;
  if (r0 >= r1) return;

  // locate tile r0
  Walk pw;   // producer cursor
  {
    long long acc = 0;   // tiles before sequence b, times n_kv
    int b = 0;
    lens_fill(pw, a, 0, lane);
    for (;;) {
      const int len = lens_get(pw, a, b, lane);
      const int nt = (len + kTileTokens - 1) / kTileTokens;
      const long long span = static_cast<long long>(nt) * a.n_kv;
      if (r0 < acc + span) {
        const long long off = r0 - acc;
        pw.b = b; pw.len = len; pw.nt = nt;
        pw.h = static_cast<int>(off / nt);
        pw.t = static_cast<int>(off - static_cast<long long>(pw.h) * nt);
        break;
      }
      acc += span;
      ++b;
    }
  }
  Walk cw = pw;   // consumer cursor

  // block-id window of the producer: lane j holds block (bid_base + j) of bid_b
  int bid_b = -1, bid_base = 0, bid_reg = 0;

  // ring bookkeeping
  long long pi = r0, ci = r0;         // next tile to issue / to consume
  unsigned tile_ok_bits = 0;          // per stage: block id was valid
  long long p_seg = -1, c_seg = -1;   // segment of the last issued / consumed tile
  int p_qslot = 1, c_qslot = 1;       // query buffer of that segment
  unsigned q_uses0 = 0, q_uses1 = 0;  // phases consumed per query buffer
  unsigned q_iss0 = 0, q_iss1 = 0;    // phases issued per query buffer
  bool p_done = false, aborted = false;

  // per-segment state
  uint32_t qa[32];
  float o[8][4];
  float mrow = -INFINITY, mc0 = -INFINITY, mc1 = -INFINITY, lsum = 0.f, zsum = 0.f;
  const auto col_row = [&](int n) -> int {
    if (GBIG) return n < G ? n : 0;
    return n < G ? n : (n < 2 * G ? n - G : 0);
  };
  const int rc0 = col_row(2 * c), rc1 = col_row(2 * c + 1);

  while (ci < r1 && !aborted) {
    // ---------------- producer: keep up to kStages tiles in flight; a new
    // segment needs a free query buffer (the consumer must have begun the
    // segment before it)
    while (!p_done && pi - ci < kStages) {
      const long long seg = segment_of(pw, a);
      const bool new_seg = seg != p_seg;
      if (new_seg && p_seg >= 0 && c_seg < p_seg) break;
      if (new_seg) {
        p_qslot ^= 1;
        if (p_qslot) ++q_iss1; else ++q_iss0;
        if (lane == 0) {
          const uint32_t bar = bars + 8 * (kStages + p_qslot);
          const uint8_t* src = static_cast<const uint8_t*>(a.q) +
                               (static_cast<long long>(pw.b) * a.n_q + static_cast<long long>(pw.h) * G) * kD * 2;
          fence_proxy_async();
          mbar_expect(bar, G * kD * 2);
          bulk_g2s_plain(qbuf + p_qslot * kQBufBytes, src, G * kD * 2, bar);
        }
        p_seg = seg;
      }
      const int stage = static_cast<int>(pi % kStages);
      const int blk_i = (pw.t << 4) >> a.log2_bs;   // block index within the sequence
      if (pw.b != bid_b || blk_i - bid_base >= 32 || blk_i < bid_base) {
        bid_b = pw.b;
        bid_base = blk_i;
        const int j = bid_base + lane;
        bid_reg = (j * a.block_size < pw.len) ? __ldg(a.block_table + static_cast<long long>(pw.b) * a.bt_stride + j) : -1;
      }
      const int blk = __shfl_sync(0xffffffffu, bid_reg, blk_i - bid_base);
      const bool ok = blk >= 0 && blk < a.num_blocks;
      if (lane == 0) {
        const uint32_t bar = bars + 8 * stage;
        if (ok) {
          const uint8_t* src = a.cache + ((static_cast<long long>(blk) * a.n_kv + pw.h) * a.tiles_per_block +
                                          (pw.t & (a.tiles_per_block - 1))) *
                                             static_cast<long long>(a.tile_bytes);
          fence_proxy_async();
          mbar_expect(bar, a.tile_bytes);
          bulk_g2s(ring + stage * a.tile_stride, src, a.tile_bytes, bar, policy);
        } else {
          mbar_expect(bar, 0);   // completes the phase with no data
        }
      }
      tile_ok_bits = ok ? (tile_ok_bits | (1u << stage)) : (tile_ok_bits & ~(1u << stage));
      ++pi;
      if (pi >= r1 || !walk_next(pw, a, lane)) p_done = true;
    }

    // ---------------- consumer
    const long long seg = segment_of(cw, a);
    if (seg != c_seg) {
      if (c_seg >= 0) {
        // ---- finalize the previous segment: combine hi/lo columns, add
        // sum p * zero, normalise, write its record
        float l = lsum, z = zsum;
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        z += __shfl_xor_sync(0xffffffffu, z, 1);
        z += __shfl_xor_sync(0xffffffffu, z, 2);
        const long long rec = c_seg + wid;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int n = 2 * c + e;            // this lane's column = query head n
          const int pc = n + G;               // its lo column when G <= 4
          const int src = 4 * g + ((pc >> 1) & 3);
          const int hh = n < G ? n : 0;
          const float lh = __shfl_sync(0xffffffffu, l, 4 * hh);
          const float zh = __shfl_sync(0xffffffffu, z, 4 * hh);
          const float mh = __shfl_sync(0xffffffffu, mrow, 4 * hh);
          const float inv = lh > 0.f ? 1.f / lh : 0.f;
          float* dst = a.rec_o + (rec * G + hh) * kD + 16 * g;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            float v0 = o[mt][e], v1 = o[mt][2 + e];
            if (!GBIG) {
              const float p0 = __shfl_sync(0xffffffffu, o[mt][0], src);
              const float p1 = __shfl_sync(0xffffffffu, o[mt][1], src);
              const float p2 = __shfl_sync(0xffffffffu, o[mt][2], src);
              const float p3 = __shfl_sync(0xffffffffu, o[mt][3], src);
              v0 += (pc & 1) ? p1 : p0;
              v1 += (pc & 1) ? p3 : p2;
            }
            if (n < G) *reinterpret_cast<float2*>(dst + 2 * mt) = make_float2((v0 + zh) * inv, (v1 + zh) * inv);
          }
          if (n < G && g == 0) a.rec_lse[rec * G + n] = lh > 0.f ? mh + __log2f(lh) : -INFINITY;
        }
      }
      // ---- begin the new segment: wait for its query rows, rotate, split
      c_qslot ^= 1;
      const unsigned uses = c_qslot ? q_uses1 : q_uses0;
      if (!mbar_wait(bars + 8 * (kStages + c_qslot), uses & 1)) { aborted = true; break; }
      if (c_qslot) ++q_uses1; else ++q_uses0;
      uint32_t hp[8][4];   // [head][hi01, lo01, hi23, lo23] of this lane's 4 coordinates
#pragma unroll
      for (int gg = 0; gg < 8; ++gg) {
        hp[gg][0] = hp[gg][1] = hp[gg][2] = hp[gg][3] = 0u;
        if (gg < G) {
          float x[4];
          u2_to_f4<TQ>(lds64(qbuf + c_qslot * kQBufBytes + gg * kD * 2 + 8 * lane), x);
          float sc = a.qscale;
          if constexpr (KMODE != kFp8) {
            fwht128(x, lane);
            sc *= 0.088388347648318440f;   // 1 / sqrt(128)
          }
          split_half2(x[0] * sc, x[1] * sc, hp[gg][0], hp[gg][1]);
          split_half2(x[2] * sc, x[3] * sc, hp[gg][2], hp[gg][3]);
        }
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) qa[i] = 0u;
#pragma unroll
      for (int gg = 0; gg < 8; ++gg) {
        if (gg < G) {
          if constexpr (KMODE == kFp8) {
#pragma unroll
            for (int s = 0; s < 8; ++s) {   // coordinates 32 c + 4 s .. +3 live in lane 8 c + s
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint32_t v = __shfl_sync(0xffffffffu, hp[gg][k], 8 * c + s);
                if (g == gg) qa[4 * s + k] = v;
              }
            }
          } else {
#pragma unroll
            for (int s = 0; s < 16; ++s) {  // coordinates 32 c + 2 s, +1 live in lane 8 c + s / 2
              const int sl = 8 * c + (s >> 1);
              const uint32_t vh = __shfl_sync(0xffffffffu, (s & 1) ? hp[gg][2] : hp[gg][0], sl);
              const uint32_t vl = __shfl_sync(0xffffffffu, (s & 1) ? hp[gg][3] : hp[gg][1], sl);
              if (g == gg) { qa[2 * s] = vh; qa[2 * s + 1] = vl; }
            }
          }
        }
      }
      __syncwarp();   // q buffer fully read before the producer may reuse it
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
      mrow = mc0 = mc1 = -INFINITY;
      lsum = zsum = 0.f;
      c_seg = seg;
    }

    const int stage = static_cast<int>(ci % kStages);
    if (!mbar_wait(bars + 8 * stage, static_cast<uint32_t>((ci / kStages) & 1))) { aborted = true; break; }
    const bool ok = (tile_ok_bits >> stage) & 1u;
    if (!ok) {
      if (lane == 0) flag(a.status, TQ_DEV_BLOCK_OUT_OF_RANGE);
      __syncwarp();
    } else {
      const uint32_t st = ring + stage * a.tile_stride;
      const int nvalid = min(kTileTokens, cw.len - (cw.t << 4));
      // ---- this lane's slice of the tile
      uint4 kq[KMODE == kFp8 ? 4 : 2];
      if constexpr (KMODE == kMse4) {
        kq[0] = lds128(st + a.k_off + g * 64 + 16 * c);
        kq[1] = lds128(st + a.k_off + (g + 8) * 64 + 16 * c);
      } else if constexpr (KMODE == kMse3) {
        const uint32_t ra = st + a.k_off + g * 48 + 12 * c, rb = st + a.k_off + (g + 8) * 48 + 12 * c;
        kq[0] = make_uint4(lds32(ra), lds32(ra + 4), lds32(ra + 8), 0u);
        kq[1] = make_uint4(lds32(rb), lds32(rb + 4), lds32(rb + 8), 0u);
      } else {
        kq[0] = lds128(st + a.k_off + g * 128 + 32 * c);
        kq[1] = lds128(st + a.k_off + g * 128 + 32 * c + 16);
        kq[2] = lds128(st + a.k_off + (g + 8) * 128 + 32 * c);
        kq[3] = lds128(st + a.k_off + (g + 8) * 128 + 32 * c + 16);
      }
      const uint4 va = lds128(st + a.v_off + c * 128 + 16 * g);
      const uint4 vb = lds128(st + a.v_off + (c + 4) * 128 + 16 * g);
      float2 n01 = make_float2(1.f, 1.f), n89 = make_float2(1.f, 1.f);
      if constexpr (KMODE != kFp8) {
        n01 = half2_bits_to_float2(lds32(st + a.knorm_off + 4 * c));
        n89 = half2_bits_to_float2(lds32(st + a.knorm_off + 16 + 4 * c));
      }
      const float2 s01 = half2_bits_to_float2(lds32(st + a.vscale_off + 4 * c));
      const float2 s89 = half2_bits_to_float2(lds32(st + a.vscale_off + 16 + 4 * c));
      const float2 z01 = half2_bits_to_float2(lds32(st + a.vzero_off + 4 * c));
      const float2 z89 = half2_bits_to_float2(lds32(st + a.vzero_off + 16 + 4 * c));
      __syncwarp();   // every lane has read the stage: the producer may refill it

      // ---- scores: tokens 2c, 2c+1 (n-tile 0) and 2c+8, 2c+9 (n-tile 1)
      float s0[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      float s1[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      qk_tile<KMODE>(s0, qa, &kq[0], lut_lane);
      qk_tile<KMODE>(s1, qa, &kq[KMODE == kFp8 ? 2 : 1], lut_lane);
      float sc[4];
      sc[0] = ((s0[0][0] + s0[1][0]) + (s0[0][2] + s0[1][2])) * n01.x;
      sc[1] = ((s0[0][1] + s0[1][1]) + (s0[0][3] + s0[1][3])) * n01.y;
      sc[2] = ((s1[0][0] + s1[1][0]) + (s1[0][2] + s1[1][2])) * n89.x;
      sc[3] = ((s1[0][1] + s1[1][1]) + (s1[0][3] + s1[1][3])) * n89.y;
      float vs[4] = {s01.x, s01.y, s89.x, s89.y};
      float vz[4] = {z01.x, z01.y, z89.x, z89.y};
      if (nvalid < kTileTokens) {   // ragged last tile of a sequence
        const int tk[4] = {2 * c, 2 * c + 1, 2 * c + 8, 2 * c + 9};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (tk[e] >= nvalid) { sc[e] = -INFINITY; vs[e] = 0.f; vz[e] = 0.f; }
      }
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
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float pe = ex2(sc[e] - mrow);   // exp2(-inf) = 0 for masked tokens
        lsum += pe;
        ps[e] = pe * vs[e];
        zsum = fmaf(pe, vz[e], zsum);
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
          const uint32_t wa = word_of(va, mt >> 1), wb = word_of(vb, mt >> 1);
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
          const uint32_t wa = word_of(va, mt >> 1), wb = word_of(vb, mt >> 1);
          const int j0 = 2 * (mt & 1);
          mma16816(o[mt], vpair(wa, j0), vpair(wa, j0 + 1), vpair(wb, j0), vpair(wb, j0 + 1), b0, b1);
        }
      }
    }
    ++ci;
    if (ci < r1) walk_next(cw, a, lane);
  }

  if (!aborted) {
    // ---- finalize the last segment
    float l = lsum, z = zsum;
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    z += __shfl_xor_sync(0xffffffffu, z, 1);
    z += __shfl_xor_sync(0xffffffffu, z, 2);
    const long long rec = c_seg + wid;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int n = 2 * c + e;
      const int pc = n + G;
      const int src = 4 * g + ((pc >> 1) & 3);
      const int hh = n < G ? n : 0;
      const float lh = __shfl_sync(0xffffffffu, l, 4 * hh);
      const float zh = __shfl_sync(0xffffffffu, z, 4 * hh);
      const float mh = __shfl_sync(0xffffffffu, mrow, 4 * hh);
      const float inv = lh > 0.f ? 1.f / lh : 0.f;
      float* dst = a.rec_o + (rec * G + hh) * kD + 16 * g;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        float v0 = o[mt][e], v1 = o[mt][2 + e];
        if (!GBIG) {
          const float p0 = __shfl_sync(0xffffffffu, o[mt][0], src);
          const float p1 = __shfl_sync(0xffffffffu, o[mt][1], src);
          const float p2 = __shfl_sync(0xffffffffu, o[mt][2], src);
          const float p3 = __shfl_sync(0xffffffffu, o[mt][3], src);
          v0 += (pc & 1) ? p1 : p0;
          v1 += (pc & 1) ? p3 : p2;
        }
        if (n < G) *reinterpret_cast<float2*>(dst + 2 * mt) = make_float2((v0 + zh) * inv, (v1 + zh) * inv);
      }
      if (n < G && g == 0) a.rec_lse[rec * G + n] = lh > 0.f ? mh + __log2f(lh) : -INFINITY;
    }
  } else {
    // a wait expired: flag it and drain this warp's own copies (bounded) so no
    // bulk copy still targets shared memory when the warp stops
    if (lane == 0) flag(a.status, TQ_DEV_TIMEOUT);
    for (long long i = ci; i < pi; ++i)
      mbar_wait(bars + 8 * static_cast<int>(i % kStages), static_cast<uint32_t>((i / kStages) & 1));
    if (q_iss0 > q_uses0) mbar_wait(bars + 8 * kStages, q_uses0 & 1);
    if (q_iss1 > q_uses1) mbar_wait(bars + 8 * (kStages + 1), q_uses1 & 1);
  }
}

// ---------------------------------------------------------------- reduce

template <typename TO>
__device__ __forceinline__ void store_out(void* out, long long i, float v) {
  if constexpr (std::is_same<TO, float>::value) static_cast<float*>(out)[i] = v;
  else if constexpr (std::is_same<TO, __half>::value) static_cast<__half*>(out)[i] = __float2half_rn(v);
  else static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
}

__device__ __forceinline__ int reduce_len(const ReduceArgs& a, int b) {
  return min(max(__ldg(a.seq_lens + b), 0), min(a.max_seq_len, a.cap));
}

// One CTA per (query head, sequence): merge the records of every
// (segment, warp) piece of this sequence's KV head.
template <typename TO>
__global__ void __launch_bounds__(kD) reduce_kernel(const ReduceArgs a) {
  __shared__ long long s_pre[2];
  const int hq = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
  const int h = hq / a.group, gg = hq - h * a.group;
  if (threadIdx.x < 32) {   // tiles before sequence b, and in total
    long long before = 0, total = 0;
    for (int b0 = 0; b0 < a.batch; b0 += 32) {
      const int j = b0 + threadIdx.x;
      long long nt = j < a.batch ? (reduce_len(a, j) + kTileTokens - 1) / kTileTokens : 0;
      long long nb = j < b ? nt : 0;
      for (int o = 1; o < 32; o <<= 1) {
        nt += __shfl_xor_sync(0xffffffffu, nt, o);
        nb += __shfl_xor_sync(0xffffffffu, nb, o);
      }
      total += nt;
      before += nb;
    }
    if (threadIdx.x == 0) { s_pre[0] = before * a.n_kv; s_pre[1] = total * a.n_kv; }
  }
  __syncthreads();
  const long long orow = static_cast<long long>(b) * a.n_q + hq;
  const int len = reduce_len(a, b);
  if (len <= 0) { store_out<TO>(a.out, orow * kD + d, 0.f); return; }
  const int nt = (len + kTileTokens - 1) / kTileTokens;
  const long long T = s_pre[1], nw = a.num_warps;
  const long long seq0 = s_pre[0] + static_cast<long long>(h) * nt;   // first tile of (b, h)
  const int ppt = a.part_tiles > 0 ? a.part_tiles : nt;
  const int parts = (nt + ppt - 1) / ppt;
  float mx = -INFINITY, acc = 0.f, den = 0.f;
  for (int pass = 0; pass < 2; ++pass) {
    for (int p = 0; p < parts; ++p) {
      const long long t0 = seq0 + static_cast<long long>(p) * ppt;
      const long long t1 = seq0 + min(static_cast<long long>(p + 1) * ppt, static_cast<long long>(nt));
      const long long seg = (static_cast<long long>(b) * a.n_kv + h) * a.num_parts + p;
      const long long wf = ((t0 + 1) * nw - 1) / T, wl = (t1 * nw - 1) / T;
      for (long long w = wf; w <= wl; ++w) {
        if (T * w / nw == T * (w + 1) / nw) continue;   // this warp owns no tile
        const long long rec = (seg + w) * a.group + gg;
        const float lse = a.rec_lse[rec];
        if (pass == 0) {
          mx = fmaxf(mx, lse);
        } else if (lse != -INFINITY) {
          const float wgt = exp2f(lse - mx);
          den += wgt;
          acc = fmaf(wgt, a.rec_o[rec * kD + d], acc);
        }
      }
    }
    if (pass == 0 && mx == -INFINITY) break;
  }
  store_out<TO>(a.out, orow * kD + d, den > 0.f ? acc / den : 0.f);
}

// ---------------------------------------------------------------- host glue

struct Plan {
  tq_layout L;
  int part_tiles, num_parts, cap, sms, num_warps;
  long long num_records;
  size_t need;
};

int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

// Host-side checks and sizes shared by both stages (no CUDA call before the
// argument checks pass; the SM count is queried last).
tq_status make_plan(const tq_config* cfg, int batch, int max_seq_len, int bt_stride, bool query_device,
                    Plan* P) {
  tq_status st = make_layout(cfg, &P->L);
  if (st != TQ_OK) return st;
  if (batch < 0 || max_seq_len < 0) return TQ_ERR_INVALID_ARG;
  if (cfg->num_q_heads <= 0 || cfg->num_q_heads % cfg->num_kv_heads) return TQ_ERR_INVALID_ARG;
  if (cfg->num_q_heads / cfg->num_kv_heads > 8) return TQ_ERR_UNSUPPORTED;
  const int pt = cfg->partition_tokens;
  if (pt < 0 || pt % kTileTokens || pt > (1 << 30)) return TQ_ERR_INVALID_ARG;
  P->part_tiles = pt / kTileTokens;
  P->num_parts = pt > 0 ? static_cast<int>((static_cast<long long>(max_seq_len) + pt - 1) / pt) : 1;
  if (P->num_parts < 1) P->num_parts = 1;
  P->cap = bt_stride * cfg->block_size;
  P->sms = query_device ? device_sms() : 0;
  if (P->sms > kMaxCtas) P->sms = kMaxCtas;
  P->num_warps = (P->sms > 0 ? P->sms : 1) * kWarps;
  const int G = cfg->num_q_heads / cfg->num_kv_heads;
  P->num_records = static_cast<long long>(batch) * cfg->num_kv_heads * P->num_parts +
                   static_cast<long long>(kMaxCtas) * kWarps;
  const long long floats = P->num_records * G * (kD + 1);
  P->need = static_cast<size_t>(((floats * 4 + 15) / 16) * 16);
  return TQ_OK;
}

int warp_buffer_bytes(int tile_bytes) {
  const int stride = (tile_bytes + 127) & ~127;
  return kStages * stride + 2 * kQBufBytes + 8 * (kStages + 2);
}

template <int KMODE, int GBIG, typename TQ>
cudaError_t launch_split_typed(DecodeArgs a, cudaStream_t s, int sms) {
  int dev = 0, optin = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  a.tile_stride = (a.tile_bytes + 127) & ~127;
  a.warp_bytes = warp_buffer_bytes(a.tile_bytes);
  const int want = kWarps * a.warp_bytes + static_cast<int>(2 * lut_bytes<KMODE>());
  a.dyn_bytes = want < optin ? want : optin;
  auto k = split_kernel<KMODE, GBIG, TQ>;
  cudaError_t err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, a.dyn_bytes);
  if (err != cudaSuccess) return err;
  k<<<static_cast<unsigned>(sms), kWarps * 32, static_cast<size_t>(a.dyn_bytes), s>>>(a);
  return cudaGetLastError();
}

template <int KMODE>
cudaError_t launch_split(const DecodeArgs& a, int q_dtype, cudaStream_t s, int sms) {
  if (q_dtype == TQ_DTYPE_BF16)
    return a.group > 4 ? launch_split_typed<KMODE, 1, __nv_bfloat16>(a, s, sms)
                       : launch_split_typed<KMODE, 0, __nv_bfloat16>(a, s, sms);
  return a.group > 4 ? launch_split_typed<KMODE, 1, __half>(a, s, sms)
                     : launch_split_typed<KMODE, 0, __half>(a, s, sms);
}

tq_status run_partials(const tq_config* cfg, const tq_codebook* cb, const void* q, int q_dtype,
                       const void* cache, long long num_blocks, const int* block_table, int bt_stride,
                       const int* seq_lens, int batch, int max_seq_len, float scale, void* workspace,
                       size_t ws_bytes, unsigned int* dev_status, cudaStream_t stream) {
  if (bt_stride < 1) return TQ_ERR_INVALID_ARG;
  Plan P;
  tq_status st = make_plan(cfg, batch, max_seq_len, bt_stride, false, &P);
  if (st != TQ_OK) return st;
  if (q_dtype != TQ_DTYPE_F16 && q_dtype != TQ_DTYPE_BF16) return TQ_ERR_INVALID_ARG;
  if (!P.L.key_fp8 && (!cb || cb->bits != P.L.key_bits || cb->head_dim != cfg->head_dim))
    return TQ_ERR_INVALID_ARG;
  if (ws_bytes < P.need) return TQ_ERR_WORKSPACE_TOO_SMALL;
  if (batch == 0) return TQ_OK;
  if (!q || !cache || !block_table || !seq_lens || !workspace) return TQ_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(cache) || !aligned16(workspace) ||
      (reinterpret_cast<unsigned long long>(block_table) & 3ull) ||
      (reinterpret_cast<unsigned long long>(seq_lens) & 3ull))
    return TQ_ERR_MISALIGNED;
  if (dev_status && (reinterpret_cast<unsigned long long>(dev_status) & 3ull)) return TQ_ERR_MISALIGNED;
  if (num_blocks < 0) return TQ_ERR_INVALID_ARG;
  make_plan(cfg, batch, max_seq_len, bt_stride, true, &P);
  if (P.sms <= 0) return TQ_ERR_CUDA;

  DecodeArgs a;
  a.cache = static_cast<const uint8_t*>(cache);
  a.num_blocks = num_blocks;
  a.q = q;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.status = dev_status;
  const int G = cfg->num_q_heads / cfg->num_kv_heads;
  a.rec_o = static_cast<float*>(workspace);
  a.rec_lse = a.rec_o + P.num_records * G * kD;
  a.batch = batch;
  a.n_q = cfg->num_q_heads;
  a.n_kv = cfg->num_kv_heads;
  a.group = G;
  a.block_size = cfg->block_size;
  a.log2_bs = __builtin_ctz(static_cast<unsigned>(cfg->block_size));
  a.tiles_per_block = cfg->block_size / kTileTokens;
  a.bt_stride = bt_stride;
  a.part_tiles = P.part_tiles;
  a.num_parts = P.num_parts;
  a.max_seq_len = max_seq_len;
  a.cap = P.cap;
  a.tile_bytes = P.L.tile_bytes;
  a.tile_stride = 0;
  a.k_off = P.L.k_off;
  a.v_off = P.L.v_off;
  a.knorm_off = P.L.knorm_off;
  a.vscale_off = P.L.vscale_off;
  a.vzero_off = P.L.vzero_off;
  a.warp_bytes = 0;
  a.dyn_bytes = 0;
  const float sm_scale = scale > 0.f ? scale : 0.088388347648318440f;   // 1/sqrt(128)
  a.qscale = sm_scale * 1.4426950408889634f;                              // log2(e)
  for (int i = 0; i < 16; ++i) a.cent[i] = (!P.L.key_fp8 && i < cb->num_levels) ? cb->centroids[i] : 0.f;

  cudaError_t err;
  if (P.L.key_fp8) err = launch_split<kFp8>(a, q_dtype, stream, P.sms);
  else if (P.L.key_bits == 4) err = launch_split<kMse4>(a, q_dtype, stream, P.sms);
  else err = launch_split<kMse3>(a, q_dtype, stream, P.sms);
  return err == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

tq_status run_reduce(const tq_config* cfg, const int* seq_lens, int batch, int max_seq_len, int bt_stride,
                     void* out, int out_dtype, const void* workspace, size_t ws_bytes, cudaStream_t stream) {
  if (bt_stride < 1) return TQ_ERR_INVALID_ARG;
  Plan P;
  tq_status st = make_plan(cfg, batch, max_seq_len, bt_stride, false, &P);
  if (st != TQ_OK) return st;
  if (out_dtype != TQ_DTYPE_F16 && out_dtype != TQ_DTYPE_BF16 && out_dtype != TQ_DTYPE_F32)
    return TQ_ERR_INVALID_ARG;
  if (ws_bytes < P.need) return TQ_ERR_WORKSPACE_TOO_SMALL;
  if (batch == 0) return TQ_OK;
  if (!seq_lens || !out || !workspace) return TQ_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(workspace)) return TQ_ERR_MISALIGNED;
  make_plan(cfg, batch, max_seq_len, bt_stride, true, &P);
  if (P.sms <= 0) return TQ_ERR_CUDA;
  ReduceArgs r;
  const int G = cfg->num_q_heads / cfg->num_kv_heads;
  r.seq_lens = seq_lens;
  r.rec_o = static_cast<const float*>(workspace);
  r.rec_lse = r.rec_o + P.num_records * G * kD;
  r.out = out;
  r.batch = batch;
  r.n_q = cfg->num_q_heads;
  r.n_kv = cfg->num_kv_heads;
  r.group = G;
  r.part_tiles = P.part_tiles;
  r.num_parts = P.num_parts;
  r.max_seq_len = max_seq_len;
  r.cap = P.cap;
  r.num_warps = P.num_warps;
  const dim3 grid(static_cast<unsigned>(cfg->num_q_heads), static_cast<unsigned>(batch));
  if (out_dtype == TQ_DTYPE_F32) reduce_kernel<float><<<grid, kD, 0, stream>>>(r);
  else if (out_dtype == TQ_DTYPE_F16) reduce_kernel<__half><<<grid, kD, 0, stream>>>(r);
  else reduce_kernel<__nv_bfloat16><<<grid, kD, 0, stream>>>(r);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // namespace
}  // namespace tq

extern "C" {

size_t tq_decode_workspace_size(const tq_config* cfg, int batch, int max_seq_len) {
  tq::Plan P;
  if (!cfg || tq::make_plan(cfg, batch, max_seq_len, 1, false, &P) != TQ_OK) return 0;
  return P.need;
}

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
