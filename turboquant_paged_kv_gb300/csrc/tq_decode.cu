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
//  Data movement. Each warp owns a ring of 2 stages in shared memory, each a
//  chunk of up to 4 consecutive tiles (64 positions) of one segment, fed by
//  cp.async.bulk (one 2144-byte copy per tile at 4bit_nc, all completing on the
//  stage's mbarrier), and two query buffers fed the same way; the ring runs
//  ahead across segment boundaries. Per-chunk work (waits, the softmax max,
//  the rescale vote) is amortised over 64 positions and the 4 tiles give the
//  tensor pipe 4 independent accumulation chains. Block ids are read 32 at a time into a lane-indexed
//  register window. Every mbarrier wait is bounded: on expiry the warp flags
//  TQ_DEV_TIMEOUT, drains its own copies (bounded again) and stops.
//
//  Math. Both contractions run on tensor cores with mma.sync.m16n8k16 (f16 in,
//  f32 accumulate; one such mma occupies a sub-partition's tensor pipe for
//  about 8 cycles on GB300, so the layout wastes as few rows as possible):
//    S[8 tok x 2 parts, 8] = K . Q^T. Rows g and 8 + g hold token g with the
//      centroid hi and lo parts (c = c_hi + c_lo in fp16); one 8-byte LUT entry
//      per key byte (32 copies, one per lane, so lookups never conflict; the
//      table is aligned so one PRMT forms the address) is exactly the (row g,
//      row 8 + g) operand pair, and the two rows are summed in the same lane.
//      Columns hold q_hi of the G <= 4 query heads and q_lo of the same heads
//      (q = q_hi + q_lo), so one mma per 16 coordinates covers all products to
//      ~2^-22 relative (fp16 operands alone miss the 2e-3 output gate). For
//      G > 4 the q_lo columns take a second mma.
//    P^T reaches the B-operand layout through movmatrix.trans (the S layout has
//      tokens in rows), one instruction per 8x8 block of fp16 hi or lo parts.
//    O^T[16 d x 8] = V^T[16 d x 16 tok] . P^T. The store interleaves the 16-bit
//      words of token pairs; masking a 32-bit word with 0x000F000F (or
//      0x00F000F0) yields a half2 of the two tokens' codes as exact fp16
//      subnormals (code * 2^-24, or code * 2^-20), so value operands cost one
//      LOP3 per pair; the per-row power of two is removed at the end. The
//      16-byte groups of the V region are XOR-swizzled by the pair index so
//      these loads are free of bank conflicts. Columns
//      carry hi and lo parts of p * scale; sum_p p * zero is kept on the side.
//  Softmax in log2 units with a lazy rescale: the running max of a head only
//  moves when it grows by more than 2^8, decided by a warp vote, so rescaling
//  the accumulators is off the common path.

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
#ifndef TQ_DECODE_WARPS
#define TQ_DECODE_WARPS 8
#endif
constexpr int kMaxWarps = TQ_DECODE_WARPS;   // warps per CTA (fewer when shared memory is short)
constexpr int kChunk = 4;               // tiles per ring stage (64 tokens)
constexpr int kStages = 2;              // ring stages per warp
constexpr float kTau = 8.0f;            // lazy rescale threshold, log2 units
constexpr uint32_t kWaitLimit = 1u << 16;
constexpr uint32_t kSuspendNs = 20000;  // try_wait suspend hint: bound ~ kWaitLimit * 20 us
constexpr int kMaxCtas = 256;           // grid cap; sizes the workspace without a device query
constexpr int kRecordWarps = 16;        // warps per CTA the workspace allows for (>= kMaxWarps)
static_assert(kMaxWarps <= kRecordWarps, "workspace sized for at most 16 warps per CTA");

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
  int tile_bytes, stage_bytes, k_off, v_off, knorm_off, vscale_off, vzero_off;
  int qbuf_bytes;      // G * d * 2
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
__device__ __forceinline__ float lds_h2f(uint32_t a) {   // one fp16 -> float
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];\n" : "=h"(v) : "r"(a));
  return __half2float(__ushort_as_half(v));
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
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendNs)
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

// Address of the LUT entry for k-step s (coordinates 32c + 2s, +1) of a key row
// slice held in kq (this lane's bytes / bits of the row).
template <int KMODE>
__device__ __forceinline__ uint32_t lut_addr(const uint4& kq, int s, uint32_t lut_lane) {
  if constexpr (KMODE == kMse4) {
    return __byte_perm(word_of(kq, s >> 2), lut_lane, 0x7604u | ((s & 3) << 4));
  } else {
    const int bit = 6 * s, wi = bit >> 5, sh = bit & 31;
    const uint32_t w0 = word_of(kq, wi);
    uint32_t f;
    if (sh <= 26) f = w0 >> sh;
    else f = __funnelshift_r(w0, word_of(kq, wi + 1), sh);
    return ((f << 8) & 0x3F00u) | lut_lane;
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

__device__ __forceinline__ int segment_of(const Walk& w, const DecodeArgs& a) {
  const int p = a.part_tiles > 0 ? w.t / a.part_tiles : 0;
  return (w.b * a.n_kv + w.h) * a.num_parts + p;
}

// ---------------------------------------------------------------- split kernel

// One consumer step handles a chunk of up to kChunk consecutive tiles of one
// segment, held in one ring stage.
template <int KMODE, int GBIG, typename TQ>
__global__ void __launch_bounds__(kMaxWarps * 32, 1)
split_kernel(const DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t s_dyn[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarp_cta = blockDim.x >> 5;
  const int g = lane >> 2;          // mma groupID
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

  const uint32_t ring = my_base;                                  // kStages chunks
  const uint32_t qbuf = ring + kStages * a.stage_bytes;           // 2 query buffers
  const uint32_t bars = qbuf + 2 * a.qbuf_bytes;                  // kStages + 2 mbarriers
  if (lane == 0) {
    for (int i = 0; i < kStages + 2; ++i) mbar_init(bars + 8 * i, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();   // LUT built, barriers initialised

  uint32_t lut_lane = 0;
  if constexpr (kLut != 0) lut_lane = lut + 8u * lane;
  const uint64_t policy = evict_first_policy();

  // ---- this warp's range of the tile line
  const long long nwarps = static_cast<long long>(gridDim.x) * nwarp_cta;
  const int wid = blockIdx.x * nwarp_cta + warp;
  long long total = 0;   // n_kv * sum_b ceil(len_b / 16)
  bool too_long = false;
  for (int b0 = 0; b0 < a.batch; b0 += 32) {
    const int j = b0 + lane;
    int nt = 0;
    if (j < a.batch) {
      const int raw = __ldg(a.seq_lens + j);
      too_long |= raw > min(a.max_seq_len, a.cap);
      nt = (clamp_len(a, raw) + kTileTokens - 1) / kTileTokens;
    }
    for (int o_ = 1; o_ < 32; o_ <<= 1) nt += __shfl_xor_sync(0xffffffffu, nt, o_);
    total += nt;
  }
  if (wid == 0 && __any_sync(0xffffffffu, too_long) && lane == 0) flag(a.status, TQ_DEV_SEQ_TOO_LONG);
  total *= a.n_kv;
  const long long r0 = total * wid / nwarps;
  const int ntiles = static_cast<int>(total * (wid + 1) / nwarps - r0);
  if (ntiles <= 0) return;

  Walk pw;   // producer cursor: locate tile r0
  {
    long long acc = 0;
    int b = 0;
    lens_fill(pw, a, 0, lane);
    for (;;) {
      const int len = lens_get(pw, a, b, lane);
      const int nt = (len + kTileTokens - 1) / kTileTokens;
      const long long span = static_cast<long long>(nt) * a.n_kv;
      if (r0 < acc + span) {
        const int off = static_cast<int>(r0 - acc);
        pw.b = b; pw.len = len; pw.nt = nt;
        pw.h = off / nt;
        pw.t = off - pw.h * nt;
        break;
      }
      acc += span;
      ++b;
    }
  }
  Walk cw = pw;   // consumer cursor

  int bid_b = -1, bid_base = 0, bid_reg = 0;   // producer block-id window
  int pi = 0, ci = 0;                           // tiles issued / consumed (relative to r0)
  int p_stage = 0, c_stage = 0;
  uint32_t c_phase = 0;                         // parity bit per stage, consumer side
  uint32_t ok_bits = 0;                         // per stage, kChunk bits: tile copied
  uint32_t stage_busy = 0;                      // per stage: issued, not yet consumed
  int p_seg = -1, c_seg = -1;
  int p_qslot = 1, c_qslot = 1;
  uint32_t q_phase = 0, q_pending = 0;
  bool p_done = false, aborted = false;

  uint32_t qb[GBIG ? 32 : 16];     // Q^T B operands (per k-step; GBIG: hi then lo)
  float o[8][4];                   // O^T accumulators, rows d, cols n = 2c, 2c+1
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f, z0 = 0.f, z1 = 0.f;

  auto finalize = [&](int seg) {
    float l_[2] = {l0, l1}, z_[2] = {z0, z1};
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
      for (int o_ = 4; o_ < 32; o_ <<= 1) {
        l_[e] += __shfl_xor_sync(0xffffffffu, l_[e], o_);
        z_[e] += __shfl_xor_sync(0xffffffffu, z_[e], o_);
      }
    const float mm[2] = {m0, m1};
    const int rec = seg + wid;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int n = 2 * c + e;
      const int pc = n + G;                      // lo column of head n (G <= 4)
      const int src = 4 * g + ((pc >> 1) & 3);
      const float inv = l_[e] > 0.f ? 1.f / l_[e] : 0.f;
      float* dst = a.rec_o + (static_cast<long long>(rec) * G + (n < G ? n : 0)) * kD + 16 * g;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        float v0 = o[mt][e], v1 = o[mt][2 + e];
        if (!GBIG) {
          v0 += __shfl_sync(0xffffffffu, o[mt][pc & 1], src);
          v1 += __shfl_sync(0xffffffffu, o[mt][2 + (pc & 1)], src);
        }
        // value operands carried code * 2^-24 (rows g) and code * 2^-20 (rows g + 8)
        if (n < G)
          *reinterpret_cast<float2*>(dst + 2 * mt) =
              make_float2(fmaf(v0, 16777216.f, z_[e]) * inv, fmaf(v1, 1048576.f, z_[e]) * inv);
      }
      if (n < G && g == 0)
        a.rec_lse[static_cast<long long>(rec) * G + n] = l_[e] > 0.f ? mm[e] + __log2f(l_[e]) : -INFINITY;
    }
  };

  while (ci < ntiles) {
    // ---------------- producer: fill free stages with chunks. A chunk is up
    // to kChunk tiles of one segment; a new segment needs a free query buffer
    // (the consumer must have begun the one before it).
    while (!p_done && !((stage_busy >> p_stage) & 1u)) {
      const int seg = segment_of(pw, a);
      if (seg != p_seg) {
        if (p_seg >= 0 && c_seg < p_seg) break;
        p_qslot ^= 1;
        q_pending |= 1u << p_qslot;
        if (lane == 0) {
          const uint32_t bar = bars + 8 * (kStages + p_qslot);
          const uint8_t* src = static_cast<const uint8_t*>(a.q) +
                               (static_cast<long long>(pw.b) * a.n_q + pw.h * G) * (kD * 2);
          fence_proxy_async();
          mbar_expect(bar, a.qbuf_bytes);
          bulk_g2s_plain(qbuf + p_qslot * a.qbuf_bytes, src, a.qbuf_bytes, bar);
        }
        p_seg = seg;
      }
      const uint32_t bar = bars + 8 * p_stage;
      if (lane == 0) fence_proxy_async();
      uint32_t okm = 0;
      int n = 0;
      for (;;) {
        const int blk_i = (pw.t << 4) >> a.log2_bs;   // block index within the sequence
        if (pw.b != bid_b || blk_i - bid_base >= 32 || blk_i < bid_base) {
          bid_b = pw.b;
          bid_base = blk_i;
          const int j = bid_base + lane;
          bid_reg = (j * a.block_size < pw.len) ? __ldg(a.block_table + static_cast<long long>(pw.b) * a.bt_stride + j) : -1;
        }
        const int blk = __shfl_sync(0xffffffffu, bid_reg, blk_i - bid_base);
        if (blk >= 0 && blk < a.num_blocks) {
          okm |= 1u << n;
          if (lane == 0) {
            const uint8_t* src = a.cache + ((static_cast<long long>(blk) * a.n_kv + pw.h) * a.tiles_per_block +
                                            (pw.t & (a.tiles_per_block - 1))) *
                                               static_cast<long long>(a.tile_bytes);
            mbar_expect_tx(bar, a.tile_bytes);
            bulk_g2s(ring + p_stage * a.stage_bytes + n * a.tile_bytes, src, a.tile_bytes, bar, policy);
          }
        }
        ++n;
        ++pi;
        if (pi >= ntiles || !walk_next(pw, a, lane)) { p_done = true; break; }
        if (n == kChunk || segment_of(pw, a) != seg) break;
      }
      if (lane == 0) mbar_arrive(bar);
      ok_bits = (ok_bits & ~(((1u << kChunk) - 1) << (kChunk * p_stage))) | (okm << (kChunk * p_stage));
      stage_busy |= 1u << p_stage;
      p_stage = p_stage + 1 == kStages ? 0 : p_stage + 1;
    }

    // ---------------- consumer
    const int seg = segment_of(cw, a);
    if (seg != c_seg) {
      if (c_seg >= 0) finalize(c_seg);
      // ---- begin the segment: its query rows, rotated, scaled, split hi/lo
      c_qslot ^= 1;
      if (!mbar_wait(bars + 8 * (kStages + c_qslot), (q_phase >> c_qslot) & 1u)) { aborted = true; break; }
      q_phase ^= 1u << c_qslot;
      q_pending &= ~(1u << c_qslot);
#pragma unroll
      for (int i = 0; i < (GBIG ? 32 : 16); ++i) qb[i] = 0u;
#pragma unroll
      for (int gg = 0; gg < 8; ++gg) {
        if (gg < G) {
          float x[4];
          u2_to_f4<TQ>(lds64(qbuf + c_qslot * a.qbuf_bytes + gg * kD * 2 + 8 * lane), x);
          float sc = a.qscale;
          if constexpr (KMODE != kFp8) {
            fwht128(x, lane);
            sc *= 0.088388347648318440f;   // 1 / sqrt(128)
          }
          uint32_t hp[4];   // hi01, lo01, hi23, lo23 of coordinates 4 lane .. +3
          split_half2(x[0] * sc, x[1] * sc, hp[0], hp[1]);
          split_half2(x[2] * sc, x[3] * sc, hp[2], hp[3]);
          // B column g takes head gg's hi part (g == gg) or lo part (g == gg + G)
          const bool take_hi = g == gg, take_lo = GBIG ? (g == gg) : (g == gg + G);
          if constexpr (KMODE == kFp8) {
#pragma unroll
            for (int s = 0; s < 8; ++s) {   // coordinates 32c + 4s .. +3 live in lane 8c + s
              const uint32_t h01 = __shfl_sync(0xffffffffu, hp[0], 8 * c + s);
              const uint32_t l01 = __shfl_sync(0xffffffffu, hp[1], 8 * c + s);
              const uint32_t h23 = __shfl_sync(0xffffffffu, hp[2], 8 * c + s);
              const uint32_t l23 = __shfl_sync(0xffffffffu, hp[3], 8 * c + s);
              if (GBIG) {
                if (take_hi) { qb[2 * s] = h01; qb[2 * s + 1] = h23; qb[16 + 2 * s] = l01; qb[16 + 2 * s + 1] = l23; }
              } else {
                if (take_hi) { qb[2 * s] = h01; qb[2 * s + 1] = h23; }
                if (take_lo) { qb[2 * s] = l01; qb[2 * s + 1] = l23; }
              }
            }
          } else {
#pragma unroll
            for (int s = 0; s < 8; ++s) {   // coordinates 32c + 4s .. +3 live in lane 8c + s
              const uint32_t h01 = __shfl_sync(0xffffffffu, hp[0], 8 * c + s);
              const uint32_t l01 = __shfl_sync(0xffffffffu, hp[1], 8 * c + s);
              const uint32_t h23 = __shfl_sync(0xffffffffu, hp[2], 8 * c + s);
              const uint32_t l23 = __shfl_sync(0xffffffffu, hp[3], 8 * c + s);
              if (GBIG) {
                if (take_hi) { qb[2 * s] = h01; qb[2 * s + 1] = h23; qb[16 + 2 * s] = l01; qb[16 + 2 * s + 1] = l23; }
              } else {
                if (take_hi) { qb[2 * s] = h01; qb[2 * s + 1] = h23; }
                if (take_lo) { qb[2 * s] = l01; qb[2 * s + 1] = l23; }
              }
            }
          }
        }
      }
      __syncwarp();   // query buffer fully read before the producer may reuse it
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
      m0 = m1 = -INFINITY;
      l0 = l1 = z0 = z1 = 0.f;
      c_seg = seg;
    }

    // chunk of this stage: n tiles from cw (same rule as the producer)
    int n = 1;
    {
      Walk t = cw;
      while (n < kChunk && ci + n < ntiles && walk_next(t, a, lane) && segment_of(t, a) == seg) ++n;
    }
    if (!mbar_wait(bars + 8 * c_stage, (c_phase >> c_stage) & 1u)) { aborted = true; break; }
    c_phase ^= 1u << c_stage;
    const uint32_t okm = (ok_bits >> (kChunk * c_stage)) & ((1u << kChunk) - 1);
    if (okm != (1u << n) - 1 && lane == 0) flag(a.status, TQ_DEV_BLOCK_OUT_OF_RANGE);
    const uint32_t st = ring + c_stage * a.stage_bytes;
    const int tok0 = cw.t << 4;   // first position of the chunk in its sequence

    // ---- S[i] = K_i . Q^T for the chunk's tiles (missing tiles compute on
    // stale bytes and are masked below)
    float S[kChunk][4];
#pragma unroll
    for (int i = 0; i < kChunk; ++i) S[i][0] = S[i][1] = S[i][2] = S[i][3] = 0.f;
    if constexpr (KMODE == kFp8) {
#pragma unroll
      for (int i = 0; i < kChunk; ++i) {
        const uint32_t kt = st + i * a.tile_bytes + a.k_off;
        const uint4 kg0 = lds128(kt + g * 128 + 32 * c), kg1 = lds128(kt + g * 128 + 32 * c + 16);
        const uint4 kh0 = lds128(kt + (g + 8) * 128 + 32 * c), kh1 = lds128(kt + (g + 8) * 128 + 32 * c + 16);
#pragma unroll
        for (int s = 0; s < 8; ++s) {   // coordinates 32c + 4s .. +3
          const uint32_t wg = word_of(s < 4 ? kg0 : kg1, s & 3), wh = word_of(s < 4 ? kh0 : kh1, s & 3);
          const __half2_raw g01 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(wg & 0xFFFFu), __NV_E4M3);
          const __half2_raw g23 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(wg >> 16), __NV_E4M3);
          const __half2_raw h01 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(wh & 0xFFFFu), __NV_E4M3);
          const __half2_raw h23 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(wh >> 16), __NV_E4M3);
          const uint32_t a0 = static_cast<uint32_t>(g01.x) | (static_cast<uint32_t>(g01.y) << 16);
          const uint32_t a1 = static_cast<uint32_t>(h01.x) | (static_cast<uint32_t>(h01.y) << 16);
          const uint32_t a2 = static_cast<uint32_t>(g23.x) | (static_cast<uint32_t>(g23.y) << 16);
          const uint32_t a3 = static_cast<uint32_t>(h23.x) | (static_cast<uint32_t>(h23.y) << 16);
          mma16816(S[i], a0, a1, a2, a3, qb[2 * s], qb[2 * s + 1]);
          if (GBIG) mma16816(S[i], a0, a1, a2, a3, qb[16 + 2 * s], qb[16 + 2 * s + 1]);
        }
      }
    } else {
      uint4 kg[kChunk], kh[kChunk];   // this lane's key slice of tokens g and g+8
#pragma unroll
      for (int i = 0; i < kChunk; ++i) {
        const uint32_t kt = st + i * a.tile_bytes + a.k_off;
        if constexpr (KMODE == kMse4) {
          kg[i] = lds128(kt + g * 64 + 16 * c);
          kh[i] = lds128(kt + (g + 8) * 64 + 16 * c);
        } else {
          const uint32_t ra = kt + g * 48 + 12 * c, rb = kt + (g + 8) * 48 + 12 * c;
          kg[i] = make_uint4(lds32(ra), lds32(ra + 4), lds32(ra + 8), 0u);
          kh[i] = make_uint4(lds32(rb), lds32(rb + 4), lds32(rb + 8), 0u);
        }
      }
      // M rows: 8 tokens x {centroid hi part, centroid lo part}; k-step s holds
      // this lane's coordinates 32c + 4s .. +3 (two key bytes = two LUT entries,
      // each entry = the (hi, lo) operand pair of one row pair)
      float Sl[kChunk][2][4];
#pragma unroll
      for (int i = 0; i < kChunk; ++i)
#pragma unroll
        for (int u = 0; u < 2; ++u) Sl[i][u][0] = Sl[i][u][1] = Sl[i][u][2] = Sl[i][u][3] = 0.f;
#pragma unroll
      for (int s2 = 0; s2 < 8; ++s2) {
#pragma unroll
        for (int i = 0; i < kChunk; ++i) {
          const uint2 g0 = lds64(lut_addr<KMODE>(kg[i], 2 * s2, lut_lane));
          const uint2 g1 = lds64(lut_addr<KMODE>(kg[i], 2 * s2 + 1, lut_lane));
          const uint2 h0 = lds64(lut_addr<KMODE>(kh[i], 2 * s2, lut_lane));
          const uint2 h1 = lds64(lut_addr<KMODE>(kh[i], 2 * s2 + 1, lut_lane));
          mma16816(Sl[i][0], g0.x, g0.y, g1.x, g1.y, qb[2 * s2], qb[2 * s2 + 1]);
          mma16816(Sl[i][1], h0.x, h0.y, h1.x, h1.y, qb[2 * s2], qb[2 * s2 + 1]);
          if (GBIG) {
            mma16816(Sl[i][0], g0.x, g0.y, g1.x, g1.y, qb[16 + 2 * s2], qb[16 + 2 * s2 + 1]);
            mma16816(Sl[i][1], h0.x, h0.y, h1.x, h1.y, qb[16 + 2 * s2], qb[16 + 2 * s2 + 1]);
          }
        }
      }
      // rows g (hi part) + g + 8 (lo part) of each token: same lane
#pragma unroll
      for (int i = 0; i < kChunk; ++i) {
        S[i][0] = Sl[i][0][0] + Sl[i][0][2];
        S[i][1] = Sl[i][0][1] + Sl[i][0][3];
        S[i][2] = Sl[i][1][0] + Sl[i][1][2];
        S[i][3] = Sl[i][1][1] + Sl[i][1][3];
      }
    }

    // ---- scores: combine q_lo columns, norms, masks; per-head chunk max
    // S[i]: [0] tok g col 2c, [1] tok g col 2c+1, [2] tok g+8 col 2c, [3] tok g+8 col 2c+1
    float sv[kChunk][2], sz[kChunk][2];   // value scale / zero of tokens g, g+8
    float cm0 = -INFINITY, cm1 = -INFINITY;
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      const uint32_t tb = st + i * a.tile_bytes;
      float* v = S[i];
      if (!GBIG) {   // add the q_lo column of each head (column + G)
        const int srcA = 4 * g + (((2 * c + G) >> 1) & 3), srcB = 4 * g + (((2 * c + 1 + G) >> 1) & 3);
        const bool odd = G & 1;
        const float t0 = __shfl_sync(0xffffffffu, odd ? v[1] : v[0], srcA);
        const float t2 = __shfl_sync(0xffffffffu, odd ? v[3] : v[2], srcA);
        const float t1 = __shfl_sync(0xffffffffu, odd ? v[0] : v[1], srcB);
        const float t3 = __shfl_sync(0xffffffffu, odd ? v[2] : v[3], srcB);
        v[0] += t0; v[1] += t1; v[2] += t2; v[3] += t3;
      }
      if constexpr (KMODE != kFp8) {
        const float ng = lds_h2f(tb + a.knorm_off + 2 * g), nh = lds_h2f(tb + a.knorm_off + 2 * g + 16);
        v[0] *= ng; v[1] *= ng; v[2] *= nh; v[3] *= nh;
      }
      sv[i][0] = lds_h2f(tb + a.vscale_off + 2 * g);
      sv[i][1] = lds_h2f(tb + a.vscale_off + 2 * g + 16);
      sz[i][0] = lds_h2f(tb + a.vzero_off + 2 * g);
      sz[i][1] = lds_h2f(tb + a.vzero_off + 2 * g + 16);
      const int nvalid = ((okm >> i) & 1u) ? min(kTileTokens, cw.len - tok0 - 16 * i) : 0;
      if (nvalid < kTileTokens) {   // missing or ragged tile
        if (g >= nvalid) { v[0] = v[1] = -INFINITY; sv[i][0] = 0.f; sz[i][0] = 0.f; }
        if (g + 8 >= nvalid) { v[2] = v[3] = -INFINITY; sv[i][1] = 0.f; sz[i][1] = 0.f; }
      }
      cm0 = fmaxf(cm0, fmaxf(v[0], v[2]));
      cm1 = fmaxf(cm1, fmaxf(v[1], v[3]));
    }
#pragma unroll
    for (int o_ = 4; o_ < 32; o_ <<= 1) {
      cm0 = fmaxf(cm0, __shfl_xor_sync(0xffffffffu, cm0, o_));
      cm1 = fmaxf(cm1, __shfl_xor_sync(0xffffffffu, cm1, o_));
    }
    const bool need = (2 * c < G && cm0 > m0 + kTau) || (2 * c + 1 < G && cm1 > m1 + kTau);
    if (__any_sync(0xffffffffu, need)) {   // rare: move the running max, rescale
      float al0 = 1.f, al1 = 1.f;
      if (cm0 > m0 + kTau) { al0 = ex2(m0 - cm0); m0 = cm0; }
      if (cm1 > m1 + kTau) { al1 = ex2(m1 - cm1); m1 = cm1; }
      l0 *= al0; z0 *= al0; l1 *= al1; z1 *= al1;
#pragma unroll
      for (int e = 0; e < 2; ++e) {   // O^T column 2c + e belongs to head hn
        const int nn = 2 * c + e;
        const int hn = GBIG ? nn : (nn < G ? nn : (nn < 2 * G ? nn - G : 0));
        const float x0 = __shfl_sync(0xffffffffu, al0, 4 * g + (hn >> 1));
        const float x1 = __shfl_sync(0xffffffffu, al1, 4 * g + (hn >> 1));
        const float al = (hn & 1) ? x1 : x0;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) { o[mt][e] *= al; o[mt][2 + e] *= al; }
      }
    }

    // ---- per tile: probabilities, P^T operands (movmatrix), O^T += V^T . P^T
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      const float* v = S[i];
      // fmaxf also maps the NaN of (-inf) - (-inf) (a fully masked chunk before
      // any valid position) to an argument whose exp2 is 0
      const float p0 = ex2(fmaxf(v[0] - m0, -200.f)), p1 = ex2(fmaxf(v[1] - m1, -200.f));
      const float p2 = ex2(fmaxf(v[2] - m0, -200.f)), p3 = ex2(fmaxf(v[3] - m1, -200.f));
      l0 += p0 + p2;
      l1 += p1 + p3;
      z0 = fmaf(p0, sz[i][0], fmaf(p2, sz[i][1], z0));
      z1 = fmaf(p1, sz[i][0], fmaf(p3, sz[i][1], z1));
      uint32_t hg, lg, hh, lh;   // hi/lo half2 of (col 2c, col 2c+1) for tokens g and g+8
      split_half2(p0 * sv[i][0], p1 * sv[i][0], hg, lg);
      split_half2(p2 * sv[i][1], p3 * sv[i][1], hh, lh);
      uint32_t mg, mh, mgl = 0u, mhl = 0u;   // P matrices [token][column] in mma layout
      if (GBIG) {
        const uint32_t keep = (2 * c + 1 < G) ? 0xFFFFFFFFu : ((2 * c < G) ? 0x0000FFFFu : 0u);
        mg = hg & keep; mh = hh & keep; mgl = lg & keep; mhl = lh & keep;
      } else {
        // column n < G: hi of head n (own); G <= n < 2G: lo of head n - G
        uint32_t sel_g = 0u, sel_h = 0u;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int nn = 2 * c + e;
          const int hn = nn - G;
          const int src = 4 * g + ((hn >> 1) & 3);
          const uint32_t wg = __shfl_sync(0xffffffffu, lg, src);
          const uint32_t wh = __shfl_sync(0xffffffffu, lh, src);
          uint32_t xg, xh;
          if (nn < G) {
            xg = e ? (hg >> 16) : (hg & 0xFFFFu);
            xh = e ? (hh >> 16) : (hh & 0xFFFFu);
          } else if (nn < 2 * G) {
            xg = (hn & 1) ? (wg >> 16) : (wg & 0xFFFFu);
            xh = (hn & 1) ? (wh >> 16) : (wh & 0xFFFFu);
          } else {
            xg = xh = 0u;
          }
          sel_g |= xg << (16 * e);
          sel_h |= xh << (16 * e);
        }
        mg = sel_g;
        mh = sel_h;
      }
      const uint32_t b0 = movmatrix_trans(mg), b1 = movmatrix_trans(mh);
      const uint32_t tb = st + i * a.tile_bytes + a.v_off + 16 * (g ^ (2 * c));
      const uint4 va = lds128(tb + 128 * c);         // tokens 2c, 2c+1
      const uint4 vb = lds128(tb + 128 * (c + 4));   // tokens 2c+8, 2c+9
      uint32_t b0l = 0u, b1l = 0u;
      if (GBIG) { b0l = movmatrix_trans(mgl); b1l = movmatrix_trans(mhl); }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t wa = word_of(va, k), wb = word_of(vb, k);
        const uint32_t wa8 = wa >> 8, wb8 = wb >> 8;
        mma16816(o[2 * k], wa & 0x000F000Fu, wa & 0x00F000F0u, wb & 0x000F000Fu, wb & 0x00F000F0u, b0, b1);
        mma16816(o[2 * k + 1], wa8 & 0x000F000Fu, wa8 & 0x00F000F0u, wb8 & 0x000F000Fu, wb8 & 0x00F000F0u, b0, b1);
        if (GBIG) {
          mma16816(o[2 * k], wa & 0x000F000Fu, wa & 0x00F000F0u, wb & 0x000F000Fu, wb & 0x00F000F0u, b0l, b1l);
          mma16816(o[2 * k + 1], wa8 & 0x000F000Fu, wa8 & 0x00F000F0u, wb8 & 0x000F000Fu, wb8 & 0x00F000F0u, b0l,
                   b1l);
        }
      }
    }
    __syncwarp();   // every lane has read the stage: the producer may refill it
    stage_busy &= ~(1u << c_stage);
    c_stage = c_stage + 1 == kStages ? 0 : c_stage + 1;
    ci += n;
    for (int i = 0; i < n && ci < ntiles; ++i) walk_next(cw, a, lane);
  }

  if (!aborted) {
    finalize(c_seg);
  } else {
    // a wait expired: flag it and drain this warp's own copies (bounded) so no
    // bulk copy still targets shared memory when the warp stops
    if (lane == 0) flag(a.status, TQ_DEV_TIMEOUT);
    for (int s = 0; s < kStages; ++s)
      if ((stage_busy >> s) & 1u) mbar_wait(bars + 8 * s, (c_phase >> s) & 1u);
    for (int qs = 0; qs < 2; ++qs)
      if ((q_pending >> qs) & 1u) mbar_wait(bars + 8 * (kStages + qs), (q_phase >> qs) & 1u);
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
  int part_tiles, num_parts, cap, sms;
  long long num_records;
  size_t need;
};

int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

// Host-side checks and sizes shared by both stages (no CUDA call unless
// query_device; the workspace size never depends on the device).
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
  const int G = cfg->num_q_heads / cfg->num_kv_heads;
  P->num_records = static_cast<long long>(batch) * cfg->num_kv_heads * P->num_parts +
                   static_cast<long long>(kMaxCtas) * kRecordWarps;
  if (P->num_records > (1ll << 30)) return TQ_ERR_UNSUPPORTED;
  const long long floats = P->num_records * G * (kD + 1);
  P->need = static_cast<size_t>(((floats * 4 + 15) / 16) * 16);
  return TQ_OK;
}

struct LaunchShape {
  int warps;        // per CTA
  int warp_bytes;
  int stage_bytes;
  int dyn_bytes;
};

// Warps whose buffers fit around a LUT aligned to its size, for a dynamic
// shared-memory window starting at `start` (the plan the kernel computes).
int warps_that_fit(uint32_t start, uint32_t dyn, uint32_t lut, uint32_t wb) {
  const uint32_t lut_at = lut ? ((start + lut - 1) & ~(lut - 1)) : start + dyn;
  if (lut && lut_at + lut > start + dyn) return 0;
  int n = 0;
  uint32_t p = start;
  for (;;) {
    if (lut && p < lut_at + lut && p + wb > lut_at) p = lut_at + lut;
    if (p + wb > start + dyn) return n;
    p += wb;
    ++n;
  }
}

template <int KMODE>
bool launch_shape(int tile_bytes, int group, LaunchShape* s) {
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return false;
  s->stage_bytes = kChunk * tile_bytes;
  s->warp_bytes = kStages * s->stage_bytes + 2 * group * kD * 2 + 8 * (kStages + 2);
  s->warp_bytes = (s->warp_bytes + 15) & ~15;
  const uint32_t lut = lut_bytes<KMODE>();
  // the window may start at 0 or after a small reserved area; take the worse
  int warps = warps_that_fit(0, optin, lut, s->warp_bytes);
  const int w2 = warps_that_fit(1024, optin, lut, s->warp_bytes);
  if (w2 < warps) warps = w2;
  if (warps > kMaxWarps) warps = kMaxWarps;
  if (warps < 1) return false;
  s->warps = warps;
  s->dyn_bytes = optin;
  return true;
}

template <int KMODE, int GBIG, typename TQ>
cudaError_t launch_split_typed(DecodeArgs a, cudaStream_t s, int sms) {
  LaunchShape sh;
  if (!launch_shape<KMODE>(a.tile_bytes, a.group, &sh)) return cudaErrorInvalidConfiguration;
  a.stage_bytes = sh.stage_bytes;
  a.warp_bytes = sh.warp_bytes;
  a.dyn_bytes = sh.dyn_bytes;
  a.qbuf_bytes = a.group * kD * 2;
  auto k = split_kernel<KMODE, GBIG, TQ>;
  cudaError_t err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, a.dyn_bytes);
  if (err != cudaSuccess) return err;
  k<<<static_cast<unsigned>(sms), sh.warps * 32, static_cast<size_t>(a.dyn_bytes), s>>>(a);
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

int split_warps_per_cta(const tq_layout& L, int group) {
  LaunchShape sh;
  bool ok;
  if (L.key_fp8) ok = launch_shape<kFp8>(L.tile_bytes, group, &sh);
  else if (L.key_bits == 4) ok = launch_shape<kMse4>(L.tile_bytes, group, &sh);
  else ok = launch_shape<kMse3>(L.tile_bytes, group, &sh);
  return ok ? sh.warps : 0;
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
  a.stage_bytes = 0;
  a.k_off = P.L.k_off;
  a.v_off = P.L.v_off;
  a.knorm_off = P.L.knorm_off;
  a.vscale_off = P.L.vscale_off;
  a.vzero_off = P.L.vzero_off;
  a.qbuf_bytes = 0;
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
  const int G = cfg->num_q_heads / cfg->num_kv_heads;
  const int warps = split_warps_per_cta(P.L, G);
  if (warps <= 0) return TQ_ERR_CUDA;
  ReduceArgs r;
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
  r.num_warps = P.sms * warps;
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
