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
//  that is cut into equal contiguous ranges, one per consumer warp of a persistent grid
//  (stream-K). A warp's range crosses (b, h) "segments" (optionally also cut at
//  every partition_tokens positions); for every segment it touches the warp
//  writes one partial record (acc / l, lse for all G query heads) at index
//  segment + warp, which is unique because both sequences are monotone. Every
//  warp does the same amount of work whatever the sequence lengths are.
//
//  Data movement. One CTA per SM: two producer warps and up to 10 consumer
//  warps (3 warps per sub-partition); producer p feeds consumers p, p + 2, ...,
//  so each producer's pass issues the copies of half the consumers (one
//  producer serving all of them was the kernel's limit: each bulk copy issue
//  costs ~95 cycles and a pass served 11 lanes one after another). The lane of
//  a producer that feeds consumer j walks consumer j's range
//  chunk by chunk (a chunk is up to 2 consecutive tiles of one segment), loads
//  the next chunk's block ids while the current one is issued (read one pass
//  later, so the load latency overlaps other lanes' work), and fills consumer
//  j's ring of 3 stages: a 16-byte descriptor (segment, first position,
//  length, tile count, valid mask, last/new-segment bits) and the tiles by
//  cp.async.bulk (one 2144-byte copy per tile at 4bit_nc), completing on the
//  stage's "full" mbarrier. A chunk that opens a segment also brings the
//  segment's query rows into the consumer's query slot, once the consumer has
//  taken the previous rows ("q empty" mbarrier). Consumers only read
//  descriptors and compute, and release a stage through its "empty" mbarrier
//  as soon as they have read it (after QK and the score loads, with the value
//  words in registers), half a chunk before they are done with its math.
//  The producer starts as soon as the barriers exist; the consumers build the
//  LUT meanwhile. Every wait is bounded: a consumer whose wait expires flags
//  TQ_DEV_TIMEOUT and stops; the producer gives up after a long stretch
//  without progress and, in every case, waits (bounded) for all copies it
//  issued before it leaves.
//
//  Math. Both contractions run on tensor cores with mma.sync.m16n8k16 (f16 in,
//  f32 accumulate; one such mma occupies a sub-partition's tensor pipe for
//  about 8 cycles on GB300, so the layout wastes as few rows as possible):
//    S[16 tok, 8] = K . Q^T. Rows are the tile's 16 tokens. The centroids are
//      held as c' = fp16(gamma c), gamma a per-codebook scale in [1, 2) chosen
//      on the host so that no centroid rounds by more than ~1e-4 relative
//      (the query is divided by gamma). One 4-byte LUT entry per key byte
//      gives a half2 of its two centroids (32 copies, one per lane, so
//      lookups never conflict; the table is aligned so one PRMT forms the
//      address). The 2 tiles of a chunk run in lock step with two
//      accumulators each, so 4 accumulation chains interleave.
//      Columns 0..3 hold q_hi of the G <= 4 query heads and columns 4..7 q_lo of
//      the same heads (q = q_hi + q_lo), so one mma per 16 coordinates covers
//      the query to ~2^-22 relative, and lanes c, c ^ 2 of a quad hold the hi
//      and lo parts of the same heads: one exchange completes the score. For G > 4 the q_lo
//      columns take a second mma.
//    P^T reaches the B-operand layout through movmatrix.trans (the S layout has
//      tokens in rows), one instruction per 8x8 block of fp16 hi or lo parts.
//    O^T[16 d x 8] = V^T[16 d x 16 tok] . P^T. The store interleaves the 16-bit
//      words of token pairs; masking a 32-bit word with 0x000F000F (or
//      0x00F000F0) yields a half2 of the two tokens' codes as exact fp16
//      subnormals (code * 2^-24, or code * 2^-20), so value operands cost one
//      LOP3 per pair; the per-row power of two is removed at the end. The
//      16-byte groups of the V region are XOR-swizzled by the pair index so
//      these loads are free of bank conflicts. Columns carry the hi part of
//      p * scale (lanes c < 2) or its lo part (lanes c >= 2, G <= 4), so both
//      come out of one mma; sum_p p * zero is kept on the side.
//  Softmax in log2 units with a lazy rescale: the running max of a head only
//  moves when it grows by more than 2^8, decided by a warp vote, so rescaling
//  the accumulators is off the common path. The max starts at -1e30 (not
//  -inf), so masked positions give exp2(-inf) = 0 without a guard.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <climits>
#include <cmath>
#include <mutex>
#include <type_traits>

#include "tq_attn.cuh"
#include "tq_store.cuh"
#include "tq_internal.h"
#include "tq_launch.cuh"

namespace tq {
namespace {

constexpr int kD = 128;
#ifndef TQ_DECODE_WARPS
#define TQ_DECODE_WARPS 10
#endif
constexpr int kMaxConsumers = TQ_DECODE_WARPS;   // consumer warps per CTA (fewer when shared memory is short)
#ifndef TQ_PRODUCER_WARPS
#define TQ_PRODUCER_WARPS 2
#endif
constexpr int kProducers = TQ_PRODUCER_WARPS;   // producer warps; producer p feeds consumers p, p + kProducers, ...
#ifndef TQ_DECODE_CHUNK
#define TQ_DECODE_CHUNK 2
#endif
#ifndef TQ_DECODE_STAGES
#define TQ_DECODE_STAGES 3
#endif
#ifndef TQ_PRODUCER_SLEEP_NS
#define TQ_PRODUCER_SLEEP_NS 64
#endif
#ifndef TQ_PRODUCER_PASSES
#define TQ_PRODUCER_PASSES 1   // chunks a producer lane may issue per pass
#endif
constexpr int kChunk = TQ_DECODE_CHUNK;     // tiles per ring stage
constexpr int kStages = TQ_DECODE_STAGES;   // ring stages per consumer warp
constexpr float kTau = 8.0f;            // lazy rescale threshold, log2 units
constexpr int kMaxCtas = 256;           // grid cap; sizes the workspace without a device query
constexpr int kRecordWarps = 16;        // consumer warps per CTA the workspace allows for
static_assert(kMaxConsumers <= kRecordWarps, "workspace sized for at most 16 consumer warps per CTA");
static_assert(kMaxConsumers <= 32 * kProducers, "one producer lane per consumer warp");
static_assert(kMaxConsumers + kProducers <= 12, "12 warps keep 168 registers per thread");
// Shared-memory head: mbarriers (full and empty per (consumer, stage), then one
// "q empty" per consumer) from the start, the key codebook for the append
// path (16 midpoints, 16 centroids) in the last 128 bytes of the first
// kBarHead bytes, then one query slot of
// G * d * 2 bytes per consumer.
constexpr uint32_t kBarHead = 1024;
constexpr uint32_t kCodebookOff = kBarHead - 128;
static_assert((2 * kMaxConsumers * kStages + kMaxConsumers) * 8 <= static_cast<int>(kCodebookOff), "barrier area");
constexpr uint32_t kRawRowBytes = kD * 2;   // append: one raw key or value row (f16 / bf16)
static_assert(kStages >= 2 && kChunk >= 1 && kChunk <= 4, "ring shape");

// ---------------------------------------------------------------- ring plan

// Address of ring stage `idx` (consumer j's stage s is idx = j * kStages + s):
// stages are packed from `first` on and skip over the LUT, which sits at an
// address aligned to its own size.
__host__ __device__ __forceinline__ uint32_t stage_at(uint32_t first, uint32_t lut, uint32_t klut,
                                                      uint32_t sb, int idx) {
  if (klut) {
    const uint32_t nb = lut > first ? (lut - first) / sb : 0u;
    if (static_cast<uint32_t>(idx) >= nb) return lut + klut + (static_cast<uint32_t>(idx) - nb) * sb;
  }
  return first + static_cast<uint32_t>(idx) * sb;
}

__host__ __device__ __forceinline__ uint32_t lut_at(uint32_t base, uint32_t klut, uint32_t head) {
  return (base + head + klut - 1) & ~(klut - 1);
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};\n" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ int clamp_len(const DecodeArgs& a, int len) {
  return min(max(len, 0), min(a.max_seq_len, a.cap));
}

// Barriers: consumer j, stage s: full at bars + 16 * (j * kStages + s), empty 8 after.
__device__ __forceinline__ uint32_t full_bar(uint32_t bars, int j, int s) {
  return bars + 16u * static_cast<uint32_t>(j * kStages + s);
}
// Consumer j has taken the query rows of its latest segment.
__device__ __forceinline__ uint32_t q_empty_bar(uint32_t bars, int W, int j) {
  return bars + 8u * static_cast<uint32_t>(2 * W * kStages + j);
}

// ---------------------------------------------------------------- producer warp

// Position in the (b, h, t) tile line of one producer lane.
struct Cursor {
  int b, h, t, nt, len;
};

// Next tile; skips empty sequences. Call only while tiles remain after this one.
__device__ __forceinline__ void cursor_next(Cursor& u, const DecodeArgs& a) {
  if (++u.t < u.nt) return;
  u.t = 0;
  if (++u.h < a.n_kv) return;
  u.h = 0;
  do {
    ++u.b;
    u.len = clamp_len(a, ld_dep_s32(a.seq_lens + u.b));
    u.nt = (u.len + kTileTokens - 1) / kTileTokens;
  } while (u.nt == 0);
}

// Lane j < W feeds consumer warp j of this CTA: it walks that warp's range of
// the tile line chunk by chunk (a chunk is up to kChunk consecutive tiles of
// one segment) and, for each chunk, fills the next free ring stage with a
// 16-byte descriptor {segment, first position, sequence length, n | valid mask
// << 4 | last << 8 | new segment << 9} and the tiles (cp.async.bulk). A chunk
// that opens a segment also brings the segment's query rows into the
// consumer's query slot, once the consumer has taken the previous rows (its
// "q empty" barrier). A consumer whose range is empty gets one descriptor with
// n = 0 and the last bit. The block ids of the next chunk are loaded when the
// current one is issued, so their latency overlaps the wait for a free stage.
__device__ void producer_warp(const DecodeArgs& a, int W, int p, uint32_t bars, uint32_t qslots, uint32_t first,
                              uint32_t lut, uint32_t klut) {
  // Everything that may read what the previous kernel wrote comes after
  // grid_dep_wait(); with early_indices the lengths and block ids are not
  // among it, so the range, its location and the first plan come before.
  auto wait_previous = [&]() {
    grid_dep_wait();
    grid_dep_launch();
    asm volatile("bar.arrive 1, %0;\n" ::"r"(blockDim.x) : "memory");
  };
  if (!a.early_indices) wait_previous();
  const int lane = threadIdx.x & 31;
  const int jc = lane * kProducers + p;   // the consumer warp this lane feeds
  const bool mine = jc < W;
  const long long nw = static_cast<long long>(gridDim.x) * W;
  const long long wid = static_cast<long long>(blockIdx.x) * W + jc;

  // the block table is read block id by block id below: start it towards L2
  // now, spread over the grid (at most 16 MB of table)
  {
    const long long bt_bytes = min(static_cast<long long>(a.batch) * a.bt_stride * 4, 16ll << 20);
    const char* bt = reinterpret_cast<const char*>(a.block_table);
    for (long long off = (static_cast<long long>(blockIdx.x) * 32 + lane) * 128; off < bt_bytes;
         off += static_cast<long long>(gridDim.x) * 32 * 128)
      asm volatile("prefetch.global.L2 [%0];\n" ::"l"(bt + off));
  }

  // tiles of the whole line: n_kv * sum_b ceil(len_b / 16)
  long long total = 0;
  bool too_long = false;
  int len0 = 0;   // clamped length of sequence `lane` (first group)
  for (int b0 = 0; b0 < a.batch; b0 += 32) {
    const int j = b0 + lane;
    int nt = 0;
    if (j < a.batch) {
      const int raw = ld_dep_s32(a.seq_lens + j);
      too_long |= raw > min(a.max_seq_len, a.cap);
      const int len = clamp_len(a, raw);
      if (b0 == 0) len0 = len;
      nt = (len + kTileTokens - 1) / kTileTokens;
    }
    for (int o_ = 1; o_ < 32; o_ <<= 1) nt += __shfl_xor_sync(0xffffffffu, nt, o_);
    total += nt;
  }
  const bool flag_too_long = blockIdx.x == 0 && __any_sync(0xffffffffu, too_long) && lane == 0;
  total *= a.n_kv;
  // range [total * wid / nw, total * (wid + 1) / nw), 32-bit division when it fits
  const bool narrow = total * nw < (1ll << 32);
  const long long r0 = !mine ? 0 : narrow ? static_cast<long long>(static_cast<unsigned>(total * wid) /
                                                                   static_cast<unsigned>(nw))
                                          : total * wid / nw;
  const long long r1 = !mine ? 0 : narrow ? static_cast<long long>(static_cast<unsigned>(total * (wid + 1)) /
                                                                   static_cast<unsigned>(nw))
                                          : total * (wid + 1) / nw;
  long long rem = r1 - r0;   // tiles left to plan

  // locate r0: per group of 32 sequences an inclusive scan of their tile
  // counts, then a per-lane binary search over it
  Cursor pc = {0, 0, 0, 0, 0};
  {
    bool found = rem <= 0;
    long long acc = 0;   // tiles before the group
    for (int b0 = 0; b0 < a.batch && __any_sync(0xffffffffu, !found); b0 += 32) {
      const int bb = b0 + lane;
      const int len = bb < a.batch ? (b0 == 0 ? len0 : clamp_len(a, ld_dep_s32(a.seq_lens + bb))) : 0;
      const int nt = (len + kTileTokens - 1) / kTileTokens;
      const long long span = static_cast<long long>(nt) * a.n_kv;
      long long inc = span;
      for (int o_ = 1; o_ < 32; o_ <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, inc, o_);
        if (lane >= o_) inc += y;
      }
      const long long gtotal = __shfl_sync(0xffffffffu, inc, 31);
      const long long key = bb < a.batch ? acc + inc : LLONG_MAX;   // end of sequence bb's tiles
      // idx = number of sequences of the group that end at or before r0
      int idx = 0;
#pragma unroll
      for (int step = 16; step >= 1; step >>= 1) {
        const long long v = __shfl_sync(0xffffffffu, key, idx + step - 1);
        if (v <= r0) idx += step;
      }
      const long long k31 = __shfl_sync(0xffffffffu, key, 31);
      if (idx == 31 && k31 <= r0) idx = 32;
      const int src = idx & 31;
      const long long e_end = __shfl_sync(0xffffffffu, key, src);
      const long long e_span = __shfl_sync(0xffffffffu, span, src);
      const int n_t = __shfl_sync(0xffffffffu, nt, src);
      const int ln = __shfl_sync(0xffffffffu, len, src);
      if (!found && idx < 32 && b0 + idx < a.batch) {
        found = true;
        const int off = static_cast<int>(r0 - (e_end - e_span));
        pc.b = b0 + idx;
        pc.h = off / n_t;
        pc.t = off - pc.h * n_t;
        pc.nt = n_t;
        pc.len = ln;
      }
      acc += gtotal;
    }
  }

  // the next chunk to issue (planned one chunk ahead, block ids in flight)
  int n_n = 0, n_seg = 0, n_len = 0, n_b = 0, n_h = 0, n_t = 0;
  int n_blk[kChunk];
#pragma unroll
  for (int i = 0; i < kChunk; ++i) n_blk[i] = -1;
  auto plan = [&]() {
    int n = min(kChunk, pc.nt - pc.t);
    if (rem < n) n = static_cast<int>(rem);
    if (a.part_tiles > 0) n = min(n, a.part_tiles - pc.t % a.part_tiles);
    n_n = n;
    n_b = pc.b;
    n_h = pc.h;
    n_t = pc.t;
    n_len = pc.len;
    n_seg = (pc.b * a.n_kv + pc.h) * a.num_parts + (a.part_tiles > 0 ? pc.t / a.part_tiles : 0);
    const int* row = a.block_table + static_cast<long long>(pc.b) * a.bt_stride;
#pragma unroll
    for (int i = 0; i < kChunk; ++i) n_blk[i] = ldg_or(row + (((pc.t + i) << 4) >> a.log2_bs), i < n, -1);
    rem -= n;
    for (int i = 0; i < n && rem > 0; ++i) cursor_next(pc, a);
  };
  if (mine && rem > 0) plan();
  if (a.early_indices) wait_previous();
  if (flag_too_long) flag(a.status, TQ_DEV_SEQ_TOO_LONG);

  const uint64_t policy = evict_first_policy();
  const long long blk_bytes = static_cast<long long>(a.n_kv) * a.tiles_per_block * a.tile_bytes;   // one cache block
  // stage_at without its division: stages [0, nb_front) lie before the LUT
  const uint32_t nb_front = klut && lut > first ? (lut - first) / a.stage_bytes : (klut ? 0u : 0xFFFFFFFFu);
  const uint32_t back = lut + klut;
  const uint32_t qslot = qslots + static_cast<uint32_t>(mine ? jc : 0) * a.qslot_bytes;
  const uint32_t qbar = q_empty_bar(bars, W, mine ? jc : 0);
  uint32_t eparity = (1u << kStages) - 1;   // empty-barrier parity to wait for, per stage
  uint32_t used = 0, fpar = 0;              // stages ever filled; parity of their next fill
  int ps = 0, prev_seg = -1;
  int qn = 0, qdone = 0;                    // query copies issued / known consumed
  bool done = !mine;
  uint64_t idle_since = 0;   // start of the current stretch without progress (0: none)
  while (__any_sync(0xffffffffu, !done)) {
    bool progressed = false;
    // one chunk per lane per pass: the block ids plan() loads for the next
    // chunk are only read on the next pass, after other lanes' work
    for (int pass = 0; pass < TQ_PRODUCER_PASSES && !done; ++pass) {
      const bool newq = n_n > 0 && n_seg != prev_seg;
      if (newq && qdone < qn) {   // the slot still holds rows the consumer has not taken
        if (!mbar_test(qbar, (qn - 1) & 1)) break;
        qdone = qn;
      }
      const uint32_t fb = full_bar(bars, jc, ps);
      if (!mbar_test(fb + 8, (eparity >> ps) & 1u)) break;
      eparity ^= 1u << ps;
      const uint32_t idx = static_cast<uint32_t>(jc * kStages + ps);
      const uint32_t sa = idx < nb_front ? first + idx * a.stage_bytes : back + (idx - nb_front) * a.stage_bytes;
      const bool last = rem <= 0;
      uint32_t okm = 0, bytes = 0;
#pragma unroll
      for (int i = 0; i < kChunk; ++i)
        if (i < n_n && n_blk[i] >= 0 && n_blk[i] < a.num_blocks) {
          okm |= 1u << i;
          bytes += a.tile_bytes;
        }
      if (newq) bytes += a.qbuf_bytes;
      sts128(sa + a.desc_off, make_uint4(static_cast<uint32_t>(n_seg), static_cast<uint32_t>(n_t << 4),
                                         static_cast<uint32_t>(n_len),
                                         static_cast<uint32_t>(n_n) | (okm << 4) | (last ? 256u : 0u) |
                                             (newq ? 512u : 0u)));
      // No proxy fence: the consumer's reads of the stage are ordered before
      // these copies by its arrive on the empty barrier (release) and the
      // test above (acquire); the descriptor goes generic store -> generic load
      // through the full barrier.
      mbar_expect(fb, bytes);
#pragma unroll
      for (int i = 0; i < kChunk; ++i)
        if ((okm >> i) & 1u) {
          const uint8_t* src = a.cache + static_cast<long long>(n_blk[i]) * blk_bytes +
                               static_cast<uint32_t>(n_h * a.tiles_per_block + ((n_t + i) & (a.tiles_per_block - 1))) *
                                   static_cast<uint32_t>(a.tile_bytes);
          bulk_g2s(sa + i * a.tile_bytes, src, a.tile_bytes, fb, policy);
        }
      if (newq) {
        const uint8_t* src = static_cast<const uint8_t*>(a.q) +
                             (static_cast<long long>(n_b) * a.n_q + n_h * a.group) * (kD * 2);
        bulk_g2s_plain(qslot, src, a.qbuf_bytes, fb);
        ++qn;
      }
      if (n_n > 0) prev_seg = n_seg;
      used |= 1u << ps;
      fpar ^= 1u << ps;
      ps = ps + 1 == kStages ? 0 : ps + 1;
      progressed = true;
      if (last) done = true;
      else plan();
    }
    if (__any_sync(0xffffffffu, progressed)) {
      idle_since = 0;
    } else {
      const uint64_t now = global_ns();
      if (!idle_since) idle_since = now;
      else if (now - idle_since > kWaitNs) {   // a consumer stopped taking stages
        if (lane == 0) flag(a.status, TQ_DEV_TIMEOUT);
        break;
      }
      if (TQ_PRODUCER_SLEEP_NS > 0) __nanosleep(TQ_PRODUCER_SLEEP_NS);
    }
  }
  // every copy this lane issued has landed before the warp leaves (bounded)
  if (mine)
    for (int s = 0; s < kStages; ++s)
      if ((used >> s) & 1u) mbar_wait(full_bar(bars, jc, s), ((fpar >> s) & 1u) ^ 1u);
}

// ---------------------------------------------------------------- append

// The newest token of the stage's segment (position len - 1, in tile i of the
// stage, row r): the warp quantises its raw key and value rows (prefetched
// into the query slot's tail at `raw`; the key in the first half-warp, the
// value in the second) with the store's arithmetic, writes the bytes into the
// cache tile in global memory and patches the same row of the stage's copy,
// which the bulk copy brought with the row's old bytes. The patch goes
// through the generic proxy; the fence orders it before the stage's next
// bulk fill (async proxy) once the consumer releases the stage.
template <int KMODE, int VBITS, typename TQ>
__device__ __noinline__ void append_newest(const DecodeArgs& a, uint32_t sa, uint4 desc, int lane, uint32_t raw,
                                           uint32_t codebook) {
  const int len = static_cast<int>(desc.z), tok0 = static_cast<int>(desc.y);
  const int p = len - 1;
  const int i = (p - tok0) >> 4, r = p & (kTileTokens - 1);
  const int bh = static_cast<int>(desc.x) / a.num_parts;
  const int b = bh / a.n_kv, h = bh - b * a.n_kv;
  // the tile was found, so this block id is in range; its load overlaps the quantisation
  const long long blk = ld_dep_s32(a.block_table + static_cast<long long>(b) * a.bt_stride + (p >> a.log2_bs));
  const int l = lane & 15;
  const TileGeom g = {a.k_off, a.k_row, a.v_off, a.v_row, a.knorm_off, a.vscale_off, a.vzero_off};
  uint8_t* gtile = a.wcache + (blk * a.n_kv + h) * a.tiles_per_block * static_cast<long long>(a.tile_bytes) +
                   static_cast<long long>((p >> 4) & (a.tiles_per_block - 1)) * a.tile_bytes;
  uint8_t* stile = static_cast<uint8_t*>(__cvta_shared_to_generic(sa + static_cast<uint32_t>(i * a.tile_bytes)));
  const float* mid = static_cast<const float*>(__cvta_shared_to_generic(codebook));
  const float* cent = mid + 16;
  // the first half quantises the key, the second the value, at the same time
  const bool kh = lane < 16;
  const unsigned hm = kh ? 0x0000ffffu : 0xffff0000u;
  const uint32_t row = raw + (kh ? 0u : kRawRowBytes) + 16u * static_cast<uint32_t>(l);
  PairBytes o;
  float x[8];
  u2_to_f4<TQ>(lds64(row), x);
  u2_to_f4<TQ>(lds64(row + 8), x + 4);
  if (kh) {
    quantize_key<KMODE>(x, l, mid, cent, o, hm);
    write_key<KMODE>(gtile, r, g, l, o);
    write_key<KMODE>(stile, r, g, l, o);
  } else {
    quantize_value<VBITS>(x, o, hm);
    write_value<VBITS>(gtile, r, g, l, o);
    write_value<VBITS>(stile, r, g, l, o);
  }
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  __syncwarp();
}

// ---------------------------------------------------------------- consumer warps

// Consumer warp j: takes its ring stages in order and runs the attention math
// on every tile. Column layout of the score and output tiles (8 columns):
//   G <= 4: column k < 4 carries the hi part of head k, column 4 + k the lo
//     part, so lanes c and c ^ 2 of a quad hold the two parts of heads
//     2 (c & 1), 2 (c & 1) + 1 and one exchange gives both the full score.
//   G > 4: column k is head k; the lo parts run in a second mma into the same
//     accumulators.
template <int KMODE, int GBIG, int VBITS, typename TQ, bool APPEND>
__device__ void consumer_warp(const DecodeArgs& a, int W, int j, uint32_t bars, uint32_t qslots, uint32_t first,
                              uint32_t lut,
                              uint32_t klut) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;   // mma groupID
  const int c = lane & 3;    // thread in group
  const int G = a.group;
  const int wid = blockIdx.x * W + j;
  const int hd0 = GBIG ? 2 * c : 2 * (c & 1);   // heads of this lane's columns: hd0, hd0 + 1
  const bool lo_lane = !GBIG && c >= 2;
  const bool colv0 = hd0 < G, colv1 = hd0 + 1 < G;
  const bool colmask = GBIG ? G < 8 : G < 4;    // some columns carry no head
  uint32_t lut_lane = 0;
  if constexpr (KMODE != kFp8) lut_lane = lut + 4u * lane;
  uint32_t stg[kStages];
#pragma unroll
  for (int s = 0; s < kStages; ++s) stg[s] = stage_at(first, lut, klut, a.stage_bytes, j * kStages + s);

  uint32_t qb[GBIG ? 32 : 16];     // Q^T B operands (per k-step; GBIG: hi then lo)
  float o[8][4];                   // O^T accumulators, rows d, cols 2c, 2c+1
  float m0 = -1e30f, m1 = -1e30f, l0 = 0.f, l1 = 0.f, z0 = 0.f, z1 = 0.f;
  int c_seg = -1;
  uint32_t fpar = 0;

  auto finalize = [&](int seg) {
    float l_[2] = {l0, l1}, z_[2] = {z0, z1};
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
      for (int o_ = GBIG ? 4 : 2; o_ < 32; o_ <<= 1) {   // G <= 4: lanes c, c ^ 2 hold tokens g, g + 8
        l_[e] += __shfl_xor_sync(0xffffffffu, l_[e], o_);
        z_[e] += __shfl_xor_sync(0xffffffffu, z_[e], o_);
      }
    const float mm[2] = {m0, m1};
    const int rec = seg + wid;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int hd = hd0 + e;
      const bool writer = hd < G && !lo_lane;
      const float inv = l_[e] > 0.f ? 1.f / l_[e] : 0.f;
      float* dst = a.rec_o + (static_cast<long long>(rec) * G + (writer ? hd : 0)) * kD + 16 * g;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        float v0 = o[mt][e], v1 = o[mt][2 + e];
        if (!GBIG) {   // add the lo-part columns held by lane ^ 2
          v0 += __shfl_xor_sync(0xffffffffu, v0, 2);
          v1 += __shfl_xor_sync(0xffffffffu, v1, 2);
        }
        // value operands carried code * 2^-24 (rows g) and code * 2^-20 (rows g + 8)
        if (writer)
          *reinterpret_cast<float2*>(dst + 2 * mt) =
              make_float2(fmaf(v0, 16777216.f, z_[e]) * inv, fmaf(v1, 1048576.f, z_[e]) * inv);
      }
      if (writer && g == 0)
        a.rec_lse[static_cast<long long>(rec) * G + hd] = l_[e] > 0.f ? mm[e] + __log2f(l_[e]) : -INFINITY;
    }
  };

  // query rows of a new segment: rotate, scale, split hi/lo, and place into the
  // B operands through the query slot itself. Each lane overwrites its own 8
  // bytes of every raw row with the hi parts (row = head, fp16), keeping the lo
  // parts in registers; each lane then loads its operand column (column g,
  // coordinates 32c .. 32c + 31: one 64-byte run); then the same for the lo
  // parts.
  auto begin_segment = [&](uint32_t qrows) {
    uint32_t lo[8][2];   // per head: lo01, lo23 of coordinates 4 lane .. +3
#pragma unroll
    for (int gg = 0; gg < 8; ++gg) {
      if (gg < G) {
        const uint32_t at = qrows + gg * kD * 2 + 8 * lane;
        float x[4];
        u2_to_f4<TQ>(lds64(at), x);
        float sc = a.qscale;
        if constexpr (KMODE != kFp8) {
          fwht128(x, lane);
          sc *= 0.088388347648318440f;   // 1 / sqrt(128)
        }
        uint32_t h01, h23;
        split_half2(x[0] * sc, x[1] * sc, h01, lo[gg][0]);
        split_half2(x[2] * sc, x[3] * sc, h23, lo[gg][1]);
        sts64(at, make_uint2(h01, h23));
      }
    }
#pragma unroll
    for (int part = 0; part < 2; ++part) {   // 0: hi parts, 1: lo parts
      if (part == 1) {
#pragma unroll
        for (int gg = 0; gg < 8; ++gg)
          if (gg < G) sts64(qrows + gg * kD * 2 + 8 * lane, make_uint2(lo[gg][0], lo[gg][1]));
      }
      __syncwarp();
      // column g of the B operand: G <= 4: hi of head g (g < 4), lo of head
      // g - 4 (g >= 4); G > 4: head g, hi then lo in the second register half
      const int row = GBIG ? g : (part == 0 ? g : g - 4);
      const bool mine = GBIG ? (g < G) : (part == 0 ? g < G : (g >= 4 && g - 4 < G));
      uint4 r[4] = {};
      if (mine) {
#pragma unroll
        for (int k = 0; k < 4; ++k) r[k] = lds128(qrows + row * kD * 2 + 64 * c + 16 * k);
      }
      const int base = GBIG ? 16 * part : 0;
      if (GBIG || mine || part == 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          qb[base + 4 * k] = r[k].x;
          qb[base + 4 * k + 1] = r[k].y;
          qb[base + 4 * k + 2] = r[k].z;
          qb[base + 4 * k + 3] = r[k].w;
        }
      }
      __syncwarp();   // every lane has read this part before the next overwrites it
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    m0 = m1 = -1e30f;
    l0 = l1 = z0 = z1 = 0.f;
  };

  // NT (1 or 2) tiles of a stage at shared address st, in lock-step phases so
  // their accumulation chains interleave; tile i has nv[i] real positions
  // (tiles past the chunk's end compute on stale bytes and are fully masked)
  auto chunk = [&](auto nt_tag, uint32_t st, const int* nv, uint32_t release_bar) {
    constexpr int NT = decltype(nt_tag)::value;
    // ---- S_i = K_i . Q^T
    float v[NT][4];   // [0] tok g col 2c, [1] tok g col 2c+1, [2] tok g+8 col 2c, [3] tok g+8 col 2c+1
    if constexpr (KMODE == kFp8) {
#pragma unroll
      for (int i = 0; i < NT; ++i) v[i][0] = v[i][1] = v[i][2] = v[i][3] = 0.f;
#pragma unroll
      for (int i = 0; i < NT; ++i) {
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
          mma16816(v[i], a0, a1, a2, a3, qb[2 * s], qb[2 * s + 1]);
          if (GBIG) mma16816(v[i], a0, a1, a2, a3, qb[16 + 2 * s], qb[16 + 2 * s + 1]);
        }
      }
    } else {
      uint4 kg[NT], kh[NT];   // this lane's key slices of tokens g and g+8
#pragma unroll
      for (int i = 0; i < NT; ++i) {
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
      // M rows: tokens g and g + 8; k-step s holds this lane's coordinates
      // 32c + 4s .. +3 (two key bytes = two LUT entries of two centroids each).
      // Two accumulators per tile (even and odd k-steps; G > 4: hi and lo query
      // parts) halve the dependent mma chains.
      float va[NT][4], vb[NT][4];
#pragma unroll
      for (int i = 0; i < NT; ++i)
#pragma unroll
        for (int k = 0; k < 4; ++k) va[i][k] = vb[i][k] = 0.f;
#pragma unroll
      for (int s2 = 0; s2 < 8; ++s2) {
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          const uint32_t g0 = lds32(lut_addr<KMODE>(kg[i], 2 * s2, lut_lane));
          const uint32_t g1 = lds32(lut_addr<KMODE>(kg[i], 2 * s2 + 1, lut_lane));
          const uint32_t h0 = lds32(lut_addr<KMODE>(kh[i], 2 * s2, lut_lane));
          const uint32_t h1 = lds32(lut_addr<KMODE>(kh[i], 2 * s2 + 1, lut_lane));
          if (GBIG) {
            mma16816(va[i], g0, h0, g1, h1, qb[2 * s2], qb[2 * s2 + 1]);
            mma16816(vb[i], g0, h0, g1, h1, qb[16 + 2 * s2], qb[16 + 2 * s2 + 1]);
          } else if ((s2 & 1) == 0) {
            mma16816(va[i], g0, h0, g1, h1, qb[2 * s2], qb[2 * s2 + 1]);
          } else {
            mma16816(vb[i], g0, h0, g1, h1, qb[2 * s2], qb[2 * s2 + 1]);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < NT; ++i)
#pragma unroll
        for (int k = 0; k < 4; ++k) v[i][k] = va[i][k] + vb[i][k];
    }

    // ---- value words of the tiles, read now so the stage can be released
    // before the softmax and O^T: the producer refills it half a chunk earlier
    uint4 vwa[NT], vwb[NT];   // the lane's words of token pairs (2c, 2c+1) and (2c+8, 2c+9)
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      if constexpr (VBITS == 4) {   // 16-byte group g of each pair, swizzled by 2 c
        const uint32_t vt = st + i * a.tile_bytes + a.v_off + 16 * (g ^ (2 * c));
        vwa[i] = lds128(vt + 128 * c);
        vwb[i] = lds128(vt + 128 * (c + 4));
      } else {                      // 12 bytes at 12 g of each 96-byte pair
        const uint32_t vt = st + i * a.tile_bytes + a.v_off + 12 * g;
        vwa[i] = make_uint4(lds32(vt + 96 * c), lds32(vt + 96 * c + 4), lds32(vt + 96 * c + 8), 0u);
        vwb[i] = make_uint4(lds32(vt + 96 * (c + 4)), lds32(vt + 96 * (c + 4) + 4), lds32(vt + 96 * (c + 4) + 8), 0u);
      }
    }
    auto release = [&]() {   // every lane has read the stage (values, norms, scales, zeros)
      if (release_bar) {
        __syncwarp();
        if (lane == 0) mbar_arrive(release_bar);
      }
    };

    // ---- scores, probabilities and O^T += V^T . P^T
    if constexpr (!GBIG) {
      // G <= 4: after the hi/lo exchange lanes c and c ^ 2 hold the same
      // scores; lane c < 2 carries on with token g, lane c >= 2 with token
      // g + 8 (its l, z are summed over the pair at the end), and one more
      // exchange gives each lane the other half of the P^T operands.
      const int tk = lo_lane ? g + 8 : g;
      float t0[NT], t1[NT], sv[NT], sz[NT];
      float cm0 = -INFINITY, cm1 = -INFINITY;
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        const uint32_t tb = st + i * a.tile_bytes;
#pragma unroll
        for (int k = 0; k < 4; ++k) v[i][k] += __shfl_xor_sync(0xffffffffu, v[i][k], 2);
        float x0 = lo_lane ? v[i][2] : v[i][0], x1 = lo_lane ? v[i][3] : v[i][1];
        if constexpr (KMODE != kFp8) {
          const float nk = lds_h2f(tb + a.knorm_off + 2 * tk);
          x0 *= nk;
          x1 *= nk;
        }
        sv[i] = lds_h2f(tb + a.vscale_off + 2 * tk);
        sz[i] = lds_h2f(tb + a.vzero_off + 2 * tk);
        if (tk >= nv[i]) { x0 = x1 = -INFINITY; sv[i] = 0.f; sz[i] = 0.f; }   // missing, ragged, past the end
        if (colmask) {
          if (!colv0) x0 = -INFINITY;
          if (!colv1) x1 = -INFINITY;
        }
        t0[i] = x0;
        t1[i] = x1;
        cm0 = fmaxf(cm0, x0);
        cm1 = fmaxf(cm1, x1);
      }
      release();
      if (__any_sync(0xffffffffu, cm0 > m0 + kTau || cm1 > m1 + kTau)) {   // rare: move the max, rescale
#pragma unroll
        for (int o_ = 2; o_ < 32; o_ <<= 1) {
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
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        const float p0 = ex2(t0[i] - m0), p1 = ex2(t1[i] - m1);
        l0 += p0;
        l1 += p1;
        z0 = fmaf(p0, sz[i], z0);
        z1 = fmaf(p1, sz[i], z1);
        uint32_t hi, lo;   // hi/lo half2 of (col 2c, col 2c+1) for token tk
        split_half2(p0 * sv[i], p1 * sv[i], hi, lo);
        // b0 (tokens 0..7): hi parts from lanes c < 2, lo parts from c >= 2;
        // b1 (tokens 8..15) the same: each lane lacks one of the two
        const uint32_t recv = __shfl_xor_sync(0xffffffffu, lo_lane ? hi : lo, 2);
        const uint32_t b0 = movmatrix_trans(lo_lane ? recv : hi), b1 = movmatrix_trans(lo_lane ? lo : recv);
        const uint4 va = vwa[i], vb = vwb[i];
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)   // rows g, g + 8 of tile mt: coordinates 16 g + 2 mt, + 1
          mma16816(o[mt], code_field<VBITS>(va, 2 * mt, 0), code_field<VBITS>(va, 2 * mt + 1, 4),
                   code_field<VBITS>(vb, 2 * mt, 0), code_field<VBITS>(vb, 2 * mt + 1, 4), b0, b1);
      }
      return;
    }

    // ---- G > 4: every lane carries both of its tokens
    float svg[NT], svh[NT], szg[NT], szh[NT];
    float cm0 = -INFINITY, cm1 = -INFINITY;
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      const uint32_t tb = st + i * a.tile_bytes;
      if (!GBIG) {
#pragma unroll
        for (int k = 0; k < 4; ++k) v[i][k] += __shfl_xor_sync(0xffffffffu, v[i][k], 2);
      }
      if constexpr (KMODE != kFp8) {
        const float ng = lds_h2f(tb + a.knorm_off + 2 * g), nh = lds_h2f(tb + a.knorm_off + 2 * g + 16);
        v[i][0] *= ng; v[i][1] *= ng; v[i][2] *= nh; v[i][3] *= nh;
      }
      svg[i] = lds_h2f(tb + a.vscale_off + 2 * g);
      svh[i] = lds_h2f(tb + a.vscale_off + 2 * g + 16);
      szg[i] = lds_h2f(tb + a.vzero_off + 2 * g);
      szh[i] = lds_h2f(tb + a.vzero_off + 2 * g + 16);
      if (nv[i] < kTileTokens) {   // missing, ragged or past the chunk's end
        if (g >= nv[i]) { v[i][0] = v[i][1] = -INFINITY; svg[i] = 0.f; szg[i] = 0.f; }
        if (g + 8 >= nv[i]) { v[i][2] = v[i][3] = -INFINITY; svh[i] = 0.f; szh[i] = 0.f; }
      }
      if (colmask) {
        if (!colv0) v[i][0] = v[i][2] = -INFINITY;
        if (!colv1) v[i][1] = v[i][3] = -INFINITY;
      }
      cm0 = fmaxf(cm0, fmaxf(v[i][0], v[i][2]));
      cm1 = fmaxf(cm1, fmaxf(v[i][1], v[i][3]));
    }
    release();
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
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      const float p0 = ex2(v[i][0] - m0), p1 = ex2(v[i][1] - m1);
      const float p2 = ex2(v[i][2] - m0), p3 = ex2(v[i][3] - m1);
      l0 += p0 + p2;
      l1 += p1 + p3;
      z0 = fmaf(p0, szg[i], fmaf(p2, szh[i], z0));
      z1 = fmaf(p1, szg[i], fmaf(p3, szh[i], z1));
      uint32_t hg, lg, hh, lh;   // hi/lo half2 of (col 2c, col 2c+1) for tokens g and g+8
      split_half2(p0 * svg[i], p1 * svg[i], hg, lg);
      split_half2(p2 * svh[i], p3 * svh[i], hh, lh);
      const uint32_t b0 = movmatrix_trans(lo_lane ? lg : hg), b1 = movmatrix_trans(lo_lane ? lh : hh);
      uint32_t b0l = 0u, b1l = 0u;
      if (GBIG) { b0l = movmatrix_trans(lg); b1l = movmatrix_trans(lh); }
      const uint4 va = vwa[i], vb = vwb[i];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {   // rows g, g + 8 of tile mt: coordinates 16 g + 2 mt, + 1
        const uint32_t a0 = code_field<VBITS>(va, 2 * mt, 0), a1 = code_field<VBITS>(va, 2 * mt + 1, 4);
        const uint32_t a2 = code_field<VBITS>(vb, 2 * mt, 0), a3 = code_field<VBITS>(vb, 2 * mt + 1, 4);
        mma16816(o[mt], a0, a1, a2, a3, b0, b1);
        if (GBIG) mma16816(o[mt], a0, a1, a2, a3, b0l, b1l);
      }
    }
  };

  int cs = 0;
  bool aborted = false;
  uint32_t rbuf = 0;   // append: offset of the current segment's raw rows in the slot's tail (two halves)
  for (;;) {
    const uint32_t fb = full_bar(bars, j, cs);
    if (!mbar_wait(fb, (fpar >> cs) & 1u)) { aborted = true; break; }
    fpar ^= 1u << cs;
    uint32_t sa = stg[0];
#pragma unroll
    for (int s = 1; s < kStages; ++s) sa = cs == s ? stg[s] : sa;
    const uint4 desc = lds128(sa + a.desc_off);
    const int n = static_cast<int>(desc.w & 7u);
    const uint32_t okm = (desc.w >> 4) & 0xFu;
    const bool last = (desc.w >> 8) & 1u;
    if (n > 0) {
      const int seg = static_cast<int>(desc.x);
      if (seg != c_seg) {
        if (c_seg >= 0) finalize(c_seg);
        begin_segment(qslots + static_cast<uint32_t>(j) * a.qslot_bytes);
        __syncwarp();   // every lane has read the query slot: the producer may refill it
        if (lane == 0) mbar_arrive(q_empty_bar(bars, W, j));
        c_seg = seg;
        if constexpr (APPEND) {
          // the segment's newest key and value rows, in case its last tile is
          // in this warp's range: one 16-byte cp.async per lane into the half
          // of the slot's tail this segment uses (the other half may still be
          // the previous segment's, in flight)
          rbuf ^= kRawRowBytes * 2;
          const long long row = static_cast<long long>(seg / a.num_parts) * kRawRowBytes + 16 * (lane & 15);
          const uint8_t* src = static_cast<const uint8_t*>(lane < 16 ? a.new_k : a.new_v) + row;
          const uint32_t dst = qslots + static_cast<uint32_t>(j) * a.qslot_bytes + static_cast<uint32_t>(a.qbuf_bytes) +
                               rbuf + (lane < 16 ? 0u : kRawRowBytes) + 16u * static_cast<uint32_t>(lane & 15);
          asm volatile("cp.async.wait_group 1;\n" ::: "memory");   // the other half's copy has landed
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
          asm volatile("cp.async.commit_group;\n" ::: "memory");
        }
      }
      const int tok0 = static_cast<int>(desc.y), len = static_cast<int>(desc.z);
      if (okm != (1u << n) - 1 && lane == 0) flag(a.status, TQ_DEV_BLOCK_OUT_OF_RANGE);
      if constexpr (APPEND) {
        // the newest position of the segment is in this chunk (a chunk never
        // passes the sequence's end, so reaching it is enough), its tile was
        // found, and the length was not cut (only a length at the limit needs
        // the raw value)
        if (tok0 + kTileTokens * n >= len && ((okm >> (n - 1)) & 1u)) {
          const int bh = seg / a.num_parts;
          if (len < min(a.max_seq_len, a.cap) || ld_dep_s32(a.seq_lens + bh / a.n_kv) == len) {
            asm volatile("cp.async.wait_all;\n" ::: "memory");
            __syncwarp();   // every lane's rows have landed
            const uint32_t raw = qslots + static_cast<uint32_t>(j) * a.qslot_bytes +
                                 static_cast<uint32_t>(a.qbuf_bytes) + rbuf;
            append_newest<KMODE, VBITS, TQ>(a, sa, desc, lane, raw, bars + kCodebookOff);
          }
        }
      }
      int nv[kChunk];
#pragma unroll
      for (int i = 0; i < kChunk; ++i)
        nv[i] = (i < n && ((okm >> i) & 1u)) ? min(kTileTokens, len - tok0 - 16 * i) : 0;
      // a stage's tiles two at a time in lock step, an odd last tile alone; the
      // last call releases the stage once it has read it
#pragma unroll
      for (int t0 = 0; t0 < kChunk; t0 += 2) {
        if (t0 > 0 && n <= t0) break;
        const uint32_t rel = t0 + 2 >= kChunk || n <= t0 + 2 ? fb + 8 : 0u;
        if (t0 + 1 < kChunk) chunk(std::integral_constant<int, 2>{}, sa + t0 * a.tile_bytes, nv + t0, rel);
        else chunk(std::integral_constant<int, 1>{}, sa + t0 * a.tile_bytes, nv + t0, rel);
      }
    } else {
      __syncwarp();   // every lane has read the descriptor: the producer may refill the stage
      if (lane == 0) mbar_arrive(fb + 8);
    }
    cs = cs + 1 == kStages ? 0 : cs + 1;
    if (last) break;
  }
  if (aborted) {
    if (lane == 0) flag(a.status, TQ_DEV_TIMEOUT);
  } else if (c_seg >= 0) {
    finalize(c_seg);
  }
  if constexpr (APPEND) asm volatile("cp.async.wait_all;\n" ::: "memory");   // no copy outlives the CTA
}

// ---------------------------------------------------------------- split kernel

// Warps 0 .. kProducers - 1 are producers; the rest are the W consumers. One
// CTA per SM.
template <int KMODE, int GBIG, int VBITS, typename TQ, bool APPEND>
__global__ void __launch_bounds__((kMaxConsumers + kProducers) * 32, 1)
split_kernel(const DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t s_dyn[];
  const int warp = threadIdx.x >> 5;
  const int W = static_cast<int>(blockDim.x >> 5) - kProducers;
  const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(s_dyn));
  const uint32_t end = base + static_cast<uint32_t>(a.dyn_bytes);
  constexpr uint32_t kLut = lut_bytes<KMODE>();
  const uint32_t head = kBarHead + static_cast<uint32_t>(W) * a.qslot_bytes;
  const uint32_t lut = kLut ? lut_at(base, kLut, head) : end;
  const uint32_t bars = base;
  const uint32_t qslots = base + kBarHead;
  const uint32_t first = base + head;
  const bool fits = W >= 1 && W <= kMaxConsumers && (!kLut || lut + kLut <= end) &&
                    stage_at(first, lut, kLut, a.stage_bytes, W * kStages - 1) + a.stage_bytes <= end;
  if (!__syncthreads_and(fits)) {   // launch misconfigured: flag and leave
    grid_dep_wait();
    if (threadIdx.x == 0) flag(a.status, TQ_DEV_TIMEOUT);
    return;
  }
  // Barrier init and the LUT (from kernel parameters) touch no global memory,
  // so they overlap the end of the previous kernel; everything after
  // grid_dep_wait() may read what that kernel wrote. The producer starts as
  // soon as the barriers exist; the consumers build the LUT meanwhile and meet
  // it on named barrier 1 (arrive / sync).
  if (warp < kProducers) {
    if (warp == 0) {
      const int lane = threadIdx.x & 31;
      for (int i = lane; i < 2 * W * kStages + W; i += 32) mbar_init(bars + 8 * i, 1);
      asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (kProducers > 1) asm volatile("bar.sync 2, %0;\n" ::"r"(kProducers * 32) : "memory");   // barriers exist
    else __syncwarp();
    producer_warp(a, W, warp, bars, qslots, first, lut, kLut);   // waits for the previous kernel itself
  } else {
    constexpr int kP = kProducers * 32;
    if constexpr (kLut != 0) build_lut<KMODE>(lut, a.cent, threadIdx.x - kP, blockDim.x - kP);
    if (APPEND && threadIdx.x - kP < 32) {   // the key codebook of the append path
      const int i = threadIdx.x - kP;
      const float v = i < 16 ? (i < 15 ? a.mid[i] : 0.f) : a.scent[i - 16];
      asm volatile("st.shared.f32 [%0], %1;\n" ::"r"(bars + kCodebookOff + 4u * i), "f"(v) : "memory");
    }
    asm volatile("bar.sync 1, %0;\n" ::"r"(blockDim.x) : "memory");
    grid_dep_wait();   // already resolved: the producers passed it before arriving
    grid_dep_launch();
    consumer_warp<KMODE, GBIG, VBITS, TQ, APPEND>(a, W, warp - kProducers, bars, qslots, first, lut, kLut);
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
  return min(max(ld_dep_s32(a.seq_lens + b), 0), min(a.max_seq_len, a.cap));
}

// The reduce. The records of a partition are those of the consumer warps
// whose ranges overlap it, a contiguous warp range; a (partition, warp)
// candidate whose warp owns no tile at all has no record. Record 0 stands in
// for such a candidate, and a select, not a multiply, drops it (the workspace
// may hold any bits). All index work depends on seq_lens only. When the launch
// directly follows the split kernel of the same decode (early_lens), that work
// runs before the dependency wait, which comes right before the first load of
// a record: the split kernel triggers this launch only after its own wait, so
// every earlier kernel has completed, and it writes no lengths.
__device__ __forceinline__ long long div_nw(long long x, long long y, bool narrow) {
  return narrow ? static_cast<long long>(static_cast<unsigned>(x) / static_cast<unsigned>(y)) : x / y;
}

// Warp-wide: tiles before sequence b and in total (x n_kv) into pre[0..1]; the
// length of b into *len.
__device__ __forceinline__ void reduce_prefix(const ReduceArgs& a, int b, int lane, long long* pre, int* len) {
  long long before = 0, total = 0;
  for (int b0 = 0; b0 < a.batch; b0 += 32) {
    const int j = b0 + lane;
    const int len_j = j < a.batch ? reduce_len(a, j) : 0;
    if (j == b) *len = len_j;
    long long nt = (len_j + kTileTokens - 1) / kTileTokens;
    long long nb = j < b ? nt : 0;
    for (int o = 1; o < 32; o <<= 1) {
      nt += __shfl_xor_sync(0xffffffffu, nt, o);
      nb += __shfl_xor_sync(0xffffffffu, nb, o);
    }
    total += nt;
    before += nb;
  }
  if (lane == 0) {
    pre[0] = before * a.n_kv;
    pre[1] = total * a.n_kv;
  }
}

// Warp-wide, lane = partition p (p >= parts: none): the first consumer warp
// whose range overlaps partition p (tiles [seq0 + p ppt, seq0 + min((p + 1)
// ppt, nt)) of a line of T tiles split over nw warps) into *wf; returns the
// inclusive scan over the lanes of the overlapping warp counts.
__device__ __forceinline__ int partition_scan(int p, int parts, long long seq0, int ppt, int nt, long long T,
                                              long long nw, bool narrow, int lane, long long* wf) {
  *wf = 0;
  int inc = 0;
  if (p < parts) {
    const long long t0 = seq0 + static_cast<long long>(p) * ppt;
    const long long t1 = seq0 + min(static_cast<long long>(p + 1) * ppt, static_cast<long long>(nt));
    *wf = div_nw((t0 + 1) * nw - 1, T, narrow);
    inc = static_cast<int>(div_nw(t1 * nw - 1, T, narrow) - *wf + 1);
  }
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  return inc;
}

// Warp w owns tiles [T w / nw, T (w + 1) / nw): does it own any?
__device__ __forceinline__ bool warp_owns_tiles(long long w, long long T, long long nw, bool narrow) {
  return div_nw(T * w, nw, narrow) != div_nw(T * (w + 1), nw, narrow);
}

// Many (sequence, KV head) pairs with few partials each: one CTA per pair,
// thread (gg, d) = query head gg of the group, coordinate d. Warp 0 computes
// the warp ranges of 32 partitions at a time and a scan of their sizes, then
// takes the (partition, warp) candidates 16 at a time, one per lane, and
// publishes their records. Every thread then loads its coordinate of all their
// partials while warp 0 loads their LSEs for every head and publishes merge
// weights per (candidate, head), so the two loads overlap. Chunks are merged
// online.
template <typename TO>
__global__ void __launch_bounds__(8 * kD) reduce_bh_kernel(const ReduceArgs a) {
  constexpr int kCand = 16;
  __shared__ long long s_pre[2];
  __shared__ long long s_wf[32];
  __shared__ int s_inc[32];
  __shared__ int s_len, s_cnt;
  __shared__ int s_rec[kCand];
  __shared__ float s_w[kCand][8];
  __shared__ float s_alpha[8];
  const int h = blockIdx.x, b = blockIdx.y;
  const int G = a.group;
  const int gg = threadIdx.x / kD, d = threadIdx.x - gg * kD;
  const int lane = threadIdx.x & 31;
  const bool w0 = threadIdx.x < 32;
  bool waited = false;
  auto wait_once = [&]() {   // every global access but the lengths comes after it
    if (!waited) {
      grid_dep_wait();
      grid_dep_launch();
      waited = true;
    }
  };
  if (!a.early_lens) wait_once();
  if (w0) reduce_prefix(a, b, lane, s_pre, &s_len);
  __syncthreads();
  const long long orow = static_cast<long long>(b) * a.n_q + static_cast<long long>(h) * G + gg;
  const int len = s_len;
  if (len <= 0) {
    wait_once();
    store_out<TO>(a.out, orow * kD + d, 0.f);
    return;
  }
  const int nt = (len + kTileTokens - 1) / kTileTokens;
  const long long T = s_pre[1], nw = a.num_warps;
  const bool narrow = (T + 1) * nw < (1ll << 32);
  const long long seq0 = s_pre[0] + static_cast<long long>(h) * nt;   // first tile of (b, h)
  const long long seg0 = (static_cast<long long>(b) * a.n_kv + h) * a.num_parts;
  const int ppt = a.part_tiles > 0 ? a.part_tiles : nt;
  const int parts = (nt + ppt - 1) / ppt;
  float acc = 0.f, den = 0.f;
  float mxh[8];   // warp 0: running LSE max per head
#pragma unroll
  for (int k = 0; k < 8; ++k) mxh[k] = -INFINITY;
  for (int p0 = 0; p0 < parts; p0 += 32) {
    if (w0) {
      long long wf;
      const int inc = partition_scan(p0 + lane, parts, seq0, ppt, nt, T, nw, narrow, lane, &wf);
      s_wf[lane] = wf;
      s_inc[lane] = inc;
    }
    __syncthreads();
    const int C = s_inc[31];   // candidates (partition, warp) of the group, partition-major
    for (int k0 = 0; k0 < C; k0 += kCand) {
      bool ok = false;
      long long rec = 0;
      if (w0) {
        const int k = k0 + lane;
        int pi = 0;   // partition of candidate k: the first with inclusive count > k
#pragma unroll
        for (int step = 16; step >= 1; step >>= 1)
          if (s_inc[pi + step - 1] <= k) pi += step;
        const long long w = s_wf[pi] + (k - (pi > 0 ? s_inc[pi - 1] : 0));
        ok = lane < kCand && k < C && warp_owns_tiles(w, T, nw, narrow);
        rec = seg0 + p0 + pi + w;
        if (lane < kCand) s_rec[lane] = ok ? static_cast<int>(rec) : 0;
        if (lane == 0) s_cnt = min(kCand, C - k0);
      }
      __syncthreads();   // candidates published
      wait_once();
      const int cnt = s_cnt;
      float x[kCand];    // this thread's coordinate of every candidate's partial
#pragma unroll
      for (int i = 0; i < kCand; ++i)
        x[i] = i < cnt ? ld_dep_f32(a.rec_o + (static_cast<long long>(s_rec[i]) * G + gg) * kD + d) : 0.f;
      if (w0) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (k < G) {
            const float lse = ok ? ld_dep_f32(a.rec_lse + rec * G + k) : -INFINITY;
            float cm = lse;
            for (int o = 1; o < 32; o <<= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
            const float nm = fmaxf(mxh[k], cm);
            if (lane < kCand) s_w[lane][k] = lse == -INFINITY ? 0.f : exp2f(lse - nm);
            if (lane == 0) s_alpha[k] = mxh[k] == -INFINITY ? 0.f : exp2f(mxh[k] - nm);
            mxh[k] = nm;
          }
        }
      }
      __syncthreads();   // weights published
      const float al = s_alpha[gg];
      acc *= al;
      den *= al;
#pragma unroll
      for (int i = 0; i < kCand; ++i) {
        if (i < cnt) {
          const float wgt = s_w[i][gg];
          den += wgt;
          acc = wgt != 0.f ? fmaf(wgt, x[i], acc) : acc;
        }
      }
      __syncthreads();   // weights and candidates used before warp 0 writes the next chunk's
    }
    __syncthreads();     // the group's scan is read before warp 0 writes the next
  }
  wait_once();
  store_out<TO>(a.out, orow * kD + d, den > 0.f ? acc / den : 0.f);
}

// Stream-K records (one partition per sequence), many (sequence, KV head)
// pairs: one CTA per pair, thread (gg, d) = query head gg of the group,
// coordinate d. A pair's tiles [seq0, seq0 + nt) of the line were split
// over a contiguous warp range, the owners of its first and last tile, so
// every thread finds its candidates by two divisions: no enumeration, no
// shared memory, no barrier. Each warp scans the lengths itself (before the
// dependency wait when the launch follows the split kernel); each thread
// then issues the loads of 8 candidates' LSEs and coordinates at once and
// merges them online.
__device__ __forceinline__ void prefix_all(const ReduceArgs& a, int b, int lane, long long* before, long long* total,
                                           int* len) {
  long long bf = 0, tt = 0;
  int ln = 0;
  for (int b0 = 0; b0 < a.batch; b0 += 32) {
    const int j = b0 + lane;
    const int len_j = j < a.batch ? reduce_len(a, j) : 0;
    if (b0 == (b & ~31)) ln = __shfl_sync(0xffffffffu, len_j, b & 31);
    long long nt = (len_j + kTileTokens - 1) / kTileTokens;
    long long nb = j < b ? nt : 0;
    for (int o = 1; o < 32; o <<= 1) {
      nt += __shfl_xor_sync(0xffffffffu, nt, o);
      nb += __shfl_xor_sync(0xffffffffu, nb, o);
    }
    tt += nt;
    bf += nb;
  }
  *before = bf * a.n_kv;
  *total = tt * a.n_kv;
  *len = ln;
}

template <typename TO>
__global__ void __launch_bounds__(8 * kD) reduce_sk_kernel(const ReduceArgs a) {
  constexpr int kCand = 8;
  const int h = blockIdx.x, b = blockIdx.y;
  const int G = a.group;
  const int gg = threadIdx.x / kD, d = threadIdx.x - gg * kD;
  const int lane = threadIdx.x & 31;
  if (!a.early_lens) {
    grid_dep_wait();
    grid_dep_launch();
  }
  long long before, T;
  int len;
  prefix_all(a, b, lane, &before, &T, &len);
  const long long orow = static_cast<long long>(b) * a.n_q + static_cast<long long>(h) * G + gg;
  const int nt = (len + kTileTokens - 1) / kTileTokens;
  const long long nw = a.num_warps;
  const bool narrow = (T + 1) * nw < (1ll << 32);
  const long long seq0 = before + static_cast<long long>(h) * nt;
  // owners of the pair's first and last tile (len > 0, so T > 0)
  const long long wf = len > 0 ? div_nw((seq0 + 1) * nw - 1, T, narrow) : 0;
  const long long wl = len > 0 ? div_nw((seq0 + nt) * nw - 1, T, narrow) : -1;
  const bool all_own = T >= nw;   // every warp owns a tile: no candidate to drop
  const long long seg = static_cast<long long>(b) * a.n_kv + h;   // record of warp w: seg + w
  if (a.early_lens) {
    grid_dep_wait();   // the records come from the split kernel
    grid_dep_launch();
  }
  if (len <= 0) {
    store_out<TO>(a.out, orow * kD + d, 0.f);
    return;
  }
  float m = -INFINITY, acc = 0.f, den = 0.f;
  for (long long w0 = wf; w0 <= wl; w0 += kCand) {
    float lse[kCand], x[kCand];
#pragma unroll
    for (int i = 0; i < kCand; ++i) {
      const long long w = w0 + i;
      const bool ok = w <= wl && (all_own || warp_owns_tiles(w, T, nw, narrow));
      const long long rec = seg + w;
      lse[i] = ok ? ld_dep_f32(a.rec_lse + rec * G + gg) : -INFINITY;
      x[i] = ok ? ld_dep_f32(a.rec_o + (rec * G + gg) * kD + d) : 0.f;
    }
    float cm = m;
#pragma unroll
    for (int i = 0; i < kCand; ++i) cm = fmaxf(cm, lse[i]);
    if (cm == -INFINITY) continue;
    const float al = m == -INFINITY ? 0.f : exp2f(m - cm);
    acc *= al;
    den *= al;
#pragma unroll
    for (int i = 0; i < kCand; ++i) {
      const float wgt = lse[i] == -INFINITY ? 0.f : exp2f(lse[i] - cm);
      den += wgt;
      acc = wgt != 0.f ? fmaf(wgt, x[i], acc) : acc;
    }
    m = cm;
  }
  store_out<TO>(a.out, orow * kD + d, den > 0.f ? acc / den : 0.f);
}

// Few pairs with many partials each: one CTA per (sequence, query head), 4
// warps; thread d of 128 = coordinate d in the final merge. Every warp scans
// the partitions 32 at a time; the (partition, warp) candidates of a group,
// partition-major, form chunks of 32 that go round robin to the 4 warps, one
// candidate per lane. A warp loads the records of its chunk (16 bytes per lane
// per record) before their weights are known, together with the candidates'
// LSEs, and merges online; the 4 warps' states are merged at the end.
constexpr int kReduceThreads = 128;

template <typename TO>
__global__ void __launch_bounds__(kReduceThreads) reduce_qh_kernel(const ReduceArgs a) {
  __shared__ long long s_pre[2];
  __shared__ int s_len;
  __shared__ float s_m[4], s_den[4];
  __shared__ __align__(16) float s_acc[4][kD];
  const int G = a.group;
  const int h = blockIdx.x / G, gg = blockIdx.x - h * G, b = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  bool waited = false;
  auto wait_once = [&]() {   // every global access but the lengths comes after it
    if (!waited) {
      grid_dep_wait();
      grid_dep_launch();
      waited = true;
    }
  };
  if (!a.early_lens) wait_once();
  if (warp == 0) reduce_prefix(a, b, lane, s_pre, &s_len);
  __syncthreads();
  const long long orow = static_cast<long long>(b) * a.n_q + static_cast<long long>(h) * G + gg;
  const int len = s_len;
  if (len <= 0) {
    wait_once();
    store_out<TO>(a.out, orow * kD + threadIdx.x, 0.f);
    return;
  }
  const int nt = (len + kTileTokens - 1) / kTileTokens;
  const long long T = s_pre[1], nw = a.num_warps;
  const bool narrow = (T + 1) * nw < (1ll << 32);
  const long long seq0 = s_pre[0] + static_cast<long long>(h) * nt;   // first tile of (b, h)
  const long long seg0 = (static_cast<long long>(b) * a.n_kv + h) * a.num_parts;
  const int ppt = a.part_tiles > 0 ? a.part_tiles : nt;
  const int parts = (nt + ppt - 1) / ppt;
  const float4* rec_o = reinterpret_cast<const float4*>(a.rec_o);
  float m = -INFINITY, den = 0.f;   // den: this lane's share of the sum of weights
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  int chunk = 0;                    // chunk number over all groups
  for (int p0 = 0; p0 < parts; p0 += 32) {
    long long wf;
    const int inc = partition_scan(p0 + lane, parts, seq0, ppt, nt, T, nw, narrow, lane, &wf);
    const int C = __shfl_sync(0xffffffffu, inc, 31);   // candidates of the group
    for (int k0 = 0; k0 < C; k0 += 32, ++chunk) {
      if ((chunk & 3) != warp) continue;
      const int k = k0 + lane;
      int pi = 0;   // partition of candidate k: the first with inclusive count > k
#pragma unroll
      for (int step = 16; step >= 1; step >>= 1)
        if (__shfl_sync(0xffffffffu, inc, pi + step - 1) <= k) pi += step;
      const long long wfp = __shfl_sync(0xffffffffu, wf, pi);
      const int excl = __shfl_sync(0xffffffffu, inc, pi > 0 ? pi - 1 : 0);
      const long long w = wfp + (k - (pi > 0 ? excl : 0));
      const bool ok = k < C && warp_owns_tiles(w, T, nw, narrow);
      const int rec = ok ? static_cast<int>(seg0 + p0 + pi + w) : 0;
      wait_once();
      const float lse = ok ? ld_dep_f32(a.rec_lse + static_cast<long long>(rec) * G + gg) : -INFINITY;
      const int n = min(32, C - k0);
      float4 x[16];   // records of candidates 0..15, loaded before the weights are known
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int r = __shfl_sync(0xffffffffu, rec, i);
        x[i] = i < n ? ld_dep_f32x4(rec_o + (static_cast<long long>(r) * G + gg) * (kD / 4) + lane)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float cm = lse;
      for (int o = 1; o < 32; o <<= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
      const float nm = fmaxf(m, cm);
      const float al = m == -INFINITY ? 0.f : exp2f(m - nm);
      m = nm;
      den *= al;
      acc.x *= al; acc.y *= al; acc.z *= al; acc.w *= al;
      const float wl = lse == -INFINITY ? 0.f : exp2f(lse - nm);
      den += wl;
      auto add = [&](float wg, const float4& v) {
        acc.x = wg != 0.f ? fmaf(wg, v.x, acc.x) : acc.x;
        acc.y = wg != 0.f ? fmaf(wg, v.y, acc.y) : acc.y;
        acc.z = wg != 0.f ? fmaf(wg, v.z, acc.z) : acc.z;
        acc.w = wg != 0.f ? fmaf(wg, v.w, acc.w) : acc.w;
      };
#pragma unroll
      for (int i = 0; i < 16; ++i) add(__shfl_sync(0xffffffffu, wl, i), x[i]);
      if (n > 16) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int r = __shfl_sync(0xffffffffu, rec, 16 + i);
          x[i] = 16 + i < n ? ld_dep_f32x4(rec_o + (static_cast<long long>(r) * G + gg) * (kD / 4) + lane)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) add(__shfl_sync(0xffffffffu, wl, 16 + i), x[i]);
      }
    }
  }
  wait_once();
  for (int o = 1; o < 32; o <<= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  if (lane == 0) { s_m[warp] = m; s_den[warp] = den; }
  *reinterpret_cast<float4*>(&s_acc[warp][4 * lane]) = acc;
  __syncthreads();
  float M = -INFINITY;
#pragma unroll
  for (int u = 0; u < 4; ++u) M = fmaxf(M, s_m[u]);
  float num = 0.f, dsum = 0.f;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float f = s_m[u] == -INFINITY ? 0.f : exp2f(s_m[u] - M);
    num = fmaf(f, s_acc[u][threadIdx.x], num);
    dsum = fmaf(f, s_den[u], dsum);
  }
  store_out<TO>(a.out, orow * kD + threadIdx.x, dsum > 0.f ? num / dsum : 0.f);
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
  int consumers;    // consumer warps per CTA (one producer warp besides)
  int stage_bytes;
  int desc_off;
  int qslot_bytes;
  int dyn_bytes;
};

// Consumer warps whose rings fit around the barrier block and the LUT in a
// dynamic shared-memory window of `dyn` bytes starting at `start` (the plan
// the kernel computes); 0 if the LUT itself does not fit.
int consumers_that_fit(uint32_t start, uint32_t dyn, uint32_t klut, uint32_t sb, uint32_t qbytes) {
  const uint32_t end = start + dyn;
  for (int w = kMaxConsumers; w > 0; --w) {
    const uint32_t head = kBarHead + static_cast<uint32_t>(w) * qbytes;
    const uint32_t lut = klut ? lut_at(start, klut, head) : end;
    if (klut && lut + klut > end) continue;
    if (stage_at(start + head, lut, klut, sb, w * kStages - 1) + sb <= end) return w;
  }
  return 0;
}

template <int KMODE>
bool launch_shape(int tile_bytes, int group, bool append, LaunchShape* s) {
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return false;
  s->desc_off = kChunk * tile_bytes;
  s->stage_bytes = (s->desc_off + 16 + 127) & ~127;
  const uint32_t klut = lut_bytes<KMODE>();
  // the window may start at 0 or after a small reserved area; take the worse
  const uint32_t qbytes = static_cast<uint32_t>(group) * kD * 2 + (append ? 4 * kRawRowBytes : 0u);
  s->qslot_bytes = static_cast<int>(qbytes);
  int w = consumers_that_fit(0, optin, klut, s->stage_bytes, qbytes);
  const int w2 = consumers_that_fit(1024, optin, klut, s->stage_bytes, qbytes);
  if (w2 < w) w = w2;
  if (w < 1) return false;
  s->consumers = w;
  s->dyn_bytes = optin;
  return true;
}

template <int KMODE, int GBIG, int VBITS, typename TQ, bool APPEND>
cudaError_t launch_split_typed(DecodeArgs a, cudaStream_t s, int sms) {
  LaunchShape sh;
  if (!launch_shape<KMODE>(a.tile_bytes, a.group, a.new_k != nullptr, &sh)) return cudaErrorInvalidConfiguration;
  a.stage_bytes = sh.stage_bytes;
  a.desc_off = sh.desc_off;
  a.qslot_bytes = sh.qslot_bytes;
  a.dyn_bytes = sh.dyn_bytes;
  a.qbuf_bytes = a.group * kD * 2;
  auto k = split_kernel<KMODE, GBIG, VBITS, TQ, APPEND>;
  cudaError_t err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, a.dyn_bytes);
  if (err != cudaSuccess) return err;
  return launch_pdl(k, dim3(static_cast<unsigned>(sms)), dim3((sh.consumers + kProducers) * 32),
                    static_cast<size_t>(a.dyn_bytes), s, a);
}

// The append variant is a separate instance, so the plain decode's kernel is
// compiled without any of its code.
template <int KMODE, int GBIG, int VBITS, typename TQ>
cudaError_t launch_split_append(const DecodeArgs& a, cudaStream_t s, int sms) {
  return a.new_k ? launch_split_typed<KMODE, GBIG, VBITS, TQ, true>(a, s, sms)
                 : launch_split_typed<KMODE, GBIG, VBITS, TQ, false>(a, s, sms);
}

template <int KMODE, int VBITS>
cudaError_t launch_split(const DecodeArgs& a, int q_dtype, cudaStream_t s, int sms) {
  if (q_dtype == TQ_DTYPE_BF16)
    return a.group > 4 ? launch_split_append<KMODE, 1, VBITS, __nv_bfloat16>(a, s, sms)
                       : launch_split_append<KMODE, 0, VBITS, __nv_bfloat16>(a, s, sms);
  return a.group > 4 ? launch_split_append<KMODE, 1, VBITS, __half>(a, s, sms)
                     : launch_split_append<KMODE, 0, VBITS, __half>(a, s, sms);
}

// Consumer warps per CTA of the split launch (the reduce needs the count).
int split_warps_per_cta(const tq_layout& L, int group, bool append) {
  LaunchShape sh;
  bool ok;
  if (L.key_fp8) ok = launch_shape<kFp8>(L.tile_bytes, group, append, &sh);
  else if (L.key_bits == 4) ok = launch_shape<kMse4>(L.tile_bytes, group, append, &sh);
  else ok = launch_shape<kMse3>(L.tile_bytes, group, append, &sh);
  return ok ? sh.consumers : 0;
}

tq_status run_partials(const tq_config* cfg, const tq_codebook* cb, const void* q, int q_dtype,
                       const void* cache, long long num_blocks, const int* block_table, int bt_stride,
                       const int* seq_lens, int batch, int max_seq_len, float scale, void* workspace,
                       size_t ws_bytes, unsigned int* dev_status, cudaStream_t stream,
                       const void* new_k = nullptr, const void* new_v = nullptr) {
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
  if ((new_k == nullptr) != (new_v == nullptr)) return TQ_ERR_INVALID_ARG;
  if (new_k && (!aligned16(new_k) || !aligned16(new_v))) return TQ_ERR_MISALIGNED;
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
  a.desc_off = 0;
  a.k_off = P.L.k_off;
  a.v_off = P.L.v_off;
  a.knorm_off = P.L.knorm_off;
  a.vscale_off = P.L.vscale_off;
  a.vzero_off = P.L.vzero_off;
  a.qbuf_bytes = 0;
  a.dyn_bytes = 0;
  const float sm_scale = scale > 0.f ? scale : 0.088388347648318440f;   // 1/sqrt(128)
  a.qscale = sm_scale * 1.4426950408889634f;                              // log2(e)
  a.early_indices = (cfg->flags & TQ_FLAG_INDICES_READY) ? 1 : 0;
  const float gamma = P.L.key_fp8 ? 1.f : centroid_scale(cb->centroids, cb->num_levels);
  a.qscale /= gamma;
  for (int i = 0; i < 16; ++i)
    a.cent[i] = (!P.L.key_fp8 && i < cb->num_levels) ? static_cast<float>(static_cast<double>(gamma) * cb->centroids[i]) : 0.f;
  a.new_k = new_k;
  a.new_v = new_v;
  a.wcache = new_k ? static_cast<uint8_t*>(const_cast<void*>(cache)) : nullptr;
  a.qslot_bytes = 0;
  a.k_row = P.L.k_row_bytes;
  a.v_row = P.L.v_row_bytes;
  for (int i = 0; i < 15; ++i) a.mid[i] = (!P.L.key_fp8 && i < cb->num_levels - 1) ? cb->midpoints[i] : 0.f;
  for (int i = 0; i < 16; ++i) a.scent[i] = (!P.L.key_fp8 && i < cb->num_levels) ? cb->centroids[i] : 0.f;

  cudaError_t err;
  if (P.L.key_fp8) err = launch_split<kFp8, 4>(a, q_dtype, stream, P.sms);
  else if (P.L.key_bits == 4) err = launch_split<kMse4, 4>(a, q_dtype, stream, P.sms);
  else if (P.L.value_bits == 4) err = launch_split<kMse3, 4>(a, q_dtype, stream, P.sms);
  else err = launch_split<kMse3, 3>(a, q_dtype, stream, P.sms);
  return err == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

tq_status run_reduce(const tq_config* cfg, const int* seq_lens, int batch, int max_seq_len, int bt_stride,
                     void* out, int out_dtype, const void* workspace, size_t ws_bytes, cudaStream_t stream,
                     bool after_split, bool append = false) {
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
  const int warps = split_warps_per_cta(P.L, G, append);
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
  r.early_lens = after_split ? 1 : 0;
  cudaError_t err;
  if (static_cast<long long>(batch) * cfg->num_kv_heads * 2 <= P.sms) {
    // few (sequence, KV head) pairs, many partials each: a CTA per query head
    const dim3 grid(static_cast<unsigned>(cfg->num_q_heads), static_cast<unsigned>(batch));
    const dim3 block(static_cast<unsigned>(kReduceThreads));
    if (out_dtype == TQ_DTYPE_F32) err = launch_pdl(reduce_qh_kernel<float>, grid, block, 0, stream, r);
    else if (out_dtype == TQ_DTYPE_F16) err = launch_pdl(reduce_qh_kernel<__half>, grid, block, 0, stream, r);
    else err = launch_pdl(reduce_qh_kernel<__nv_bfloat16>, grid, block, 0, stream, r);
  } else if (P.part_tiles == 0) {
    // stream-K: each pair's records are one contiguous warp range
    const dim3 grid(static_cast<unsigned>(cfg->num_kv_heads), static_cast<unsigned>(batch));
    const dim3 block(static_cast<unsigned>(G * kD));
    if (out_dtype == TQ_DTYPE_F32) err = launch_pdl(reduce_sk_kernel<float>, grid, block, 0, stream, r);
    else if (out_dtype == TQ_DTYPE_F16) err = launch_pdl(reduce_sk_kernel<__half>, grid, block, 0, stream, r);
    else err = launch_pdl(reduce_sk_kernel<__nv_bfloat16>, grid, block, 0, stream, r);
  } else {
    const dim3 grid(static_cast<unsigned>(cfg->num_kv_heads), static_cast<unsigned>(batch));
    const dim3 block(static_cast<unsigned>(G * kD));
    if (out_dtype == TQ_DTYPE_F32) err = launch_pdl(reduce_bh_kernel<float>, grid, block, 0, stream, r);
    else if (out_dtype == TQ_DTYPE_F16) err = launch_pdl(reduce_bh_kernel<__half>, grid, block, 0, stream, r);
    else err = launch_pdl(reduce_bh_kernel<__nv_bfloat16>, grid, block, 0, stream, r);
  }
  return err == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
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
                        workspace_bytes, reinterpret_cast<cudaStream_t>(stream), false);
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
                        workspace_bytes, s, true);
}

tq_status tq_decode_append(const tq_config* cfg, const tq_codebook* cb, const void* q, int q_dtype,
                           const void* new_k, const void* new_v, void* cache, long long num_blocks,
                           const int* block_table, int bt_stride, const int* seq_lens, int batch, int max_seq_len,
                           float scale, void* out, int out_dtype, void* workspace, size_t workspace_bytes,
                           unsigned int* dev_status, tq_stream_t stream) {
  if (out_dtype != TQ_DTYPE_F16 && out_dtype != TQ_DTYPE_BF16 && out_dtype != TQ_DTYPE_F32)
    return TQ_ERR_INVALID_ARG;
  if (batch > 0 && (!out || !new_k || !new_v)) return TQ_ERR_INVALID_ARG;
  if (batch > 0 && !tq::aligned16(out)) return TQ_ERR_MISALIGNED;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  tq_status st = tq::run_partials(cfg, cb, q, q_dtype, cache, num_blocks, block_table, bt_stride, seq_lens,
                                  batch, max_seq_len, scale, workspace, workspace_bytes, dev_status, s,
                                  new_k, new_v);
  if (st != TQ_OK) return st;
  return tq::run_reduce(cfg, seq_lens, batch, max_seq_len, bt_stride, out, out_dtype, workspace,
                        workspace_bytes, s, true, true);
}

}  // extern "C"
