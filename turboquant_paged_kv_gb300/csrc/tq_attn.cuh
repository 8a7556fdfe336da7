// Attention building blocks shared by the decode kernels (tq_decode.cu) and
// the multi-query continuation kernel (tq_continue.cu): PTX wrappers, the
// fp16 operand helpers, the query rotation, value-code operands, the
// centroid LUT and the host-side centroid scale. Internal, not ABI.
#ifndef TQ_ATTN_CUH_
#define TQ_ATTN_CUH_

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>
#include <mutex>
#include <type_traits>

#include "tq_launch.cuh"

namespace tq {
namespace {

constexpr uint64_t kWaitNs = 20000000;  // every wait gives up after 20 ms without progress
constexpr uint32_t kSuspendNs = 1000;     // try_wait suspend-time hint

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
  int tile_bytes, k_off, v_off, knorm_off, vscale_off, vzero_off;
  int stage_bytes;     // ring stage: kChunk tiles, then the descriptor
  int desc_off;        // offset of the descriptor in a stage
  int qbuf_bytes;      // G * d * 2: the query rows of a segment
  int qslot_bytes;     // a consumer's query slot: the query rows, then (append) two halves of raw K and V rows
  int dyn_bytes;
  float qscale;        // softmax scale * log2(e)
  int early_indices;   // TQ_FLAG_INDICES_READY: lengths and block ids read before the dependency wait
  float cent[16];
  // append (tq_decode_append; new_k null: off): each sequence's newest token,
  // position seq_lens[b] - 1, is quantised and written into the cache by the
  // consumer warp that reads its tile
  const void* new_k;   // [batch][n_kv][d], the query's dtype
  const void* new_v;
  uint8_t* wcache;     // the cache, writable
  int k_row, v_row;    // bytes per position of the key and value regions
  float mid[15];       // key codebook midpoints and centroids (unscaled)
  float scent[16];
};

struct ReduceArgs {
  const int* seq_lens;
  const float* rec_o;
  const float* rec_lse;
  void* out;
  int batch, n_q, n_kv, group, part_tiles, num_parts, max_seq_len, cap, num_warps;
  int early_lens;   // launched right after the split kernel of the same decode
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
__device__ __forceinline__ void sts32(uint32_t a, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;\n" ::"r"(a), "r"(v));
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
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
  return t;
}
// Bounded wait for the phase of parity `parity`: returns false once kWaitNs
// have passed without it completing.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  do {
    if (mbar_try(bar, parity)) return true;
  } while (global_ns() - t0 < kWaitNs);
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

// *p if pred, else dflt: a predicated load into a preset register, so nothing
// consumes the loaded value here and the warp does not wait for it (a select
// on the loaded value would); the address is not touched when !pred. L2 only,
// like every load of data another kernel may write (tq_launch.cuh).
__device__ __forceinline__ int ldg_or(const int* p, bool pred, int dflt) {
  int v = dflt;
  asm volatile("{\n .reg .pred q;\n setp.ne.u32 q, %2, 0;\n @q ld.global.cg.b32 %0, [%1];\n}\n"
               : "+r"(v)
               : "l"(p), "r"(static_cast<unsigned>(pred)));
  return v;
}

__device__ __forceinline__ void flag(unsigned int* status, unsigned int bit) {
  if (status) atomicOr(status, bit);
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// w >> n for n >= 0, w << -n otherwise (n is a compile-time constant here).
__device__ __forceinline__ uint32_t shift_right(uint32_t w, int n) { return n >= 0 ? w >> n : w << -n; }

// Value codes as mma A operands. The cache interleaves the 16-bit words of a
// token pair, so a 32-bit word holds the same 16-bit word of both tokens, and
// one mask turns code t of this lane into a half2 of the two tokens' codes as
// exact fp16 subnormals at bit p (value code * 2^(p - 24)). x[] holds the
// lane's words of one pair:
//   4-bit: x[k] = word 4 g + k (coordinates 16 g + 4 k .. + 3), code t at bit 4 t;
//   3-bit: x[k] = word 3 g + k (48 bits from bit 48 g), code t at bit 3 t, where
//          codes 5 and 10 straddle two words and take one bit field from each.
template <int VBITS>
__device__ __forceinline__ uint32_t code_field(const uint4& x, int t, int p) {
  if constexpr (VBITS == 4) {
    return shift_right(word_of(x, t >> 2), 4 * (t & 3) - p) & (0x000F000Fu << p);
  } else {
    const int bit = 3 * t, wi = bit >> 4, s = bit & 15;
    if (s <= 13) return shift_right(word_of(x, wi), s - p) & (0x00070007u << p);
    const int nlo = 16 - s, nhi = 3 - nlo;   // bits from word wi, from word wi + 1
    return (shift_right(word_of(x, wi), s - p) & ((((1u << nlo) - 1) << p) * 0x10001u)) |
           (shift_right(word_of(x, wi + 1), -(nlo + p)) & ((((1u << nhi) - 1) << (p + nlo)) * 0x10001u));
  }
}

// ---------------------------------------------------------------- LUT

// Entry e (a key byte, or a 6-bit pair of 3-bit indices) holds 32 copies of
// half2(c'[lo idx], c'[hi idx]), one per lane, so a warp's lookups never
// conflict; c' = fp16(gamma * c), gamma the per-codebook scale chosen on the
// host (the query is divided by it). Entry stride 256 bytes, of which the
// copies fill 128. The table is aligned to its own size, so the address of
// (entry, lane) is the entry number OR-ed into bits 8.. of the lane's base: for
// 4-bit keys a single byte permute of the key word.
template <int KMODE>
__host__ __device__ constexpr uint32_t lut_bytes() { return KMODE == kMse4 ? 65536u : (KMODE == kMse3 ? 16384u : 0u); }

template <int KMODE>
__device__ void build_lut(uint32_t lut, const float* cent, int tid, int nthreads) {
  constexpr int kEntries = KMODE == kMse4 ? 256 : 64;
  constexpr int kShift = KMODE == kMse4 ? 4 : 3;
  constexpr int kMask = (1 << kShift) - 1;
  for (int i = tid; i < kEntries * 32; i += nthreads) {
    const int e = i >> 5;
    sts32(lut + 256u * e + 4u * (i & 31), pack_half2(cent[e & kMask], cent[(e >> kShift) & kMask]));
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

// ---------------------------------------------------------------- host

// fp16 round-to-nearest-even of a double in the fp16 normal or subnormal range.
double round_fp16(double x) {
  if (x == 0.0) return 0.0;
  int e = 0;
  const double f = std::frexp(x, &e);   // x = f 2^e, 0.5 <= |f| < 1
  if (e <= -14) return std::ldexp(std::nearbyint(std::ldexp(x, 24)), -24);   // subnormal: steps of 2^-24
  return std::ldexp(std::nearbyint(std::ldexp(f, 11)), e - 11);              // 11 significant bits
}

// The decode holds the centroids c as fp16(gamma c) and divides the query by
// gamma, so its scores carry only the rounding of gamma c. gamma is the step of
// [1, 2) (2^-16 grid) whose largest relative rounding error over the nonzero
// centroids is smallest: for the d = 128, 4-bit codebook about 9e-5 against
// 3.5e-4 at gamma = 1. Memoised per codebook (the search takes a few ms).
float centroid_scale(const float* c, int n) {
  static std::mutex mu;
  struct Memo { int n; float c[16]; float g; };
  static Memo memo[8];
  static int used = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int m = 0; m < used; ++m) {
    bool same = memo[m].n == n;
    for (int i = 0; same && i < n; ++i) same = memo[m].c[i] == c[i];
    if (same) return memo[m].g;
  }
  double best_err = 1e300;
  float best = 1.f;
  for (int step = 0; step < 65536; ++step) {
    const float g = 1.f + static_cast<float>(step) * (1.f / 65536.f);
    double err = 0.0;
    for (int i = 0; i < n && err < best_err; ++i) {
      if (c[i] == 0.f) continue;
      const double x = static_cast<double>(static_cast<float>(static_cast<double>(g) * c[i]));
      err = std::fmax(err, std::fabs(round_fp16(x) - static_cast<double>(g) * c[i]) / std::fabs(static_cast<double>(g) * c[i]));
    }
    if (err < best_err) { best_err = err; best = g; }
  }
  Memo& slot = memo[used < 8 ? used++ : 7];
  slot.n = n;
  for (int i = 0; i < 16; ++i) slot.c[i] = i < n ? c[i] : 0.f;
  slot.g = best;
  return best;
}

}  // namespace
}  // namespace tq

#endif  // TQ_ATTN_CUH_
