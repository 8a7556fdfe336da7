// tq_dequant: the cached keys and values of whole sequences expanded back to
// 16- or 32-bit vectors in the original (unrotated) basis.
//
// Method: "vLLM 源码完全拆解(十九):TurboQuant KV Cache 量化" (pinghaoyang.com.cn),
// section "续写 prefill:小 chunk 走 decode,大 chunk 走反量化", subsection
// "反量化 kernel:_tq_full_dequant_kv": every cached (position, KV head) slot is
// unpacked exactly as the decode unpacks it, with no softmax, and the keys are
// rotated back. The rotation H / sqrt(d) is symmetric and orthonormal (section
// "为什么先旋转"), so it is its own inverse:
//   index-coded keys  k = stored_norm * (H / sqrt(d)) c[idx]
//   FP8 keys          k = e4m3 value (never rotated)
//   values            v = fp16(scale) * code + fp16(zero)
//
// Differences from the pages' design: the pages expand to fp16 in one kernel
// and then rotate back with an fp16 matrix product against a copy of the
// Hadamard matrix; here a half-warp per (position, KV head) holds the 128
// coordinates in registers (8 per lane), applies the inverse rotation as an
// fp32 butterfly (3 in-lane stages + 4 xor-shuffle stages) and rounds once, to
// the caller's output type. Nothing intermediate is written.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "tq_internal.h"
#include "tq_launch.cuh"

namespace tq {
namespace {

constexpr int kDequantWarps = 8;
constexpr int kD = 128;

struct DequantArgs {
  const uint8_t* cache;
  const int* block_table;
  const int* seq_lens;
  void* key_out;
  void* value_out;
  unsigned int* status;
  long long num_blocks;
  int n_kv;
  int max_seq_len;
  int batch;
  int len_cap;               // min(max_seq_len, bt_stride * block_size)
  int seq_tiles;             // ceil(max_seq_len / 16): CTAs per (sequence, KV head)
  int bt_stride;
  int log2_bs;
  int tiles_per_block;
  int tile_bytes;
  int k_off, k_row;
  int v_off, v_row;
  int knorm_off, vscale_off, vzero_off;
  float cent[16];
};

enum KeyMode { kMse4 = 4, kMse3 = 3, kFp8 = 8 };

// Sylvester-order Walsh-Hadamard transform of 128 coordinates held by a
// half-warp, 8 consecutive values per lane (coordinate 8 * l + j for lane l of
// the half), unnormalised: coordinate strides 1, 2, 4 inside the lane, then
// 8 .. 64 across lanes l ^ 1 .. l ^ 8. The lane whose stride bit is set keeps
// (partner - own), the other (own + partner); both as one exact fma with +-1.
__device__ __forceinline__ void fwht128_half(float v[8], int l) {
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j & h) continue;
      const float a = v[j], b = v[j + h];
      v[j] = a + b;
      v[j + h] = a - b;
    }
  }
#pragma unroll
  for (int m = 1; m <= 8; m <<= 1) {
    const float sgn = (l & m) ? -1.f : 1.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = fmaf(sgn, v[j], __shfl_xor_sync(0xffffffffu, v[j], m));
  }
}

template <typename T>
__device__ __forceinline__ void store8(void* base, long long elem, const float x[8]) {
  if constexpr (std::is_same<T, float>::value) {
    float4* d = reinterpret_cast<float4*>(static_cast<float*>(base) + elem);
    d[0] = make_float4(x[0], x[1], x[2], x[3]);
    d[1] = make_float4(x[4], x[5], x[6], x[7]);
  } else {
    uint4 w;
    uint32_t* wp = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if constexpr (std::is_same<T, __nv_bfloat16>::value) {
        const __nv_bfloat162 t = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
        wp[i] = *reinterpret_cast<const uint32_t*>(&t);
      } else {
        const __half2 t = __floats2half2_rn(x[2 * i], x[2 * i + 1]);
        wp[i] = *reinterpret_cast<const uint32_t*>(&t);
      }
    }
    *reinterpret_cast<uint4*>(static_cast<T*>(base) + elem) = w;
  }
}

__device__ __forceinline__ float half_bits(const uint8_t* p) {
  return __half2float(__ushort_as_half(ld_dep_u16(p)));
}

// One CTA per (sequence, 16-position tile, KV head): grid (seq_tiles * batch,
// n_kv). Warp w expands positions 2w and 2w + 1 of the tile, one per
// half-warp; lane l of a half holds coordinates 8l .. 8l + 7.
template <int KMODE, int VBITS, typename T>
__global__ void __launch_bounds__(kDequantWarps * 32)
dequant_kernel(const DequantArgs a) {
  grid_dep_wait();   // cache, tables and lengths may come from the previous kernel
  grid_dep_launch();
  __shared__ float s_cent[16];
  if (threadIdx.x < 16) s_cent[threadIdx.x] = a.cent[threadIdx.x];
  __syncthreads();

  const int b = static_cast<int>(blockIdx.x / static_cast<unsigned>(a.seq_tiles));
  const int t = static_cast<int>(blockIdx.x - static_cast<unsigned>(b) * static_cast<unsigned>(a.seq_tiles));
  const int h = blockIdx.y;
  const int lane = threadIdx.x & 31;
  const int l = lane & 15;
  const int r = 2 * (threadIdx.x >> 5) + (lane >> 4);   // row of the tile
  const int p = 16 * t + r;
  // rows past max_seq_len (the last tile) are not in the output; their lanes
  // stay to the end, since the butterfly's shuffles need the whole warp
  const bool in_out = p < a.max_seq_len;
  const long long elem = ((static_cast<long long>(b) * a.max_seq_len + p) * a.n_kv + h) * kD + 8 * l;

  const int raw_len = ld_dep_s32(a.seq_lens + b);
  if (p == 0 && h == 0 && lane == 0 && raw_len > a.len_cap && a.status) atomicOr(a.status, TQ_DEV_SEQ_TOO_LONG);
  const int len = min(max(raw_len, 0), a.len_cap);
  float k[8], v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) k[j] = v[j] = 0.f;
  // the whole tile lies in one cache block; its id is read only if the tile
  // holds a cached position
  int blk = -1;
  if (16 * t < len) {
    blk = ld_dep_s32(a.block_table + static_cast<long long>(b) * a.bt_stride + ((16 * t) >> a.log2_bs));
    if ((blk < 0 || blk >= a.num_blocks) && threadIdx.x == 0 && a.status) atomicOr(a.status, TQ_DEV_BLOCK_OUT_OF_RANGE);
  }
  const bool live = p < len && blk >= 0 && blk < a.num_blocks;
  if (live) {
    const int off = (16 * t) & ((1 << a.log2_bs) - 1);
    const uint8_t* tile = a.cache + ((static_cast<long long>(blk) * a.n_kv + h) * a.tiles_per_block + (off >> 4)) *
                                        static_cast<long long>(a.tile_bytes);
    const uint8_t* krow = tile + a.k_off + r * a.k_row;
    if constexpr (KMODE == kFp8) {
      const uint2 w = ld_dep_u32x2(krow + 8 * l);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t word = i < 2 ? w.x : w.y;
        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(
            static_cast<__nv_fp8x2_storage_t>((word >> (16 * (i & 1))) & 0xFFFFu), __NV_E4M3);
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
        k[2 * i] = f.x;
        k[2 * i + 1] = f.y;
      }
    } else {
      uint32_t w;
      if constexpr (KMODE == kMse4) {
        w = ld_dep_u32(krow + 4 * l);
      } else {
        const uint8_t* g = krow + 3 * l;   // 24 bits, LSB first
        w = ld_dep_u8(g) | (ld_dep_u8(g + 1) << 8) | (ld_dep_u8(g + 2) << 16);
      }
      const float nrm = half_bits(tile + a.knorm_off + 2 * r);
#pragma unroll
      for (int j = 0; j < 8; ++j) k[j] = nrm * s_cent[(w >> (KMODE * j)) & ((1u << KMODE) - 1)];
    }
    const int pair = r >> 1;
    uint32_t codes;   // this lane's codes, LSB-first: coordinate 8 l + j at bit VBITS j
    if constexpr (VBITS == 4) {
      // value words 2l and 2l + 1 of token r = 2 * pair + (r & 1): one 8-byte
      // group holding both words of both tokens of the pair (pair-interleaved,
      // 16-byte groups swizzled by the pair index when rows are 64 bytes)
      const int swz = (a.v_row % 64 == 0) ? 2 * (pair & 3) : 0;
      const uint2 vw = ld_dep_u32x2(tile + a.v_off + pair * 2 * a.v_row + 16 * ((l >> 1) ^ swz) + 8 * (l & 1));
      codes = ((vw.x >> (16 * (r & 1))) & 0xFFFFu) | (((vw.y >> (16 * (r & 1))) & 0xFFFFu) << 16);
    } else {
      // 24 bits from bit 24 l of the token's stream: 16-bit words 3 m and
      // 3 m + 1 (l = 2 m, bits 0-23 of the pair) or 3 m + 1 and 3 m + 2 (l =
      // 2 m + 1, bits 8-31); the pair's 32-bit word i (no swizzle at 48-byte
      // rows) holds word i of both tokens
      const int w0 = 3 * (l >> 1) + (l & 1);
      const uint8_t* pw = tile + a.v_off + pair * 2 * a.v_row + 4 * w0;
      const int sh = 16 * (r & 1);
      const uint32_t lo = (ld_dep_u32(pw) >> sh) & 0xFFFFu, hi = (ld_dep_u32(pw + 4) >> sh) & 0xFFFFu;
      codes = (lo | (hi << 16)) >> (8 * (l & 1));
    }
    const float s = half_bits(tile + a.vscale_off + 2 * r);
    const float z = half_bits(tile + a.vzero_off + 2 * r);
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = fmaf(s, static_cast<float>((codes >> (VBITS * j)) & ((1u << VBITS) - 1)), z);
  }
  if constexpr (KMODE != kFp8) {
    // every half-warp of the warp runs the butterfly (its shuffles need all
    // 32 lanes); rows that hold no key transform zeros
    fwht128_half(k, l);
#pragma unroll
    for (int j = 0; j < 8; ++j) k[j] *= 0.088388347648318440f;   // 1 / sqrt(128)
  }
  if (in_out) {
    store8<T>(a.key_out, elem, k);
    store8<T>(a.value_out, elem, v);
  }
}

// ---------------------------------------------------------------- tensor-core form
//
// Index-coded keys, a warp per (sequence, 16-position tile, KV head). The
// inverse rotation H / sqrt(128) is a Kronecker product: with the 7 bits of a
// coordinate split into R = {0, 1, 5, 6} and S = {2, 3, 4},
//   H[a][b] = (-1)^popc(a & b) = H_R[a_R][b_R] * H_S[a_S][b_S],
// so the 16 x 128 tile of rotated-basis keys C (rows: positions, C = c[idx])
// is multiplied by H_R on tensor cores, one m16n8k16 per (S-block, 8 output
// columns), and by H_S with a 3-stage butterfly over the 8 S-blocks held in
// registers. Lane (g, t) holds the key bytes of rows g and g + 8 for
// coordinates 32 t .. 32 t + 31, which is the decode's QK operand layout: in
// S-block s its operand pairs are coordinates 32 t + 4 s + {0, 1} and
// + {2, 3}, so the mma's k index kappa = e0 + 2 t + 8 e1 stands for a_R bits
// (a0 = e0, a5 a6 = t, a1 = e1). The centroids enter as fp16 hi + lo parts
// from a LUT (one 8-byte entry per key byte: both parts of both centroids, 32
// copies so lookups never conflict), the H_R entries as exact fp16 +-1; the
// only roundings are fp32 sums. Output column n = x + 2 t + 8 nt of S-block
// s' is coordinate b = x + 2 (t & 1) + 32 (t >> 1) + 64 nt + 4 s'. Results
// are multiplied by stored_norm / sqrt(128), staged per warp in shared memory
// and written back as full rows. Values are expanded in the same pass with a
// row-major lane map (lane: token pair lane >> 2, coordinates 8 (lane & 3) +
// 32 k), so their 16-byte stores cover whole sectors.

template <int KMODE>
__host__ __device__ constexpr int lut_entries() { return KMODE == kMse4 ? 256 : 64; }

// LUT entry index of operand step `st` (coordinates 32 t + 2 st, + 1) of this
// lane's key slice kq: a key byte (4-bit keys) or a 6-bit pair (3-bit keys).
template <int KMODE>
__device__ __forceinline__ uint32_t key_entry(const uint4& kq, int st) {
  const uint32_t w[4] = {kq.x, kq.y, kq.z, kq.w};
  if constexpr (KMODE == kMse4) {
    return (w[st >> 2] >> (8 * (st & 3))) & 0xFFu;
  } else {
    const int bit = 6 * st, wi = bit >> 5, sh = bit & 31;
    const uint32_t f = sh <= 26 ? (w[wi] >> sh) : __funnelshift_r(w[wi], w[wi + 1], sh);
    return f & 0x3Fu;
  }
}

__device__ __forceinline__ void mma16816(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <typename T>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    const __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&t);
  } else {
    const __half2 t = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&t);
  }
}

// Codes of coordinates 8 l .. 8 l + 7 of token j (0, 1) of the pair, LSB first.
template <int VBITS>
__device__ __forceinline__ uint32_t token_codes(uint2 vw, int j, int l) {
  const int sh = 16 * j;
  if constexpr (VBITS == 4) {
    return ((vw.x >> sh) & 0xFFFFu) | (((vw.y >> sh) & 0xFFFFu) << 16);
  } else {
    return (((vw.x >> sh) & 0xFFFFu) | (((vw.y >> sh) & 0xFFFFu) << 16)) >> (8 * (l & 1));
  }
}

template <typename T>
__host__ __device__ constexpr int dq_warps() { return sizeof(T) == 4 ? 8 : 16; }   // shared memory per CTA
constexpr int kMaxTileBytes = 2144;   // largest index-coded-key tile (4bit_nc)

// The 8-byte value words of token pair `pair` (tile in shared memory) that
// hold, for both tokens, the codes of coordinates 8 l .. 8 l + 7.
template <int VBITS>
__device__ __forceinline__ uint2 value_pair_words_s(const uint8_t* tile, const DequantArgs& a, int pair, int l) {
  if constexpr (VBITS == 4) {
    const int swz = (a.v_row % 64 == 0) ? 2 * (pair & 3) : 0;
    return *reinterpret_cast<const uint2*>(tile + a.v_off + pair * 2 * a.v_row + 16 * ((l >> 1) ^ swz) + 8 * (l & 1));
  } else {
    const int w0 = 3 * (l >> 1) + (l & 1);
    const uint32_t* pw = reinterpret_cast<const uint32_t*>(tile + a.v_off + pair * 2 * a.v_row + 4 * w0);
    return make_uint2(pw[0], pw[1]);
  }
}

// Where tile u of the (sequence, tile, KV head) order lives. The length and
// block id are loaded here and used a tile later, so the loads overlap work.
struct DqTile {
  int b, tl, h, raw_len, blk;   // blk: -2 when no entry is read
};

__device__ __forceinline__ DqTile dq_resolve(const DequantArgs& a, unsigned u, unsigned total) {
  DqTile r{0, 0, 0, 0, -2};
  if (u < total) {
    const unsigned bt = u / static_cast<unsigned>(a.n_kv);
    r.h = static_cast<int>(u - bt * static_cast<unsigned>(a.n_kv));
    r.b = static_cast<int>(bt / static_cast<unsigned>(a.seq_tiles));
    r.tl = static_cast<int>(bt - static_cast<unsigned>(r.b) * static_cast<unsigned>(a.seq_tiles));
    r.raw_len = ld_dep_s32(a.seq_lens + r.b);
    if (16 * r.tl < a.len_cap)
      r.blk = ld_dep_s32(a.block_table + static_cast<long long>(r.b) * a.bt_stride + ((16 * r.tl) >> a.log2_bs));
  }
  return r;
}

// The tile's address (null when it holds no cached position) and its number of
// cached rows; flags a bad block id or an over-long length (lane 0).
__device__ __forceinline__ const uint8_t* dq_address(const DequantArgs& a, const DqTile& r, int lane, int* live) {
  const int len = min(max(r.raw_len, 0), a.len_cap);
  if (lane == 0 && r.tl == 0 && r.h == 0 && r.raw_len > a.len_cap && a.status) atomicOr(a.status, TQ_DEV_SEQ_TOO_LONG);
  *live = 0;
  if (16 * r.tl >= len) return nullptr;
  if (r.blk < 0 || r.blk >= a.num_blocks) {
    if (lane == 0 && a.status) atomicOr(a.status, TQ_DEV_BLOCK_OUT_OF_RANGE);
    return nullptr;
  }
  *live = min(16, len - 16 * r.tl);
  return a.cache + ((static_cast<long long>(r.blk) * a.n_kv + r.h) * a.tiles_per_block +
                    (((16 * r.tl) & ((1 << a.log2_bs) - 1)) >> 4)) * static_cast<long long>(a.tile_bytes);
}

__device__ __forceinline__ void dq_copy(uint8_t* slot, const uint8_t* src, int chunks, int lane) {
  if (src) {
    for (int c = lane; c < chunks; c += 32) {
      const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(slot + 16 * c));
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(src + 16 * c) : "memory");
    }
  }
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}

// Persistent: warp w of CTA c takes tiles c * warps + w, + all warps, ...; each
// tile's bytes arrive by cp.async in one of two per-warp slots while the
// previous tile is computed.
template <int KMODE, int VBITS, typename T>
__global__ void __launch_bounds__(dq_warps<T>() * 32, 1) dequant_mma_kernel(const DequantArgs a) {
  extern __shared__ __align__(16) uint8_t s_dq[];
  constexpr int kWarpsT = dq_warps<T>();
  constexpr int kRow = kD * static_cast<int>(sizeof(T)) + 16;   // staging row stride (bytes)
  uint2* lut = reinterpret_cast<uint2*>(s_dq);                   // [entry][lane]: (hi, lo) half2 pair
  grid_dep_wait();   // cache, tables and lengths may come from the previous kernel
  grid_dep_launch();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, t = lane & 3;
  uint8_t* stage = s_dq + lut_entries<KMODE>() * 32 * 8 + warp * (16 * kRow + 2 * kMaxTileBytes);
  uint8_t* slots = stage + 16 * kRow;
  constexpr int kShift = KMODE == kMse4 ? 4 : 3;
  for (int i = tid; i < lut_entries<KMODE>() * 32; i += blockDim.x) {
    const int e = i >> 5;
    const float c0 = a.cent[e & ((1 << kShift) - 1)], c1 = a.cent[e >> kShift];
    const __half h0 = __float2half_rn(c0), h1 = __float2half_rn(c1);
    const __half l0 = __float2half_rn(c0 - __half2float(h0)), l1 = __float2half_rn(c1 - __half2float(h1));
    lut[i] = make_uint2(static_cast<uint32_t>(__half_as_ushort(h0)) | (static_cast<uint32_t>(__half_as_ushort(h1)) << 16),
                        static_cast<uint32_t>(__half_as_ushort(l0)) | (static_cast<uint32_t>(__half_as_ushort(l1)) << 16));
  }
  // B operands: H_R[kappa][n] = (-1)^(k0 n0 + k3 n1 + k1 n2 + k2 n3), kappa = 2 t + {0, 1} (+ 8), n = 8 nt + g
  uint32_t hb[2][2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      uint32_t v = 0;
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int k = 2 * t + x + 8 * r, n = 8 * nt + g;
        const int par = ((k & 1) & (n & 1)) ^ (((k >> 3) & 1) & ((n >> 1) & 1)) ^ (((k >> 1) & 1) & ((n >> 2) & 1)) ^
                        (((k >> 2) & 1) & ((n >> 3) & 1));
        v |= (par ? 0xBC00u : 0x3C00u) << (16 * x);
      }
      hb[nt][r] = v;
    }
  }
  __syncthreads();   // LUT

  // tiles in (sequence, tile, KV head) order, so neighbouring warps write neighbouring output rows
  const unsigned total = static_cast<unsigned>(a.seq_tiles) * static_cast<unsigned>(a.batch) * static_cast<unsigned>(a.n_kv);
  const unsigned nwarps = gridDim.x * kWarpsT;
  const int chunks = a.tile_bytes >> 4;
  unsigned u = blockIdx.x * kWarpsT + warp;
  DqTile cur = dq_resolve(a, u, total);
  int cur_live = 0;
  const uint8_t* cur_src = dq_address(a, cur, lane, &cur_live);
  dq_copy(slots, cur_src, chunks, lane);
  DqTile nxt = dq_resolve(a, u + nwarps, total);
  for (int i = 0; u < total; ++i, u += nwarps) {
    // next tile's copies, the one after's indices
    int nxt_live = 0;
    const uint8_t* nxt_src = u + nwarps < total ? dq_address(a, nxt, lane, &nxt_live) : nullptr;
    dq_copy(slots + ((i + 1) & 1) * kMaxTileBytes, nxt_src, chunks, lane);
    const DqTile nn = dq_resolve(a, u + 2 * nwarps, total);
    asm volatile("cp.async.wait_group 1;\n" ::: "memory");   // this lane's copies of tile i
    __syncwarp();                                              // and every lane's
    const uint8_t* tile = slots + (i & 1) * kMaxTileBytes;
    const int live = cur_live, b = cur.b, h = cur.h, p0 = 16 * cur.tl;

    // ---- keys: C . H_R on tensor cores, then H_S across the 8 S-blocks
    float d[8][2][4];
#pragma unroll
    for (int s2 = 0; s2 < 8; ++s2)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) d[s2][nt][0] = d[s2][nt][1] = d[s2][nt][2] = d[s2][nt][3] = 0.f;
    float ng = 0.f, nh = 0.f;
    if (live > 0) {
      uint4 kg, kh;
      const uint8_t* kr = tile + a.k_off;
      if constexpr (KMODE == kMse4) {
        kg = *reinterpret_cast<const uint4*>(kr + g * a.k_row + 16 * t);
        kh = *reinterpret_cast<const uint4*>(kr + (g + 8) * a.k_row + 16 * t);
      } else {
        const uint32_t* ra = reinterpret_cast<const uint32_t*>(kr + g * a.k_row + 12 * t);
        const uint32_t* rb = reinterpret_cast<const uint32_t*>(kr + (g + 8) * a.k_row + 12 * t);
        kg = make_uint4(ra[0], ra[1], ra[2], 0u);
        kh = make_uint4(rb[0], rb[1], rb[2], 0u);
      }
      if (g < live) ng = __half2float(*reinterpret_cast<const __half*>(tile + a.knorm_off + 2 * g));
      if (g + 8 < live) nh = __half2float(*reinterpret_cast<const __half*>(tile + a.knorm_off + 2 * (g + 8)));
#pragma unroll
      for (int s2 = 0; s2 < 8; ++s2) {
        const uint2 eg0 = lut[key_entry<KMODE>(kg, 2 * s2) * 32 + lane];
        const uint2 eh0 = lut[key_entry<KMODE>(kh, 2 * s2) * 32 + lane];
        const uint2 eg1 = lut[key_entry<KMODE>(kg, 2 * s2 + 1) * 32 + lane];
        const uint2 eh1 = lut[key_entry<KMODE>(kh, 2 * s2 + 1) * 32 + lane];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          mma16816(d[s2][nt], eg0.x, eh0.x, eg1.x, eh1.x, hb[nt][0], hb[nt][1]);
          mma16816(d[s2][nt], eg0.y, eh0.y, eg1.y, eh1.y, hb[nt][0], hb[nt][1]);
        }
      }
    }
    // H_S: Sylvester butterfly over the S-block index
#pragma unroll
    for (int m = 1; m < 8; m <<= 1)
#pragma unroll
      for (int s2 = 0; s2 < 8; ++s2) {
        if (s2 & m) continue;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float x0 = d[s2][nt][e], x1 = d[s2 + m][nt][e];
            d[s2][nt][e] = x0 + x1;
            d[s2 + m][nt][e] = x0 - x1;
          }
      }
    // stored_norm / sqrt(128) (zero for rows without a cached position), staged row-major
    const float fg = ng * 0.088388347648318440f, fh = nh * 0.088388347648318440f;
#pragma unroll
    for (int s2 = 0; s2 < 8; ++s2)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int col = 2 * (t & 1) + 32 * (t >> 1) + 64 * nt + 4 * s2;   // coordinates col, col + 1
        uint8_t* rg = stage + g * kRow + col * static_cast<int>(sizeof(T));
        uint8_t* rh = stage + (g + 8) * kRow + col * static_cast<int>(sizeof(T));
        if constexpr (std::is_same<T, float>::value) {
          *reinterpret_cast<float2*>(rg) = make_float2(d[s2][nt][0] * fg, d[s2][nt][1] * fg);
          *reinterpret_cast<float2*>(rh) = make_float2(d[s2][nt][2] * fh, d[s2][nt][3] * fh);
        } else {
          *reinterpret_cast<uint32_t*>(rg) = pack2<T>(d[s2][nt][0] * fg, d[s2][nt][1] * fg);
          *reinterpret_cast<uint32_t*>(rh) = pack2<T>(d[s2][nt][2] * fh, d[s2][nt][3] * fh);
        }
      }

    // ---- values: lane (pair lane >> 2, q = lane & 3) expands coordinates 8 q + 32 k of both tokens
    const int pair = lane >> 2, q = lane & 3;
    float sv[2] = {0.f, 0.f}, zv[2] = {0.f, 0.f};
    uint2 vw[4] = {};
    if (live > 0) {
#pragma unroll
      for (int k = 0; k < 4; ++k) vw[k] = value_pair_words_s<VBITS>(tile, a, pair, q + 4 * k);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        if (2 * pair + j < live) {
          sv[j] = __half2float(*reinterpret_cast<const __half*>(tile + a.vscale_off + 2 * (2 * pair + j)));
          zv[j] = __half2float(*reinterpret_cast<const __half*>(tile + a.vzero_off + 2 * (2 * pair + j)));
        }
      }
    }
    __syncwarp();   // staged key rows complete; every lane has read the slot
    // whole key rows out: 16 rows x 128 coordinates, 16 bytes a lane
    constexpr int kChunks = kD * static_cast<int>(sizeof(T)) / 16;   // 16-byte chunks per row
#pragma unroll
    for (int i2 = 0; i2 < 16 * kChunks / 32; ++i2) {
      const int c = i2 * 32 + lane, r = c / kChunks, k = c - r * kChunks;
      const int p = p0 + r;
      if (p < a.max_seq_len) {
        const uint4 v = *reinterpret_cast<const uint4*>(stage + r * kRow + 16 * k);
        *reinterpret_cast<uint4*>(static_cast<T*>(a.key_out) +
                                  ((static_cast<long long>(b) * a.max_seq_len + p) * a.n_kv + h) * kD + k * 16 / sizeof(T)) = v;
      }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int p = p0 + 2 * pair + j;
      const bool row_live = 2 * pair + j < live;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t codes = token_codes<VBITS>(vw[k], j, q + 4 * k);
        float v[8];
#pragma unroll
        for (int i3 = 0; i3 < 8; ++i3)
          v[i3] = row_live ? fmaf(sv[j], static_cast<float>((codes >> (VBITS * i3)) & ((1u << VBITS) - 1)), zv[j]) : 0.f;
        if (p < a.max_seq_len)
          store8<T>(a.value_out, ((static_cast<long long>(b) * a.max_seq_len + p) * a.n_kv + h) * kD + 8 * (q + 4 * k), v);
      }
    }
    __syncwarp();   // the staged rows have been read before the next tile writes them
    cur = nxt;
    cur_live = nxt_live;
    nxt = nn;
  }
  asm volatile("cp.async.wait_all;\n" ::: "memory");   // no copy outlives the CTA
}

template <int KMODE, int VBITS, typename T>
cudaError_t launch_dequant_mma(const DequantArgs& a, int batch, cudaStream_t stream) {
  if (a.tile_bytes > kMaxTileBytes) return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(lut_entries<KMODE>()) * 32 * 8 +
                      static_cast<size_t>(dq_warps<T>()) * (16 * (kD * sizeof(T) + 16) + 2 * kMaxTileBytes);
  auto k = dequant_mma_kernel<KMODE, VBITS, T>;
  cudaError_t err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  int dev = 0, sms = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
  const long long total = static_cast<long long>(a.seq_tiles) * batch * a.n_kv;
  const long long want = (total + dq_warps<T>() - 1) / dq_warps<T>();
  return launch_pdl(k, dim3(static_cast<unsigned>(want < sms ? want : sms)), dim3(dq_warps<T>() * 32), smem, stream, a);
}

template <int KMODE, int VBITS>
cudaError_t launch_dequant(const DequantArgs& a, int batch, int out_dtype, cudaStream_t stream) {
  if constexpr (KMODE != kFp8) {   // index-coded keys: the tensor-core form
    if (out_dtype == TQ_DTYPE_BF16) return launch_dequant_mma<KMODE, VBITS, __nv_bfloat16>(a, batch, stream);
    if (out_dtype == TQ_DTYPE_F16) return launch_dequant_mma<KMODE, VBITS, __half>(a, batch, stream);
    return launch_dequant_mma<KMODE, VBITS, float>(a, batch, stream);
  }
  const dim3 grid(static_cast<unsigned>(static_cast<long long>(a.seq_tiles) * batch), static_cast<unsigned>(a.n_kv));
  const dim3 block(kDequantWarps * 32);
  if (out_dtype == TQ_DTYPE_BF16)
    return launch_pdl(dequant_kernel<KMODE, VBITS, __nv_bfloat16>, grid, block, 0, stream, a);
  if (out_dtype == TQ_DTYPE_F16) return launch_pdl(dequant_kernel<KMODE, VBITS, __half>, grid, block, 0, stream, a);
  return launch_pdl(dequant_kernel<KMODE, VBITS, float>, grid, block, 0, stream, a);
}

}  // namespace
}  // namespace tq

extern "C" tq_status tq_dequant(const tq_config* cfg, const tq_codebook* cb,
                                const void* cache, long long num_blocks,
                                const int* block_table, int bt_stride,
                                const int* seq_lens, int batch, int max_seq_len,
                                void* key_out, void* value_out, int out_dtype,
                                unsigned int* dev_status, tq_stream_t stream) {
  using namespace tq;
  tq_layout L;
  const tq_status st = make_layout(cfg, &L);
  if (st != TQ_OK) return st;
  if (batch < 0 || max_seq_len < 0 || num_blocks < 0 || bt_stride < 1) return TQ_ERR_INVALID_ARG;
  if (out_dtype != TQ_DTYPE_F16 && out_dtype != TQ_DTYPE_BF16 && out_dtype != TQ_DTYPE_F32)
    return TQ_ERR_INVALID_ARG;
  if (!L.key_fp8 && (!cb || cb->bits != L.key_bits || cb->head_dim != cfg->head_dim)) return TQ_ERR_INVALID_ARG;
  if (batch == 0 || max_seq_len == 0) return TQ_OK;
  if (!cache || !block_table || !seq_lens || !key_out || !value_out) return TQ_ERR_INVALID_ARG;
  if (!aligned16(cache) || !aligned16(key_out) || !aligned16(value_out) ||
      (reinterpret_cast<unsigned long long>(block_table) & 3ull) ||
      (reinterpret_cast<unsigned long long>(seq_lens) & 3ull))
    return TQ_ERR_MISALIGNED;
  if (dev_status && (reinterpret_cast<unsigned long long>(dev_status) & 3ull)) return TQ_ERR_MISALIGNED;
  const long long seq_tiles = (static_cast<long long>(max_seq_len) + kTileTokens - 1) / kTileTokens;
  if (seq_tiles * batch > 0x7fffffffll || cfg->num_kv_heads > 65535) return TQ_ERR_INVALID_ARG;
  if (seq_tiles * batch * cfg->num_kv_heads >= (1ll << 32)) return TQ_ERR_UNSUPPORTED;   // 32-bit tile index

  DequantArgs a;
  a.cache = static_cast<const uint8_t*>(cache);
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.key_out = key_out;
  a.value_out = value_out;
  a.status = dev_status;
  a.num_blocks = num_blocks;
  a.n_kv = cfg->num_kv_heads;
  a.max_seq_len = max_seq_len;
  a.batch = batch;
  a.seq_tiles = static_cast<int>(seq_tiles);
  const long long cap = static_cast<long long>(bt_stride) * cfg->block_size;
  a.len_cap = static_cast<int>(cap < max_seq_len ? cap : max_seq_len);
  a.bt_stride = bt_stride;
  a.log2_bs = __builtin_ctz(static_cast<unsigned>(cfg->block_size));
  a.tiles_per_block = cfg->block_size / kTileTokens;
  a.tile_bytes = L.tile_bytes;
  a.k_off = L.k_off;
  a.k_row = L.k_row_bytes;
  a.v_off = L.v_off;
  a.v_row = L.v_row_bytes;
  a.knorm_off = L.knorm_off;
  a.vscale_off = L.vscale_off;
  a.vzero_off = L.vzero_off;
  for (int i = 0; i < 16; ++i) a.cent[i] = (!L.key_fp8 && i < cb->num_levels) ? cb->centroids[i] : 0.f;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t err;
  if (L.key_fp8) err = launch_dequant<kFp8, 4>(a, batch, out_dtype, s);
  else if (L.key_bits == 4) err = launch_dequant<kMse4, 4>(a, batch, out_dtype, s);
  else if (L.value_bits == 4) err = launch_dequant<kMse3, 4>(a, batch, out_dtype, s);
  else err = launch_dequant<kMse3, 3>(a, batch, out_dtype, s);
  return err == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}
