// Per-vector store arithmetic shared by the store kernel (tq_store.cu) and the
// decode's append path (tq_decode.cu): a half-warp holds the key and the value
// of one (token, KV head), 8 coordinates per lane (coordinate 8 l + j in lane
// l of the half), quantises both and writes their bytes into a cache tile.
//
// Method: "vLLM 源码完全拆解(十九):TurboQuant KV Cache 量化" (pinghaoyang.com.cn),
// section "写入内核:store 路径如何旋转、量化与打包":
//   n = ||k||, x = k / (n + 1e-8), y = (H / sqrt(d)) x            ("K 的归一化与旋转")
//   idx_i = #{j : y_i >= mid_j}                                    ("二分查找")
//   stored norm = n / sqrt(sum c[idx]^2 + 1e-16), fp16            ("norm correction 的折叠")
//   LSB-first bit packing of idx                                   ("位打包")
//   V: s = (max-min)/(2^b-1) floored at 1e-8, q = int((v-min)/s+0.5) clamped,
//      fp16 scale and zero                                         ("V 的 min/max 均匀量化")
//   FP8 keys: e4m3(k), no rotation, no norm                       ("FP8 K 路径")
//
// The value-quantisation arithmetic uses explicitly rounded fp32 operations
// (no contraction), so V codes are reproducible bit for bit; the key's scalars
// use the hardware approximations (a few ulp), see quantize_pair.
#ifndef TQ_STORE_CUH_
#define TQ_STORE_CUH_

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "tq_vec.cuh"

namespace tq {
namespace {

// Byte offsets and row strides of the regions of one cache tile.
struct TileGeom {
  int k_off, k_row, v_off, v_row, knorm_off, vscale_off, vzero_off;
};

// What one lane of the half writes for its pair.
struct PairBytes {
  uint32_t kw[2];                  // key run: 4-bit codes kw[0]; 3-bit codes the low 3 bytes of kw[0]; e4m3 kw[0..1]
  uint32_t vw;                     // value run, VBITS * 8 bits
  uint32_t vother;                 // 3-bit values: the run of lane l ^ 1
  uint16_t knorm, vscale, vzero;   // fp16 bits; lane 0 of the half writes them
};

// Codes of 8 values of one vector: trunc(fp32((v - min) / s) + 1/2), clamped
// to [0, kLevels], with IEEE division as specified. The product with an
// approximate reciprocal is within 4e-6 of the quotient (t <= 15), so
// away from a rounding boundary it gives the same code; a value within 1e-5
// of one takes the exact quotient, on a branch that is rarely taken (the
// division is a long instruction sequence, so it must not run for every
// coordinate).
template <int kLevels>
__device__ __forceinline__ void value_codes(const float v[8], float mn, float s, int q[8]) {
  const float rs = __fdividef(1.f, s);   // approximate: within a few ulp, far inside the band
  float dv[8];
  uint32_t near = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    dv[j] = __fsub_rn(v[j], mn);
    const float u = fmaf(dv[j], rs, 0.5f);
    near |= fabsf(u - rintf(u)) < 1e-5f ? (1u << j) : 0u;
    q[j] = __float2int_rz(u);
  }
  if (near) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if ((near >> j) & 1u) q[j] = __float2int_rz(__fadd_rn(__fdiv_rn(dv[j], s), 0.5f));
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) q[j] = min(q[j], kLevels);   // v >= min, so no code is negative
}

// Quantises the key held by a half-warp; every lane named in `mask` calls it
// (the reductions shuffle within the half). k is rotated in place. mid (15
// ascending midpoints) and cent (16 centroids) are the codebook's; unused for
// e4m3 keys.
template <int KMODE>
__device__ __forceinline__ void quantize_key(float k[8], int l, const float* mid, const float* cent, PairBytes& o,
                                             unsigned mask = 0xffffffffu) {
  if constexpr (KMODE == 8) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(k[4 * i], k[4 * i + 1]), __NV_SATFINITE, __NV_E4M3);
      const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(k[4 * i + 2], k[4 * i + 3]), __NV_SATFINITE, __NV_E4M3);
      o.kw[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
    }
    o.knorm = 0;
  } else {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) ss = fmaf(k[j], k[j], ss);
    // The key's scalars use the hardware approximations (a few ulp): the
    // pages' own pipeline forms y in fp32 through a matrix product, so y is
    // only defined to fp32 rounding, and the index decisions are checked
    // against the exact value with a 1e-5 band; the stored norm is an fp16.
    const float ss16 = half_sum(ss, mask);
    const float n = ss16 > 0.f ? ss16 * rsqrtf(ss16) : 0.f;
    fwht128_half(k, l, mask);
    const float sc = __fdividef(0.088388347648318440f, n + 1e-8f);   // 1/sqrt(128) / (n + 1e-8)
    int idx[8];
    float cs = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float y = k[j] * sc;
      // #{m : y >= mid_m} over the ascending midpoints, by binary search
      int c = 0;
#pragma unroll
      for (int step = 1 << (KMODE - 1); step >= 1; step >>= 1) c += (y >= mid[c + step - 1]) ? step : 0;
      idx[j] = c;
      const float cv = cent[c];
      cs = fmaf(cv, cv, cs);
    }
    cs = half_sum(cs, mask);
    uint32_t w = 0;   // LSB-first: coordinate 8 l + j at bit KMODE * j of the lane's run
#pragma unroll
    for (int j = 0; j < 8; ++j) w |= static_cast<uint32_t>(idx[j]) << (KMODE * j);
    o.kw[0] = w;
    o.kw[1] = 0u;
    o.knorm = __half_as_ushort(__float2half_rn(n * rsqrtf(cs + 1e-16f)));
  }
}

// Quantises the value held by a half-warp; every lane named in `mask` calls
// it (min and max shuffle within the half, the 3-bit runs across lanes l and
// l ^ 1).
template <int VBITS>
__device__ __forceinline__ void quantize_value(const float v[8], PairBytes& o, unsigned mask = 0xffffffffu) {
  constexpr int kLevels = (1 << VBITS) - 1;
  float mn = v[0], mx = v[0];
#pragma unroll
  for (int j = 1; j < 8; ++j) {
    mn = fminf(mn, v[j]);
    mx = fmaxf(mx, v[j]);
  }
  mn = half_min(mn, mask);
  mx = half_max(mx, mask);
  float s = __fdiv_rn(__fsub_rn(mx, mn), static_cast<float>(kLevels));
  s = (s > 1e-8f) ? s : 1e-8f;
  int q[8];
  value_codes<kLevels>(v, mn, s, q);
  uint32_t w = 0;   // this lane's LSB-first run: coordinate 8 l + j at bit VBITS * j
#pragma unroll
  for (int j = 0; j < 8; ++j) w |= static_cast<uint32_t>(q[j]) << (VBITS * j);
  o.vw = w;
  o.vother = VBITS == 3 ? __shfl_xor_sync(mask, w, 1) : 0u;
  o.vscale = __half_as_ushort(__float2half_rn(s));
  o.vzero = __half_as_ushort(__float2half_rn(mn));
}

// The writers put lane l's bytes of a quantised key or value into row r of a
// tile (a generic pointer: global or shared memory). No shuffles: callable by
// any subset of lanes.
template <int KMODE>
__device__ __forceinline__ void write_key(uint8_t* tile, int r, const TileGeom& g, int l, const PairBytes& o) {
  uint8_t* row = tile + g.k_off + r * g.k_row;
  if constexpr (KMODE == 8) {
    *reinterpret_cast<uint2*>(row + 8 * l) = make_uint2(o.kw[0], o.kw[1]);
  } else {
    if constexpr (KMODE == 4) {
      *reinterpret_cast<uint32_t*>(row + 4 * l) = o.kw[0];
    } else {   // 3 bytes at 3 l
      row[3 * l] = static_cast<uint8_t>(o.kw[0]);
      row[3 * l + 1] = static_cast<uint8_t>(o.kw[0] >> 8);
      row[3 * l + 2] = static_cast<uint8_t>(o.kw[0] >> 16);
    }
    if (l == 0) *reinterpret_cast<uint16_t*>(tile + g.knorm_off + 2 * r) = o.knorm;
  }
}

// Value words: the runs form 16-bit words; word i of token r = 2 p + t sits at
// v_off + 2 p v_row + 16 ((i >> 2) ^ x) + 4 (i & 3) + 2 t, x = 2 (p & 3) when
// v_row is a multiple of 64, else 0 (pair-interleaved, swizzled).
template <int VBITS>
__device__ __forceinline__ void write_value(uint8_t* tile, int r, const TileGeom& g, int l, const PairBytes& o) {
  const int pair = r >> 1;
  const int swz = (g.v_row % 64 == 0) ? 2 * (pair & 3) : 0;
  uint8_t* vbase = tile + g.v_off + pair * 2 * g.v_row + 2 * (r & 1);
  auto put_word = [&](int i, uint32_t bits16) {
    *reinterpret_cast<uint16_t*>(vbase + 16 * ((i >> 2) ^ swz) + 4 * (i & 3)) = static_cast<uint16_t>(bits16);
  };
  if constexpr (VBITS == 4) {   // lane l holds words 2 l and 2 l + 1
    put_word(2 * l, o.vw);
    put_word(2 * l + 1, o.vw >> 16);
  } else {   // 3-bit: lanes 2 m, 2 m + 1 hold the 48 bits of words 3 m .. 3 m + 2
    const int m = l >> 1;
    if ((l & 1) == 0) {
      put_word(3 * m, o.vw);                                         // bits 0-15
      put_word(3 * m + 1, (o.vw >> 16) | ((o.vother & 0xFFu) << 8));  // bits 16-23 | partner's 0-7
    } else {
      put_word(3 * m + 2, o.vw >> 8);                                // bits 8-23
    }
  }
  if (l == 0) {
    *reinterpret_cast<uint16_t*>(tile + g.vscale_off + 2 * r) = o.vscale;
    *reinterpret_cast<uint16_t*>(tile + g.vzero_off + 2 * r) = o.vzero;
  }
}

// Both halves of a pair: quantise k (rotated in place) and v, then write them.
template <int KMODE, int VBITS>
__device__ __forceinline__ void quantize_pair(float k[8], const float v[8], int l, const float* mid,
                                              const float* cent, PairBytes& o) {
  quantize_key<KMODE>(k, l, mid, cent, o);
  quantize_value<VBITS>(v, o);
}
template <int KMODE, int VBITS>
__device__ __forceinline__ void write_pair(uint8_t* tile, int r, const TileGeom& g, int l, const PairBytes& o) {
  write_key<KMODE>(tile, r, g, l, o);
  write_value<VBITS>(tile, r, g, l, o);
}

}  // namespace
}  // namespace tq

#endif  // TQ_STORE_CUH_
