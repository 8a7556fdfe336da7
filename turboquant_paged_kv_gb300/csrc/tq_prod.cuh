// TurboQuant_prod key cache: the tile layout and host checks shared by the
// store (tq_prod_store.cu) and the scores path (tq_prod.cu).
//
// A tile holds 16 positions of one KV head: the 2-bit Lloyd-Max codes (32
// bytes a position), the 128 QJL sign bits of the residual's projection (16
// bytes), ||k|| and ||r|| as fp16, 52 bytes a position in all.
#ifndef TQ_PROD_CUH_
#define TQ_PROD_CUH_

#include <cuda_runtime.h>
#include <stdint.h>

#include "tq_internal.h"

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
constexpr int kThreads = 256;
constexpr float kQjlScale = 1.2533141373155003f / kD;   // sqrt(pi / 2) / d

__device__ __forceinline__ void flag(unsigned int* status, unsigned int bit) {
  if (status) atomicOr(status, bit);
}

inline tq_status prod_layout(const tq_config* cfg, tq_prod_layout* out) {
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

inline int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

}  // namespace
}  // namespace tq

#endif  // TQ_PROD_CUH_
