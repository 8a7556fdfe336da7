// Host side of libtq: Lloyd-Max codebook solver, preset table, cache layout
// arithmetic and status strings.
//
// Method source: "vLLM 源码完全拆解(十九):TurboQuant KV Cache 量化" (pinghaoyang.com.cn),
// sections "Lloyd-Max 量化器" (codebook) and "存储布局" (slot sizes).

#include <cmath>
#include <cstring>

#include "tq_internal.h"

namespace tq {

bool preset_info(int preset, PresetInfo* out) {
  switch (preset) {
    case TQ_PRESET_K8V4:    *out = {8, 4, true, false}; return true;
    case TQ_PRESET_4BIT_NC: *out = {4, 4, false, true}; return true;
    case TQ_PRESET_K3V4_NC: *out = {3, 4, false, true}; return true;
    case TQ_PRESET_3BIT_NC: *out = {3, 3, false, true}; return true;
    case TQ_PRESET_PROD3:   *out = {2, 0, false, false}; return true;   // keys only: its own layout
    default: return false;
  }
}

tq_status make_layout(const tq_config* cfg, tq_layout* out) {
  if (!cfg || !out) return TQ_ERR_INVALID_ARG;
  PresetInfo pi;
  if (!preset_info(cfg->preset, &pi)) return TQ_ERR_INVALID_ARG;
  const int d = cfg->head_dim;
  if (d <= 0 || cfg->block_size <= 0 || cfg->num_kv_heads <= 0) return TQ_ERR_INVALID_ARG;
  if (cfg->flags & ~TQ_FLAG_INDICES_READY) return TQ_ERR_INVALID_ARG;
  if (d != 128) return TQ_ERR_UNSUPPORTED;
  const int bs = cfg->block_size;
  if (bs != 16 && bs != 32 && bs != 64 && bs != 128) return TQ_ERR_UNSUPPORTED;
  if (pi.value_bits == 0) return TQ_ERR_UNSUPPORTED;   // the prod preset has a key-only cache (tq_prod_layout_for)

  tq_layout L;
  std::memset(&L, 0, sizeof(L));
  L.key_bits = pi.key_bits;
  L.value_bits = pi.value_bits;
  L.key_fp8 = pi.key_fp8;
  L.norm_correction = pi.norm_correction;
  const int kb = pi.key_fp8 ? d : (d * pi.key_bits + 7) / 8;
  const int vb = (d * pi.value_bits + 7) / 8;
  // slot arithmetic of "从 slot_size 的三项算术开始"
  L.key_packed_bytes = pi.key_fp8 ? d : kb + 2;
  L.value_packed_bytes = vb + 4;
  L.slot_bytes = L.key_packed_bytes + L.value_packed_bytes;
  L.tile_tokens = kTileTokens;
  L.k_off = 0;
  L.k_row_bytes = kb;
  L.v_off = kTileTokens * kb;
  L.v_row_bytes = vb;
  int meta = L.v_off + kTileTokens * vb;
  L.knorm_off = pi.key_fp8 ? -1 : meta;
  L.vscale_off = meta + (pi.key_fp8 ? 0 : 2 * kTileTokens);
  L.vzero_off = L.vscale_off + 2 * kTileTokens;
  L.tile_bytes = L.vzero_off + 2 * kTileTokens;
  if (L.tile_bytes != kTileTokens * L.slot_bytes) return TQ_ERR_INVALID_ARG;
  L.block_bytes = static_cast<long long>(bs) * cfg->num_kv_heads * L.slot_bytes;
  *out = L;
  return TQ_OK;
}

namespace {

// P[x >= t] and sigma^2 * pdf(t) for x ~ N(0, sigma^2).
double upper_tail(double t, double sigma) {
  if (std::isinf(t)) return t > 0 ? 0.0 : 1.0;
  return 0.5 * std::erfc(t / (sigma * std::sqrt(2.0)));
}
double scaled_density(double t, double sigma) {
  if (std::isinf(t)) return 0.0;
  const double z = t / sigma;
  return sigma / std::sqrt(2.0 * M_PI) * std::exp(-0.5 * z * z);
}

}  // namespace
}  // namespace tq

extern "C" {

tq_status tq_build_codebook(int head_dim, int bits, tq_codebook* out) {
  if (!out || head_dim <= 0 || bits < 1 || bits > 4) return TQ_ERR_INVALID_ARG;
  const int n = 1 << bits;
  const double sigma = 1.0 / std::sqrt(static_cast<double>(head_dim));
  double c[16], next[16], edge[17];
  // uniform start on [-3.5 sigma, 3.5 sigma] (subsection "Lloyd-Max 的两个最优性条件")
  for (int i = 0; i < n; ++i) c[i] = -3.5 * sigma + 7.0 * sigma * (i + 0.5) / n;
  bool converged = false;
  for (int it = 0; it < 100000 && !converged; ++it) {
    edge[0] = -INFINITY;
    edge[n] = INFINITY;
    for (int i = 1; i < n; ++i) edge[i] = 0.5 * (c[i - 1] + c[i]);   // condition 1
    double change = 0.0;
    for (int i = 0; i < n; ++i) {                                     // condition 2
      const double mass = tq::upper_tail(edge[i], sigma) - tq::upper_tail(edge[i + 1], sigma);
      const double first = tq::scaled_density(edge[i], sigma) - tq::scaled_density(edge[i + 1], sigma);
      next[i] = first / mass;
      change = std::fmax(change, std::fabs(next[i] - c[i]));
    }
    for (int i = 0; i < n; ++i) c[i] = next[i];
    converged = change < 1e-13;
  }
  if (!converged) return TQ_ERR_INVALID_ARG;
  tq_codebook cb;
  std::memset(&cb, 0, sizeof(cb));
  cb.head_dim = head_dim;
  cb.bits = bits;
  cb.num_levels = n;
  for (int i = 0; i < n; ++i) {
    const double sym = 0.5 * (c[i] - c[n - 1 - i]);   // exact antisymmetry
    cb.centroids[i] = static_cast<float>(sym);
  }
  for (int i = 0; i + 1 < n; ++i) {
    // fp32 (c_i + c_{i+1}) / 2 as the kernels' midpoints ("vLLM 内置的 Lloyd-Max 码本")
    volatile float s = cb.centroids[i] + cb.centroids[i + 1];
    cb.midpoints[i] = s * 0.5f;
  }
  *out = cb;
  return TQ_OK;
}

tq_status tq_layout_for(const tq_config* cfg, tq_layout* out) { return tq::make_layout(cfg, out); }

const char* tq_status_string(int status) {
  switch (status) {
    case TQ_OK: return "ok";
    case TQ_ERR_INVALID_ARG: return "invalid argument";
    case TQ_ERR_UNSUPPORTED: return "unsupported shape or preset";
    case TQ_ERR_MISALIGNED: return "misaligned pointer";
    case TQ_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case TQ_ERR_CUDA: return "CUDA launch failed";
    default: return "unknown status";
  }
}

int tq_version(void) { return TQ_ABI_VERSION; }

}  // extern "C"
