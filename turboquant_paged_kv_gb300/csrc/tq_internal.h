// Internal declarations shared by the libtq translation units (not ABI).
#ifndef TQ_INTERNAL_H_
#define TQ_INTERNAL_H_

#include "tq.h"

namespace tq {

constexpr int kTileTokens = 16;

// Decoded preset parameters ([vLLM-TQ] "四个预设对应什么").
struct PresetInfo {
  int key_bits;        // 3, 4, or 8 (e4m3)
  int value_bits;      // 3 or 4
  bool key_fp8;
  bool norm_correction;
};

bool preset_info(int preset, PresetInfo* out);

// Fills the layout; returns TQ_OK or an error for bad/unsupported shapes.
tq_status make_layout(const tq_config* cfg, tq_layout* out);

// Shared argument checks.
inline bool aligned16(const void* p) { return (reinterpret_cast<unsigned long long>(p) & 15ull) == 0; }
inline int effective_partition(const tq_config* cfg) {
  return cfg->partition_tokens > 0 ? cfg->partition_tokens : 512;
}

}  // namespace tq

#endif  // TQ_INTERNAL_H_
