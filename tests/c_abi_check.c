/* A plain C99 caller of libtq's host-side entry points: the header must
 * compile as C, and the library must link and answer without Python.
 * Prints one line per check; exits non-zero on the first failure. No GPU
 * call is made (codebook, layout, workspace size, argument errors). */
#include <math.h>
#include <stdio.h>
#include <string.h>

#include "tq.h"

static int fail(const char* what) {
  printf("FAIL %s\n", what);
  return 1;
}

int main(void) {
  tq_codebook cb;
  tq_layout lay;
  tq_config cfg;
  int i;

  if (tq_version() != TQ_ABI_VERSION) return fail("version");
  printf("version %d\n", tq_version());

  if (tq_build_codebook(128, 4, &cb) != TQ_OK) return fail("codebook status");
  if (cb.num_levels != 16 || cb.bits != 4 || cb.head_dim != 128) return fail("codebook header");
  for (i = 0; i < 16; ++i)
    if (cb.centroids[i] != -cb.centroids[15 - i]) return fail("codebook antisymmetry");
  for (i = 0; i + 1 < 16; ++i)
    if (!(cb.centroids[i] < cb.midpoints[i] && cb.midpoints[i] < cb.centroids[i + 1])) return fail("midpoints");
  printf("codebook c15 %.6f\n", cb.centroids[15]);

  memset(&cfg, 0, sizeof(cfg));
  cfg.preset = TQ_PRESET_4BIT_NC;
  cfg.head_dim = 128;
  cfg.block_size = 16;
  cfg.num_q_heads = 32;
  cfg.num_kv_heads = 8;
  if (tq_layout_for(&cfg, &lay) != TQ_OK) return fail("layout status");
  if (lay.slot_bytes != 134 || lay.tile_bytes != 16 * 134 || lay.block_bytes != 16LL * 8 * 134) return fail("layout");
  printf("slot %d tile %d block %lld\n", lay.slot_bytes, lay.tile_bytes, lay.block_bytes);

  if (tq_decode_workspace_size(&cfg, 32, 4096) == 0) return fail("workspace size");
  printf("workspace %zu\n", tq_decode_workspace_size(&cfg, 32, 4096));

  /* host-side argument errors come back before any launch */
  if (tq_store(&cfg, &cb, NULL, NULL, TQ_DTYPE_BF16, 4, NULL, NULL, 1, NULL, NULL) != TQ_ERR_INVALID_ARG)
    return fail("store null pointers");
  if (tq_dequant(&cfg, &cb, NULL, 1, NULL, 1, NULL, 0, 16, NULL, NULL, TQ_DTYPE_BF16, NULL, NULL) != TQ_OK)
    return fail("dequant empty batch");
  cfg.preset = TQ_PRESET_3BIT_NC;
  if (tq_layout_for(&cfg, &lay) != TQ_OK || lay.slot_bytes != 102 || lay.v_row_bytes != 48) return fail("3bit_nc layout");
  cfg.head_dim = 96;
  if (tq_layout_for(&cfg, &lay) != TQ_ERR_UNSUPPORTED) return fail("d 96 unsupported");
  if (strlen(tq_status_string(TQ_ERR_UNSUPPORTED)) == 0) return fail("status string");
  printf("errors ok: %s\n", tq_status_string(TQ_ERR_UNSUPPORTED));
  printf("ALL OK\n");
  return 0;
}
