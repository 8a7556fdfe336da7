"""Oracle: a plain, slow, obviously-correct CPU reference for TurboQuant over a
paged KV cache.

THIS PACKAGE IS TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import it. The product path (the
CUDA library under ``turboquant_paged_kv_gb300/`` and its Python binding) never
imports, calls or links anything here, and this package never imports the
product. The two share no code; only the seeded input generators in
``workloads.py`` (which hold none of the method's arithmetic) feed both.

Everything is computed in float64 with NumPy, except where the pages fix a
narrower precision for a *decision* (the fp32 midpoints the keys are compared
against, the fp32 value-quantisation arithmetic, fp16 metadata, e4m3 keys);
there the oracle rounds exactly as the pages say, so that both sides take the
same decision in the same precision.

Sources (the pages this restates):

  [vLLM-TQ]  "vLLM 源码完全拆解(十九):TurboQuant KV Cache 量化——Hadamard 旋转、
             Lloyd-Max 标量量化与分页缓存内核" (pinghaoyang.com.cn). The main
             source: codebook solver, slot layout, store and decode kernels.
  [TQ-intro] "vLLM TurboQuant 介绍:极低比特 KV Cache 量化" (beaiera.top).
  [NVFP4-TQ] "NVIDIA KV Cache 量化中的 NVFP4 与 TurboQuant" (moonnryan.github.io).

Modules:
  codebook  Lloyd-Max centroids and decision midpoints for N(0, 1/d).
  rotation  Normalised Sylvester-Hadamard rotation.
  numerics  fp16 / e4m3 encodings and the fp32 value-quantisation steps.
  layout    preset table, slot sizes and the paged tile layout (byte addresses).
  store     quantise K/V vectors and write slots into a paged cache.
  decode    attention over the packed cache (exact softmax, no split), and the
            continuation-chunk form of it (one decode request per query).
  dequant   the cached keys and values expanded back to the original basis.
"""
