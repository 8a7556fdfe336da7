"""Full dequantisation of the cached keys and values back to the original
basis — oracle (test infrastructure).

Restates [vLLM-TQ] section "续写 prefill:小 chunk 走 decode,大 chunk 走反量化",
subsection "反量化 kernel:_tq_full_dequant_kv": for each cached position and KV
head the packed slot is expanded exactly as the decode unpacks it (no softmax),
and the keys are then turned back from the rotated basis by the inverse
rotation. The rotation H / sqrt(d) is symmetric and orthonormal (section "为什么
先旋转"), so its inverse is itself:

  index-coded keys  k_hat = stored_norm * (H / sqrt(d)) c[idx]
  FP8 keys          k_hat = e4m3(k)             (never rotated, "FP8 K 路径")
  values            v_hat = fp16(scale) * code + fp16(zero)

Readings where the pages leave a step open:
  * The pages round the expanded keys to fp16 and rotate them back with an
    fp16 copy of the Hadamard matrix; here the result is the exact value, and
    the output precision is the caller's choice (the rounding is the only
    difference).
  * The output holds max_seq_len positions per sequence (the pages' alloc_len)
    in [batch][position][KV head][d] order, the token-major layout the current
    chunk's raw keys and values have; positions at or beyond a sequence's
    length are zero.

Everything is float64.
"""

from __future__ import annotations

import numpy as np

from . import numerics, rotation
from .decode import dequantized_values, read_positions
from .layout import Preset, TileLayout
from .store import unpack_bits

__all__ = ["dequantize"]

_E4M3 = numerics.e4m3_decode_table()


def dequantize(cache: np.ndarray, layout: TileLayout, preset: Preset, centroids,
               block_table: np.ndarray, seq_lens: np.ndarray, max_seq_len: int,
               sequences=None):
    """(k_hat, v_hat), each float64 [batch, max_seq_len, n_kv, d].

    ``sequences`` optionally restricts the computed sequences (others stay 0).
    """
    block_table = np.asarray(block_table)
    seq_lens = np.asarray(seq_lens)
    bsz = len(seq_lens)
    d = layout.d
    n_kv = layout.n_kv
    k_hat = np.zeros((bsz, max_seq_len, n_kv, d), dtype=np.float64)
    v_hat = np.zeros_like(k_hat)
    c = None if preset.key_fp8 else np.asarray(centroids, np.float32).astype(np.float64)
    want = range(bsz) if sequences is None else sequences
    for b in want:
        length = min(int(seq_lens[b]), max_seq_len)
        if length <= 0:
            continue
        pos = np.arange(length)
        blocks = block_table[b][pos // layout.block_size]
        offs = pos % layout.block_size
        for h in range(n_kv):
            kbytes, vbytes, knorm, vscale, vzero = read_positions(cache, layout, blocks, offs, h)
            if preset.key_fp8:
                k_hat[b, :length, h] = _E4M3[kbytes]
            else:
                idx = unpack_bits(kbytes, preset.key_bits, d)
                k_rot = numerics.fp16_value(knorm)[:, None] * c[idx]   # rotated basis
                k_hat[b, :length, h] = rotation.rotate(k_rot)           # H / sqrt(d) is its own inverse
            v_hat[b, :length, h] = dequantized_values(vbytes, vscale, vzero, preset.value_bits, d)
    return k_hat, v_hat
