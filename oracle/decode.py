"""Attention read straight from the packed paged cache — oracle.

Restates [vLLM-TQ] section "读取内核:decode 如何从 packed slot 还原 K/V 并保持
Softmax 数值稳定":

* "程序入口:split 区间怎么算": query head h reads KV head h // (n_q / n_kv).
* "页内寻址" (section "存储布局"): position p of sequence b lives in block
  block_table[b][p // bs] at offset p % bs.
* "分数计算:FP8 K 与 MSE K 的两条路径": with index-coded keys the score is
  stored_norm * (q_rot . c[idx]) * scale with q_rot = (H / sqrt(d)) q, because
  the keys live in the rotated basis; with FP8 keys it is (q . e4m3(k)) * scale
  and q is not rotated. scale defaults to 1 / sqrt(d).
* "V 的解包:3-bit 的跨字节与 4-bit 的 nibble": value codes are unpacked from the
  LSB-first stream; the reconstruction is fp16(scale) * code + fp16(zero) (the
  zero point is the stored minimum, [vLLM-TQ] "V 的 min/max 均匀量化").
* "在线 softmax": the split-K online softmax with an LSE merge is an exact
  regrouping of softmax(scores) @ V; the oracle evaluates the plain,
  max-subtracted softmax over all positions at once, in float64.

A sequence of length 0 yields zeros (the pages are silent; this library's
reading).
"""

from __future__ import annotations

import math

import numpy as np

from . import numerics, rotation
from .layout import Preset, TileLayout, TILE_TOKENS, v_word_offset
from .store import unpack_bits

__all__ = ["read_positions", "dequantized_values", "decode", "continuation_decode"]

_E4M3 = numerics.e4m3_decode_table()


def _u16(cache: np.ndarray, addr: np.ndarray) -> np.ndarray:
    return cache[addr].astype(np.uint16) | (cache[addr + 1].astype(np.uint16) << 8)


def read_positions(cache: np.ndarray, layout: TileLayout, blocks: np.ndarray,
                   offsets: np.ndarray, head: int):
    """Raw fields of the slots at (blocks[i], offsets[i], head).

    Returns (key bytes [L, KB], value bytes [L, VB], knorm bits or None,
    vscale bits, vzero bits).
    """
    blocks = np.asarray(blocks, dtype=np.int64)
    offsets = np.asarray(offsets, dtype=np.int64)
    base = ((blocks * layout.n_kv + head) * layout.tiles_per_block
            + offsets // TILE_TOKENS) * layout.tile_bytes
    r = offsets % TILE_TOKENS
    pair, j = r // 2, r % 2
    kaddr = (base + layout.k_off + r * layout.kb)[:, None] + np.arange(layout.kb)[None, :]
    kbytes = cache[kaddr]
    wi = np.arange(layout.vb // 2)[None, :]
    vaddr = (base + layout.v_off)[:, None] + v_word_offset(layout.vb, pair[:, None], wi, j[:, None])
    vbytes = np.empty((len(blocks), layout.vb), dtype=np.uint8)
    vbytes[:, 0::2] = cache[vaddr]
    vbytes[:, 1::2] = cache[vaddr + 1]
    knorm = _u16(cache, base + layout.knorm_off + 2 * r) if layout.has_knorm else None
    vscale = _u16(cache, base + layout.vscale_off + 2 * r)
    vzero = _u16(cache, base + layout.vzero_off + 2 * r)
    return kbytes, vbytes, knorm, vscale, vzero


def dequantized_values(vbytes, vscale, vzero, bits: int, d: int) -> np.ndarray:
    codes = unpack_bits(vbytes, bits, d).astype(np.float64)
    s = numerics.fp16_value(vscale)[:, None]
    z = numerics.fp16_value(vzero)[:, None]
    return s * codes + z


def decode(q: np.ndarray, cache: np.ndarray, layout: TileLayout, preset: Preset,
           centroids, block_table: np.ndarray, seq_lens: np.ndarray,
           scale: float | None = None, heads=None) -> np.ndarray:
    """out[b, h, :] for q [B, n_q, d] (float64 values); float64 result.

    ``heads`` optionally restricts the computed query heads (others stay 0).
    """
    q = np.asarray(q, dtype=np.float64)
    bsz, n_q, d = q.shape
    n_kv = layout.n_kv
    group = n_q // n_kv
    if scale is None or scale <= 0:
        scale = 1.0 / math.sqrt(d)
    c = None if preset.key_fp8 else np.asarray(centroids, np.float32).astype(np.float64)
    out = np.zeros((bsz, n_q, d), dtype=np.float64)
    want = range(n_q) if heads is None else heads
    for b in range(bsz):
        length = int(seq_lens[b])
        if length == 0:
            continue
        pos = np.arange(length)
        blocks = np.asarray(block_table[b])[pos // layout.block_size]
        offs = pos % layout.block_size
        for kvh in range(n_kv):
            hs = [h for h in want if h // group == kvh]
            if not hs:
                continue
            kbytes, vbytes, knorm, vscale, vzero = read_positions(cache, layout, blocks, offs, kvh)
            vhat = dequantized_values(vbytes, vscale, vzero, preset.value_bits, d)
            if preset.key_fp8:
                kval = _E4M3[kbytes]
            else:
                idx = unpack_bits(kbytes, preset.key_bits, d)
                keys_rot = c[idx]                           # [L, d] rotated-basis keys
                nrm = numerics.fp16_value(knorm)
            for h in hs:
                if preset.key_fp8:
                    scores = scale * (kval @ q[b, h])
                else:
                    qr = rotation.rotate(q[b, h])
                    scores = scale * nrm * (keys_rot @ qr)
                p = np.exp(scores - scores.max())
                out[b, h] = (p @ vhat) / p.sum()
    return out


def continuation_decode(q_chunk: np.ndarray, cache: np.ndarray, layout: TileLayout, preset: Preset,
                        centroids, block_row: np.ndarray, cached_len: int,
                        scale: float | None = None) -> np.ndarray:
    """Attention of the q_len queries of a continuation chunk, float64 [q_len, n_q, d].

    Restates [vLLM-TQ] section "续写 prefill:小 chunk 走 decode,大 chunk 走反量化":
    the chunk's keys and values are already in the cache, and query i of the
    chunk (0-based) is served as a decode request of length cached_len + i + 1
    over the sequence's one block-table row, which is what makes the attention
    causal without a mask.
    """
    q_chunk = np.asarray(q_chunk, dtype=np.float64)
    q_len = q_chunk.shape[0]
    table = np.broadcast_to(np.asarray(block_row)[None, :], (q_len, len(block_row)))
    lens = cached_len + 1 + np.arange(q_len)
    return decode(q_chunk, cache, layout, preset, centroids, table, lens, scale)
