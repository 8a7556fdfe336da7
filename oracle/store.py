"""Quantise K/V vectors and write slots into the paged cache — oracle.

Restates [vLLM-TQ] section "写入内核:store 路径如何旋转、量化与打包":

* "K 的归一化与旋转为什么放在 kernel 外面": n = ||k||, x = k / (n + 1e-8),
  y = (H / sqrt(d)) x.
* "二分查找:3 到 4 次比较替代线性扫描": the index of a coordinate is the
  lower-bound position among the fp32 midpoints with ``y >= mid`` going right,
  i.e. idx = #{j : y >= m_j}; the oracle counts directly.
* "向量范数的存储与 norm correction 的折叠": with norm correction the stored
  norm is n / sqrt(sum_i c[idx_i]^2 + 1e-16), cast to fp16.
* "位打包:3-bit 的 8 个一组与 4-bit 的 2 个一组": indices form an LSB-first
  bitstream, bit (b*i + j) being bit j of idx_i (4-bit: even coordinate in the
  low nibble; 3-bit: 8 indices per little-endian 24-bit group).
* "V 的 min/max 均匀量化": see ``numerics.value_quant_fp32``; scale and the
  minimum (the zero point) are stored as fp16.
* "FP8 K 路径:不旋转,直接 cast": k8v4 stores e4m3(k) with no rotation and no norm.
* "融合 kernel 的骨架": slot s goes to block s // bs, offset s % bs; s < 0 writes
  nothing.

Byte placement follows ``layout.tile_layout``. The rotation, norm and
centroid arithmetic are float64; the comparison against the fp32 midpoints
uses y rounded to fp32, the precision the pages compute y in.
"""

from __future__ import annotations

import numpy as np

from . import numerics, rotation
from .layout import Preset, TileLayout, TILE_TOKENS, v_word_offset

__all__ = ["pack_bits", "unpack_bits", "quantize_keys", "quantize_values", "store"]


def pack_bits(idx: np.ndarray, bits: int) -> np.ndarray:
    """LSB-first bitstream of each row of ``idx`` -> uint8 [..., ceil(d*bits/8)]."""
    idx = np.asarray(idx, dtype=np.int64)
    d = idx.shape[-1]
    shifts = np.arange(bits)
    bitarr = ((idx[..., :, None] >> shifts) & 1).astype(np.uint8)   # [..., d, bits]
    bitarr = bitarr.reshape(idx.shape[:-1] + (d * bits,))
    return np.packbits(bitarr, axis=-1, bitorder="little")


def unpack_bits(packed: np.ndarray, bits: int, d: int) -> np.ndarray:
    """Inverse of ``pack_bits``: uint8 rows -> int64 indices [..., d]."""
    packed = np.asarray(packed, dtype=np.uint8)
    bitarr = np.unpackbits(packed, axis=-1, bitorder="little")[..., : d * bits]
    bitarr = bitarr.reshape(packed.shape[:-1] + (d, bits)).astype(np.int64)
    return (bitarr << np.arange(bits)).sum(axis=-1)


def quantize_keys(k: np.ndarray, centroids: np.ndarray, midpoints: np.ndarray,
                  bits: int, norm_correction: bool):
    """MSE key path for rows of ``k`` [M, d] (float64 values of the inputs).

    Returns dict with packed index bytes, fp16 norm bits and intermediates.
    """
    k = np.asarray(k, dtype=np.float64)
    n = np.sqrt((k * k).sum(axis=-1))
    x = k / (n[:, None] + 1e-8)
    y = rotation.rotate(x)
    y32 = y.astype(np.float32)
    mids = np.asarray(midpoints, dtype=np.float32)
    idx = (y32[:, :, None] >= mids[None, None, :]).sum(axis=-1).astype(np.int64)
    c = np.asarray(centroids, dtype=np.float32).astype(np.float64)
    if norm_correction:
        cn = np.sqrt((c[idx] ** 2).sum(axis=-1) + 1e-16)
        stored = n / cn
    else:
        stored = n
    return {
        "packed": pack_bits(idx, bits),
        "norm_bits": numerics.fp16_bits(stored),
        "idx": idx,
        "y": y,
        "norm": n,
        "stored_norm": stored,
    }


def quantize_values(v: np.ndarray, bits: int):
    """Value path for rows of ``v`` [M, d]."""
    q, s, mn = numerics.value_quant_fp32(v, bits)
    return {
        "packed": pack_bits(q, bits),
        "codes": q,
        "scale32": s,
        "min32": mn,
        "scale_bits": numerics.fp16_bits(s),
        "zero_bits": numerics.fp16_bits(mn),
    }


def store(k: np.ndarray, v: np.ndarray, slot_mapping: np.ndarray, cache: np.ndarray,
          layout: TileLayout, preset: Preset, centroids=None, midpoints=None):
    """Write each (token, kv head) of k, v [N, n_kv, d] into ``cache`` (flat uint8).

    Returns (info dict of per-vector intermediates, list of skipped
    out-of-range (token, slot) pairs).
    """
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n_tok, n_kv, d = k.shape
    rows_k = k.reshape(n_tok * n_kv, d)
    rows_v = v.reshape(n_tok * n_kv, d)
    if preset.key_fp8:
        kinfo = {"packed": numerics.e4m3_encode(rows_k)}
    else:
        kinfo = quantize_keys(rows_k, centroids, midpoints, preset.key_bits,
                              preset.norm_correction)
    vinfo = quantize_values(rows_v, preset.value_bits)
    num_blocks = cache.size // layout.block_bytes
    slots = np.asarray(slot_mapping, dtype=np.int64)
    block = slots // layout.block_size
    off = slots % layout.block_size
    in_range = (slots >= 0) & (block < num_blocks)
    skipped = [(int(t), int(slots[t])) for t in np.nonzero((slots >= 0) & ~in_range)[0]]
    toks = np.nonzero(in_range)[0]
    if toks.size == 0:
        return {"k": kinfo, "v": vinfo}, skipped
    heads = np.arange(n_kv)
    # tile base of every written (token, head): [T, n_kv]
    base = ((block[toks, None] * n_kv + heads[None, :]) * layout.tiles_per_block
            + off[toks, None] // TILE_TOKENS) * layout.tile_bytes
    r = (off[toks] % TILE_TOKENS)[:, None]                     # row inside the tile
    pair, j = r // 2, r % 2
    rows = (toks[:, None] * n_kv + heads[None, :]).reshape(-1)  # vector index m
    base = base.reshape(-1, 1)
    r = np.broadcast_to(r, (toks.size, n_kv)).reshape(-1, 1)
    pair = np.broadcast_to(pair, (toks.size, n_kv)).reshape(-1, 1)
    j = np.broadcast_to(j, (toks.size, n_kv)).reshape(-1, 1)

    # K region: row r holds the token's key bytes
    kcol = np.arange(layout.kb)[None, :]
    cache[base + layout.k_off + r * layout.kb + kcol] = kinfo["packed"][rows]
    # V region: pair-interleaved 16-bit words
    words = layout.vb // 2
    wi = np.arange(words)[None, :]
    vaddr = base + layout.v_off + v_word_offset(layout.vb, pair, wi, j)
    vbytes = vinfo["packed"][rows]
    cache[vaddr] = vbytes[:, 0::2]
    cache[vaddr + 1] = vbytes[:, 1::2]

    def put_u16(field_off, bits):
        addr = base[:, 0] + field_off + 2 * r[:, 0]
        bits = np.asarray(bits, dtype=np.uint16)[rows]
        cache[addr] = (bits & 0xFF).astype(np.uint8)
        cache[addr + 1] = (bits >> 8).astype(np.uint8)

    if layout.has_knorm:
        put_u16(layout.knorm_off, kinfo["norm_bits"])
    put_u16(layout.vscale_off, vinfo["scale_bits"])
    put_u16(layout.vzero_off, vinfo["zero_bits"])
    return {"k": kinfo, "v": vinfo}, skipped
