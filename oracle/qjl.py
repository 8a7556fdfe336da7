"""TurboQuant_prod keys: a Lloyd-Max code plus a 1-bit QJL residual — oracle.

THIS MODULE IS TEST INFRASTRUCTURE (see the package docstring).

Restates the product-quantizer variant the pages describe next to the MSE one:

* [vLLM-TQ] section "Lloyd-Max 量化器", the TurboQuant_mse / TurboQuant_prod
  passage: TurboQuant_prod adds a 1-bit QJL layer on the residual of the MSE
  quantizer, which makes the inner-product estimate unbiased (vLLM ships only
  the MSE quantizer; section "TurboQuant 在 vLLM 中的位置", "为什么不用 QJL").
* [TQ-proj] the page on the open-source "turboquant" project
  (kwkr.cn/news/555717), subsection "最后 1 bit 的巧思:QJL 残差符号位让估计无偏": the
  key's b-bit budget is split into a (b - 1)-bit Lloyd-Max code of the rotated
  unit vector, giving an approximation x~; the residual r = x - x~ is
  multiplied by a random Gaussian matrix S and only the sign of each projected
  coordinate is kept (one bit per dimension, 8 per byte), together with ||r||;
  the inner product with a query y is estimated as
      <y, x~> + ||r|| * sqrt(pi / 2) / d * <S^T y, signs>,
  whose expectation over S is <y, x> (unbiased).

Readings of this library (the pages leave them open):

* Rotation: the normalised Sylvester-Hadamard rotation of the main method
  (``rotation.rotate``), as for the MSE presets; x is the rotated unit vector
  y = (H / sqrt(d)) k / (||k|| + 1e-8) and the query is rotated the same way.
* S has d rows (one sign per dimension, as the page says); S is an input (the
  random numbers the method draws are passed in), i.i.d. N(0, 1) entries.
* sign(0) = +1: a projection of exactly zero stores bit 1.
* The key norm is stored as fp16 without norm correction (the correction is
  the MSE quantizer's bias fix; the QJL term replaces it), and ||r|| as fp16.
* The (b - 1)-bit code is the store's: idx = #{j : y_j >= mid_j} over the fp32
  midpoints of ``codebook(d, b - 1)``, y compared in fp32.
* Sign bits are packed LSB-first: bit i of byte i // 8 is the sign of
  projection i.

Everything else is float64; the estimate for key k and query q is
    n * (<q_r, c[idx]> + ||r|| * sqrt(pi/2) / d * <S q_r, signs>)
with q_r = (H / sqrt(d)) q, which estimates <q, k> (H / sqrt(d) is orthonormal).
"""

from __future__ import annotations

import math

import numpy as np

from . import numerics, rotation
from .store import pack_bits, unpack_bits

__all__ = ["PROD_PRESETS", "prod_quantize", "prod_estimate", "pack_signs", "unpack_signs",
           "prod_tile_layout", "prod_store", "prod_read", "prod_scores"]

# preset name -> (total key bits per coordinate, Lloyd-Max bits)
PROD_PRESETS = {"prod3": (3, 2)}


def pack_signs(bits: np.ndarray) -> np.ndarray:
    """{0, 1} bits [..., d] -> uint8 [..., d / 8], LSB-first."""
    return np.packbits(np.asarray(bits, dtype=np.uint8), axis=-1, bitorder="little")


def unpack_signs(packed: np.ndarray, d: int) -> np.ndarray:
    """uint8 [..., d / 8] -> signs in {-1, +1} [..., d] (float64)."""
    b = np.unpackbits(np.asarray(packed, dtype=np.uint8), axis=-1, bitorder="little")[..., :d]
    return 2.0 * b.astype(np.float64) - 1.0


def prod_quantize(k: np.ndarray, S: np.ndarray, centroids: np.ndarray, midpoints: np.ndarray, mse_bits: int,
                  idx: np.ndarray | None = None):
    """Quantise rows of k [M, d] (float64 values of the inputs).

    Returns a dict: idx [M, d] (Lloyd-Max indices), norm [M] (float64 ||k||),
    rnorm [M] (float64 ||r||), proj [M, d] (float64 S r), sign_bits [M, d]
    ({0, 1}, 1 where S r >= 0), plus the packed forms and fp16 bit patterns.

    ``idx`` [M, d], when given, replaces the nearest-centroid decision: the
    residual, its norm and its signs are then those of that code. A
    coordinate whose rotated value lies on a midpoint to within rounding may
    be coded to either neighbour by an implementation computing in another
    precision; this lets a comparison follow its choice instead of counting
    the one flip again in every sign of the vector.
    """
    k = np.asarray(k, dtype=np.float64)
    S = np.asarray(S, dtype=np.float64)
    n = np.sqrt((k * k).sum(axis=-1))
    y = rotation.rotate(k / (n[:, None] + 1e-8))
    y32 = y.astype(np.float32)
    mids = np.asarray(midpoints, dtype=np.float32)
    if idx is None:
        idx = (y32[:, :, None] >= mids[None, None, :]).sum(axis=-1).astype(np.int64)
    else:
        idx = np.asarray(idx, dtype=np.int64).reshape(y.shape)
    c = np.asarray(centroids, dtype=np.float32).astype(np.float64)
    r = y - c[idx]
    rnorm = np.sqrt((r * r).sum(axis=-1))
    proj = r @ S.T
    sign_bits = (proj >= 0).astype(np.uint8)
    return {
        "idx": idx, "y": y, "norm": n, "rnorm": rnorm, "residual": r, "proj": proj, "sign_bits": sign_bits,
        "packed_idx": pack_bits(idx, mse_bits), "packed_signs": pack_signs(sign_bits),
        "norm_bits": numerics.fp16_bits(n), "rnorm_bits": numerics.fp16_bits(rnorm),
    }


def prod_estimate(q: np.ndarray, S: np.ndarray, centroids: np.ndarray, idx: np.ndarray, signs: np.ndarray,
                  norm: np.ndarray, rnorm: np.ndarray) -> np.ndarray:
    """Estimates of <q_a, k_m> for queries q [A, d] and quantised keys m
    (idx [M, d], signs in {-1, +1} [M, d], norm [M], rnorm [M]) -> [A, M]."""
    q = np.asarray(q, dtype=np.float64)
    d = q.shape[-1]
    S = np.asarray(S, dtype=np.float64)
    c = np.asarray(centroids, dtype=np.float32).astype(np.float64)
    qr = rotation.rotate(q)                       # [A, d]
    mse = qr @ c[idx].T                           # [A, M]
    qjl = (qr @ S.T) @ np.asarray(signs, dtype=np.float64).T
    return np.asarray(norm)[None, :] * (mse + np.asarray(rnorm)[None, :] * math.sqrt(math.pi / 2) / d * qjl)


# ---------------------------------------------------------------- paged key cache

class ProdTileLayout:
    """Key-only paged cache of the prod presets (this library's layout):

      cache[num_blocks][n_kv][block_size / 16][tile_bytes]

    A tile holds 16 positions of one KV head as regions: the LSB-first
    Lloyd-Max index streams (16 rows of d * mse_bits / 8 bytes), the sign
    streams (16 rows of d / 8 bytes), the fp16 key norms and the fp16 residual
    norms (16 each). Position p of sequence b is in block block_table[b][p //
    bs], row p % bs, as for the main cache.
    """

    def __init__(self, d: int, block_size: int, n_kv: int, mse_bits: int):
        self.d, self.block_size, self.n_kv, self.mse_bits = d, block_size, n_kv, mse_bits
        self.kb = d * mse_bits // 8
        self.sb = d // 8
        self.k_off = 0
        self.s_off = 16 * self.kb
        self.norm_off = self.s_off + 16 * self.sb
        self.rnorm_off = self.norm_off + 32
        self.tile_bytes = self.rnorm_off + 32
        self.slot_bytes = self.tile_bytes // 16

    @property
    def tiles_per_block(self) -> int:
        return self.block_size // 16

    @property
    def block_bytes(self) -> int:
        return self.n_kv * self.tiles_per_block * self.tile_bytes

    def tile_base(self, block, head: int, offset):
        return ((np.asarray(block) * self.n_kv + head) * self.tiles_per_block + np.asarray(offset) // 16) * self.tile_bytes


def prod_tile_layout(d: int, block_size: int, n_kv: int, mse_bits: int) -> ProdTileLayout:
    if block_size % 16 or d % 8:
        raise ValueError("block_size must be a multiple of 16 and d of 8")
    return ProdTileLayout(d, block_size, n_kv, mse_bits)


def prod_store(k: np.ndarray, slot_mapping: np.ndarray, S: np.ndarray, cache: np.ndarray, layout: ProdTileLayout,
               centroids, midpoints):
    """Quantise k [N, n_kv, d] and write each (token, head) into ``cache``
    (flat uint8) at its slot; slot < 0 or a block past the cache writes nothing."""
    k = np.asarray(k, dtype=np.float64)
    n_tok, n_kv, d = k.shape
    info = prod_quantize(k.reshape(-1, d), S, centroids, midpoints, layout.mse_bits)
    slots = np.asarray(slot_mapping, dtype=np.int64)
    num_blocks = cache.size // layout.block_bytes
    block, off = slots // layout.block_size, slots % layout.block_size
    for t in np.nonzero((slots >= 0) & (block < num_blocks))[0]:
        r = off[t] % 16
        for h in range(n_kv):
            m = t * n_kv + h
            base = int(layout.tile_base(block[t], h, off[t]))
            a = base + layout.k_off + r * layout.kb
            cache[a: a + layout.kb] = info["packed_idx"][m]
            a = base + layout.s_off + r * layout.sb
            cache[a: a + layout.sb] = info["packed_signs"][m]
            for field, bits in ((layout.norm_off, info["norm_bits"][m]), (layout.rnorm_off, info["rnorm_bits"][m])):
                cache[base + field + 2 * r] = int(bits) & 0xFF
                cache[base + field + 2 * r + 1] = int(bits) >> 8
    return info


def prod_read(cache: np.ndarray, layout: ProdTileLayout, blocks, offsets, head: int):
    """Fields of the slots at (blocks[i], offsets[i], head): idx [L, d],
    signs in {-1, +1} [L, d], fp16 norm and residual-norm values [L]."""
    blocks = np.asarray(blocks, dtype=np.int64)
    offsets = np.asarray(offsets, dtype=np.int64)
    base = layout.tile_base(blocks, head, offsets)
    r = offsets % 16
    ka = (base + layout.k_off + r * layout.kb)[:, None] + np.arange(layout.kb)[None, :]
    sa = (base + layout.s_off + r * layout.sb)[:, None] + np.arange(layout.sb)[None, :]

    def u16(a):
        return (cache[a].astype(np.uint16) | (cache[a + 1].astype(np.uint16) << 8))

    idx = unpack_bits(cache[ka], layout.mse_bits, layout.d)
    signs = unpack_signs(cache[sa], layout.d)
    norm = numerics.fp16_value(u16(base + layout.norm_off + 2 * r))
    rnorm = numerics.fp16_value(u16(base + layout.rnorm_off + 2 * r))
    return idx, signs, norm, rnorm


def prod_scores(q: np.ndarray, S: np.ndarray, cache: np.ndarray, layout: ProdTileLayout, centroids,
                block_table: np.ndarray, seq_lens: np.ndarray, max_seq_len: int, scale: float | None = None):
    """scale * estimate of <q[b, h], k_p> for every cached position p of
    sequence b, query head h reading KV head h // (n_q / n_kv); float64
    [B, n_q, max_seq_len], positions at or past the length are 0.
    scale defaults to 1 / sqrt(d)."""
    q = np.asarray(q, dtype=np.float64)
    bsz, n_q, d = q.shape
    group = n_q // layout.n_kv
    scale = 1.0 / math.sqrt(d) if scale is None or scale <= 0 else scale
    out = np.zeros((bsz, n_q, max_seq_len))
    for b in range(bsz):
        length = int(seq_lens[b])
        if length == 0:
            continue
        pos = np.arange(length)
        blocks = np.asarray(block_table[b])[pos // layout.block_size]
        offs = pos % layout.block_size
        for h in range(layout.n_kv):
            idx, signs, norm, rnorm = prod_read(cache, layout, blocks, offs, h)
            heads = list(range(h * group, (h + 1) * group))
            out[b, heads, :length] = scale * prod_estimate(q[b, heads], S, centroids, idx, signs, norm, rnorm)
    return out
