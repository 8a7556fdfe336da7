"""Presets, slot sizes and the paged tile layout — oracle (test infrastructure).

Presets and slot arithmetic restate [vLLM-TQ] section "TurboQuant 在 vLLM 中的
位置" / subsection "四个预设对应什么" (the TQ_PRESETS table) and section
"存储布局" / subsection "从 slot_size 的三项算术开始":

  key bytes   = d                      (FP8 keys)
              = ceil(d * bk / 8) + 2   (index bits + fp16 norm)
  value bytes = ceil(d * bv / 8) + 4   (index bits + fp16 scale + fp16 zero)
  slot        = key + value, rounded up to even.

Byte placement is this library's paged tile layout (the pages leave the
physical order to the backend and themselves describe two, an AoS slot and an
SoA page; the layout below is the SoA family, fixed here as the ABI):

  cache[num_blocks][n_kv][block_size / 16][tile_bytes]   (bytes)

A tile holds 16 consecutive token positions of one KV head. Inside a tile:

  K region   16 rows x KB bytes   (KB = ceil(d*bk/8), or d for FP8); row r is
             token r's LSB-first index stream (or its e4m3 bytes).
  V region   16 x VB bytes        (VB = ceil(d*bv/8)); tokens are taken in
             pairs (2p, 2p+1) and the two LSB-first index streams of a pair
             are interleaved in 16-bit words, four words of each token per
             16-byte group: word i of token 2p+j sits at byte
             p*2*VB + 16*((i >> 2) ^ x) + 4*(i & 3) + 2*j of the region, with
             the group swizzle x = 2*(p & 3) when VB is a multiple of 64 (so a
             quarter warp reading group g of pairs c = 0..3 touches 8 distinct
             16-byte bank groups) and x = 0 otherwise.
  K norms    16 x fp16            (only for index-coded keys)
  V scales   16 x fp16
  V zeros    16 x fp16

so tile_bytes = 16 * slot_bytes and block_bytes = block_size * n_kv *
slot_bytes, which is the page size the pages give (e.g. 16 x 8 x 118 = 15104).
Token position p of a sequence lives in block block_table[b][p // bs] at
offset p % bs ([vLLM-TQ] "页内寻址:一页多少字节,slot 落在哪里"); a store slot
s maps to block s // bs, offset s % bs ([vLLM-TQ] "融合 kernel 的骨架").
"""

from __future__ import annotations

import math
from dataclasses import dataclass

__all__ = ["PRESETS", "Preset", "TileLayout", "preset_slot_sizes", "tile_layout", "TILE_TOKENS",
           "v_word_offset"]

TILE_TOKENS = 16


@dataclass(frozen=True)
class Preset:
    name: str
    key_bits: int        # 8 means FP8 (e4m3) keys
    value_bits: int
    norm_correction: bool

    @property
    def key_fp8(self) -> bool:
        return self.key_bits == 8


PRESETS = {
    "k8v4": Preset("k8v4", 8, 4, False),
    "4bit_nc": Preset("4bit_nc", 4, 4, True),
    "k3v4_nc": Preset("k3v4_nc", 3, 4, True),
    "3bit_nc": Preset("3bit_nc", 3, 3, True),
}


def preset_slot_sizes(preset: Preset, d: int):
    """(key_packed, value_packed, slot, slot_aligned) bytes for head_dim d."""
    if preset.key_fp8:
        key = d
    else:
        key = math.ceil(d * preset.key_bits / 8) + 2
    value = math.ceil(d * preset.value_bits / 8) + 4
    slot = key + value
    return key, value, slot, slot + (slot % 2)


@dataclass(frozen=True)
class TileLayout:
    d: int
    block_size: int
    n_kv: int
    kb: int              # K bytes per token (indices or e4m3)
    vb: int              # V index bytes per token
    has_knorm: bool
    slot_bytes: int
    tile_bytes: int
    k_off: int
    v_off: int
    knorm_off: int       # -1 when absent
    vscale_off: int
    vzero_off: int

    @property
    def tiles_per_block(self) -> int:
        return self.block_size // TILE_TOKENS

    @property
    def block_bytes(self) -> int:
        return self.n_kv * self.tiles_per_block * self.tile_bytes

    def tile_base(self, block: int, head: int, offset: int) -> int:
        """Byte offset of the tile holding (block, head, in-block offset)."""
        return ((block * self.n_kv + head) * self.tiles_per_block
                + offset // TILE_TOKENS) * self.tile_bytes


def v_word_offset(vb: int, pair, word, j):
    """Byte offset inside the V region of 16-bit word ``word`` of token 2*pair+j."""
    swz = (2 * (pair & 3)) if vb % 64 == 0 else 0
    return pair * 2 * vb + 16 * ((word >> 2) ^ swz) + 4 * (word & 3) + 2 * j


def tile_layout(preset: Preset, d: int, block_size: int, n_kv: int) -> TileLayout:
    if block_size % TILE_TOKENS:
        raise ValueError("block_size must be a multiple of 16")
    kb = d if preset.key_fp8 else math.ceil(d * preset.key_bits / 8)
    vb = math.ceil(d * preset.value_bits / 8)
    if vb % 2:
        raise ValueError("value bytes per token must be even")
    has_knorm = not preset.key_fp8
    slot = kb + vb + (2 if has_knorm else 0) + 4
    t = TILE_TOKENS
    k_off = 0
    v_off = t * kb
    meta = v_off + t * vb
    knorm_off = meta if has_knorm else -1
    vscale_off = meta + (2 * t if has_knorm else 0)
    vzero_off = vscale_off + 2 * t
    tile_bytes = vzero_off + 2 * t
    assert tile_bytes == t * slot
    return TileLayout(d, block_size, n_kv, kb, vb, has_knorm, slot, tile_bytes,
                      k_off, v_off, knorm_off, vscale_off, vzero_off)
