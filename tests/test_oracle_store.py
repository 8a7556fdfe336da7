"""Pins for the oracle's store (quantise, pack, write) path."""

import math

import numpy as np
import pytest

from oracle import codebook as cb
from oracle import decode as od
from oracle import layout as L
from oracle import numerics
from oracle import store as st


def test_pack_bit_order_examples():
    # 4-bit: even coordinate in the low nibble
    assert st.pack_bits(np.array([[0x3, 0xA, 0xF, 0x1]]), 4).tolist() == [[0xA3, 0x1F]]
    # 3-bit: 8 indices in a little-endian 24-bit group, index i at bits 3i..3i+2
    idx = np.array([[1, 2, 3, 4, 5, 6, 7, 0]])
    word = sum(int(v) << (3 * i) for i, v in enumerate(idx[0]))
    assert st.pack_bits(idx, 3).tolist() == [[word & 0xFF, (word >> 8) & 0xFF, word >> 16]]


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5, 8])
def test_pack_unpack_identity(bits):
    rng = np.random.default_rng(bits)
    idx = rng.integers(0, 2 ** bits, size=(17, 128))
    packed = st.pack_bits(idx, bits)
    assert packed.shape == (17, math.ceil(128 * bits / 8))
    assert np.array_equal(st.unpack_bits(packed, bits, 128), idx)


def _keys(n=300, seed=0):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((n, 128))
    k[:, 5] *= 8
    return k.astype(np.float16).astype(np.float64)


@pytest.mark.parametrize("bits", [3, 4])
def test_bucketize_is_nearest_centroid(bits):
    c = cb.codebook(128, bits)
    m = cb.midpoints_fp32(c)
    info = st.quantize_keys(_keys(), c, m, bits, True)
    y = info["y"].astype(np.float32).astype(np.float64)
    dist = np.abs(y[:, :, None] - c.astype(np.float64)[None, None, :])
    brute = dist.argmin(axis=-1)
    # exact ties between two centroids are the only allowed disagreement
    sd = np.sort(dist, axis=-1)
    tie = np.isclose(sd[..., 0], sd[..., 1], rtol=0, atol=1e-9)
    assert np.array_equal(info["idx"][~tie], brute[~tie])


def test_norm_correction_identity():
    c = cb.codebook(128, 4)
    m = cb.midpoints_fp32(c)
    k = _keys(seed=1)
    info = st.quantize_keys(k, c, m, 4, True)
    stored = numerics.fp16_value(info["norm_bits"])
    recon = stored[:, None] * c.astype(np.float64)[info["idx"]]
    rel = np.abs(np.linalg.norm(recon, axis=1) / np.linalg.norm(k, axis=1) - 1)
    assert np.all(rel <= 2.0 ** -11 + 1e-9)          # fp16 rounding of the stored norm
    raw = st.quantize_keys(k, c, m, 4, False)
    assert np.array_equal(numerics.fp16_value(raw["norm_bits"]),
                          numerics.fp16_value(numerics.fp16_bits(np.linalg.norm(k, axis=1))))


def _fill(preset_name, n_tok=40, n_kv=2, bs=32, num_blocks=5, slots=None, seed=0):
    preset = L.PRESETS[preset_name]
    lay = L.tile_layout(preset, 128, bs, n_kv)
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((n_tok, n_kv, 128)).astype(np.float16).astype(np.float64)
    v = rng.standard_normal((n_tok, n_kv, 128)).astype(np.float16).astype(np.float64)
    if slots is None:
        slots = rng.permutation(num_blocks * bs)[:n_tok]
    c = None if preset.key_fp8 else cb.codebook(128, preset.key_bits)
    m = None if preset.key_fp8 else cb.midpoints_fp32(c)
    cache = np.zeros(num_blocks * lay.block_bytes, dtype=np.uint8)
    info, skipped = st.store(k, v, slots, cache, lay, preset, c, m)
    return preset, lay, k, v, np.asarray(slots), cache, info, skipped


@pytest.mark.parametrize("name", list(L.PRESETS))
def test_written_fields_read_back(name):
    preset, lay, k, v, slots, cache, info, _ = _fill(name)
    n_tok, n_kv, _ = k.shape
    blocks, offs = slots // lay.block_size, slots % lay.block_size
    for h in range(n_kv):
        kb, vb, kn, vs, vz = od.read_positions(cache, lay, blocks, offs, h)
        rows = np.arange(n_tok) * n_kv + h
        assert np.array_equal(kb, info["k"]["packed"][rows])
        assert np.array_equal(vb, info["v"]["packed"][rows])
        assert np.array_equal(vs, info["v"]["scale_bits"][rows])
        assert np.array_equal(vz, info["v"]["zero_bits"][rows])
        if preset.key_fp8:
            assert kn is None
            assert np.array_equal(kb, numerics.e4m3_encode(k[:, h]))
        else:
            assert np.array_equal(kn, info["k"]["norm_bits"][rows])


def test_negative_and_out_of_range_slots_write_nothing():
    bs, nb = 16, 3
    slots = np.array([-1, 5, -7, 3 * 16 + 2, 17])
    preset, lay, k, v, slots, cache, info, skipped = _fill("4bit_nc", n_tok=5, bs=bs, num_blocks=nb, slots=slots)
    assert skipped == [(3, 3 * 16 + 2)]
    ref = np.zeros_like(cache)
    _, _, _, _, _, ref, _, _ = _fill("4bit_nc", n_tok=5, bs=bs, num_blocks=nb,
                                     slots=np.array([-1, 5, -1, -1, 17]))
    assert np.array_equal(cache, ref)
    # only the two valid slots' tiles are touched
    touched = np.nonzero(cache)[0]
    tiles = set(touched // lay.tile_bytes)
    assert tiles <= {(0 * lay.n_kv + h) * lay.tiles_per_block for h in range(2)} | \
        {(1 * lay.n_kv + h) * lay.tiles_per_block for h in range(2)}


def test_value_pair_interleave_layout():
    # tokens 6 and 7 form pair 3: their 16-bit words interleave, four words of
    # each per 16-byte group, and group r is stored at slot r ^ (2 * (3 & 3))
    preset, lay, k, v, slots, cache, info, _ = _fill("4bit_nc", n_tok=2, n_kv=1, bs=16,
                                                     num_blocks=1, slots=np.array([6, 7]))
    a = info["v"]["packed"][0].reshape(8, 4, 2)   # [group][word][byte]
    b = info["v"]["packed"][1].reshape(8, 4, 2)
    region = cache[lay.v_off + 3 * 2 * lay.vb: lay.v_off + 4 * 2 * lay.vb].reshape(8, 4, 2, 2)
    for r in range(8):
        slot = r ^ 6
        assert np.array_equal(region[slot, :, 0, :], a[r])
        assert np.array_equal(region[slot, :, 1, :], b[r])


def test_exact_tie_goes_to_upper_cell():
    # k = e0 + e1 rotates to coordinates (h_i0 + h_i1) / sqrt(2 d): exactly 0
    # wherever h_i1 = -1, and 0 is the middle midpoint; ">=" sends it right.
    c = cb.codebook(128, 4)
    m = cb.midpoints_fp32(c)
    k = np.zeros((1, 128))
    k[0, 0] = k[0, 1] = 1.0
    info = st.quantize_keys(k, c, m, 4, True)
    h = np.array([(-1) ** bin(i & 1).count("1") for i in range(128)])
    zero_coords = h == -1
    assert np.all(info["y"][0, zero_coords] == 0.0)
    assert np.all(info["idx"][0, zero_coords] == 8)
    assert np.all(info["idx"][0, ~zero_coords] > 8)
