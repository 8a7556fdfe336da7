"""Pins for the oracle's Hadamard rotation and slot/tile layout."""

import json
import math
import os

import numpy as np
import pytest
from scipy.linalg import hadamard

from oracle import layout as L
from oracle import rotation


@pytest.mark.parametrize("d", [1, 2, 4, 8, 16, 64, 128, 256])
def test_sylvester_equals_library_hadamard(d):
    assert np.array_equal(rotation.sylvester_hadamard(d), hadamard(d))


@pytest.mark.parametrize("d", [64, 128, 256])
def test_hadamard_identities(d):
    h = rotation.sylvester_hadamard(d)
    assert np.array_equal(h, h.T)
    assert np.array_equal(h @ h.T, d * np.eye(d))


def test_rotation_is_orthonormal_involution():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((50, 128))
    y = rotation.rotate(x)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    np.testing.assert_allclose(rotation.rotate(y), x, atol=1e-12)
    e0 = np.zeros(128)
    e0[0] = 1
    np.testing.assert_allclose(rotation.rotate(e0), np.full(128, 1 / math.sqrt(128)), rtol=1e-14)


def test_rotation_matches_fwht_butterfly():
    # textbook in-place Walsh-Hadamard butterfly in natural (Sylvester) order
    rng = np.random.default_rng(4)
    x = rng.standard_normal(128)
    a = x.copy()
    h = 1
    while h < 128:
        for i in range(0, 128, 2 * h):
            for j in range(i, i + h):
                a[j], a[j + h] = a[j] + a[j + h], a[j] - a[j + h]
        h *= 2
    np.testing.assert_allclose(rotation.rotate(x), a / math.sqrt(128), atol=1e-12)


def test_slot_sizes_match_pages(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "slot_sizes.json")))
    for name, row in g["presets"].items():
        key, value, slot, aligned = L.preset_slot_sizes(L.PRESETS[name], g["d"])
        assert key == row["k_data"] + row["k_meta"]
        assert value == row["v_data"] + row["v_meta"]
        assert slot == row["slot"] and aligned == row["aligned"]
        lay = L.tile_layout(L.PRESETS[name], g["d"], 16, 8)
        assert lay.slot_bytes == row["slot"]


def test_page_bytes_and_compression(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "slot_sizes.json")))
    p = g["page_example"]
    lay = L.tile_layout(L.PRESETS["k3v4_nc"], 128, p["block_size"], p["n_kv"])
    assert lay.block_bytes == p["page_bytes"]
    assert p["block_size"] * p["n_kv"] * 128 * 2 * 2 == p["fp16_page_bytes"]
    c = g["compression_example"]
    lay4 = L.tile_layout(L.PRESETS["4bit_nc"], 128, 16, 1)
    assert lay4.slot_bytes == c["pair_bytes"] == c["k_bytes"] + c["v_bytes"]
    assert round(c["bf16_bytes"] / lay4.slot_bytes, 2) == c["ratio"]


@pytest.mark.parametrize("name", list(L.PRESETS))
@pytest.mark.parametrize("bs", [16, 32, 64, 128])
def test_tile_fields_partition_the_tile(name, bs):
    lay = L.tile_layout(L.PRESETS[name], 128, bs, 8)
    used = np.zeros(lay.tile_bytes, dtype=int)
    used[lay.k_off: lay.k_off + 16 * lay.kb] += 1
    used[lay.v_off: lay.v_off + 16 * lay.vb] += 1
    if lay.has_knorm:
        used[lay.knorm_off: lay.knorm_off + 32] += 1
    used[lay.vscale_off: lay.vscale_off + 32] += 1
    used[lay.vzero_off: lay.vzero_off + 32] += 1
    assert np.all(used == 1)
    # every region and every key/value row starts on a 16-byte boundary
    assert lay.tile_bytes % 16 == 0 and lay.v_off % 16 == 0
    assert (lay.kb % 16 == 0) and ((2 * lay.vb) % 16 == 0)
    assert lay.block_bytes == bs * 8 * lay.slot_bytes
