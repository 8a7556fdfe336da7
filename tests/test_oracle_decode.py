"""Pins for the oracle's decode against independent formulations.

The brute-force check reconstructs every key in the ORIGINAL basis
(k = stored_norm * (H / sqrt(d)) c[idx], the inverse rotation being the same
symmetric matrix) and runs textbook softmax attention with the unrotated
query, so a wrong rotation of q, a wrong norm or a wrong GQA mapping in the
oracle's rotated-basis formula shows up as a mismatch.
"""

import math

import numpy as np
import pytest

import workloads
from oracle import codebook as cb
from oracle import decode as od
from oracle import layout as L
from oracle import numerics
from oracle import rotation
from oracle import store as st


def build(name, **over):
    w = workloads.get(name, **over)
    inp = workloads.make_inputs(w)
    preset = L.PRESETS[w.preset]
    lay = L.tile_layout(preset, w.d, w.block_size, w.n_kv)
    c = None if preset.key_fp8 else cb.codebook(w.d, preset.key_bits)
    m = None if preset.key_fp8 else cb.midpoints_fp32(c)
    cache = np.zeros(inp.num_blocks * lay.block_bytes, dtype=np.uint8)
    ks, vs = [], []
    for b in range(w.batch):
        k, v = inp.kv_for_sequence(b)
        ks.append(k.double().numpy())
        vs.append(v.double().numpy())
    st.store(np.concatenate(ks), np.concatenate(vs), inp.fill_slots.numpy(), cache, lay, preset, c, m)
    return w, inp, preset, lay, c, cache, ks, vs


def brute_force(w, inp, preset, lay, c, cache, q):
    out = np.zeros_like(q)
    group = w.n_q // w.n_kv
    h_mat = rotation.sylvester_hadamard(w.d) / math.sqrt(w.d)
    e4m3 = numerics.e4m3_decode_table()
    for b in range(w.batch):
        length = int(inp.seq_lens[b])
        if length == 0:
            continue
        pos = np.arange(length)
        blocks = inp.block_table[b].numpy()[pos // w.block_size]
        offs = pos % w.block_size
        for h in range(w.n_q):
            kb, vb, kn, vsc, vz = od.read_positions(cache, lay, blocks, offs, h // group)
            if preset.key_fp8:
                keys = e4m3[kb]
            else:
                idx = st.unpack_bits(kb, preset.key_bits, w.d)
                keys = numerics.fp16_value(kn)[:, None] * (c.astype(np.float64)[idx] @ h_mat)
            codes = st.unpack_bits(vb, preset.value_bits, w.d)
            vals = numerics.fp16_value(vsc)[:, None] * codes + numerics.fp16_value(vz)[:, None]
            s = keys @ q[b, h] / math.sqrt(w.d)
            e = np.exp(s - s.max())
            out[b, h] = (e / e.sum()) @ vals
    return out


@pytest.mark.parametrize("name", ["tiny", "k8v4_small", "k3v4_small"])
def test_decode_matches_brute_force(name):
    w, inp, preset, lay, c, cache, _, _ = build(name)
    q = inp.q.double().numpy()
    got = od.decode(q, cache, lay, preset, c, inp.block_table.numpy(), inp.seq_lens.numpy())
    ref = brute_force(w, inp, preset, lay, c, cache, q)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-10)


def test_single_token_returns_its_value():
    w, inp, preset, lay, c, cache, _, vs = build("tiny", lens=(1, 1))
    q = inp.q.double().numpy()
    got = od.decode(q, cache, lay, preset, c, inp.block_table.numpy(), inp.seq_lens.numpy())
    blk = int(inp.block_table[0, 0])
    _, vb, _, vsc, vz = od.read_positions(cache, lay, np.array([blk]), np.array([0]), 0)
    vhat = od.dequantized_values(vb, vsc, vz, 4, 128)[0]
    np.testing.assert_allclose(got[0, 0], vhat, atol=1e-12)
    # the reconstruction is close to the input (error within half a step + fp16)
    assert np.max(np.abs(vhat - vs[0][0, 0])) < 0.5 * (vs[0][0, 0].max() - vs[0][0, 0].min()) / 15 + 1e-2


def test_zero_query_is_mean_of_values():
    w, inp, preset, lay, c, cache, _, _ = build("tiny")
    q = np.zeros((2, 1, 128))
    got = od.decode(q, cache, lay, preset, c, inp.block_table.numpy(), inp.seq_lens.numpy())
    for b in range(2):
        length = int(inp.seq_lens[b])
        pos = np.arange(length)
        blocks = inp.block_table[b].numpy()[pos // 16]
        _, vb, _, vsc, vz = od.read_positions(cache, lay, blocks, pos % 16, 0)
        np.testing.assert_allclose(got[b, 0], od.dequantized_values(vb, vsc, vz, 4, 128).mean(0), atol=1e-12)


def test_empty_sequence_gives_zeros():
    w, inp, preset, lay, c, cache, _, _ = build("tiny")
    lens = inp.seq_lens.numpy().copy()
    lens[1] = 0
    got = od.decode(inp.q.double().numpy(), cache, lay, preset, c, inp.block_table.numpy(), lens)
    assert np.all(got[1] == 0) and np.any(got[0] != 0)


def test_block_table_permutation_invariance():
    w, inp, preset, lay, c, cache, ks, vs = build("gqa_small")
    q = inp.q.double().numpy()
    ref = od.decode(q, cache, lay, preset, c, inp.block_table.numpy(), inp.seq_lens.numpy())
    # move every physical block to a new place and rewrite the table accordingly
    nb = inp.num_blocks
    perm = np.random.default_rng(9).permutation(nb)
    moved = np.zeros_like(cache)
    for old in range(nb):
        new = perm[old]
        moved[new * lay.block_bytes:(new + 1) * lay.block_bytes] = cache[old * lay.block_bytes:(old + 1) * lay.block_bytes]
    table = inp.block_table.numpy().copy()
    table[table >= 0] = perm[table[table >= 0]]
    got = od.decode(q, moved, lay, preset, c, table, inp.seq_lens.numpy())
    np.testing.assert_allclose(got, ref, atol=1e-13)


def test_gqa_head_mapping():
    # give each KV head its own constant value vector: query head h must return
    # the constant of KV head h // group
    w = workloads.get("gqa_small", lens=(20, 33, 16))
    inp = workloads.make_inputs(w)
    preset = L.PRESETS[w.preset]
    lay = L.tile_layout(preset, 128, 16, 8)
    c = cb.codebook(128, 4)
    m = cb.midpoints_fp32(c)
    cache = np.zeros(inp.num_blocks * lay.block_bytes, dtype=np.uint8)
    n = int(inp.seq_lens.sum())
    rng = np.random.default_rng(0)
    k = rng.standard_normal((n, 8, 128)).astype(np.float16).astype(np.float64)
    v = np.broadcast_to((np.arange(8) + 1.0)[None, :, None] * 0.25, (n, 8, 128)).copy()
    st.store(k, v, inp.fill_slots.numpy(), cache, lay, preset, c, m)
    got = od.decode(inp.q.double().numpy(), cache, lay, preset, c, inp.block_table.numpy(), inp.seq_lens.numpy())
    for h in range(32):
        np.testing.assert_allclose(got[:, h], 0.25 * (h // 4 + 1), atol=1e-12)


@pytest.mark.parametrize("name", ["tiny", "gqa_small"])
def test_decode_matches_brute_force_3bit_values(name):
    # 3bit_nc: 3-bit keys and 3-bit values (48-byte value rows, no swizzle)
    w, inp, preset, lay, c, cache, _, _ = build(name, preset="3bit_nc")
    assert preset.value_bits == 3 and lay.vb == 48
    q = inp.q.double().numpy()
    got = od.decode(q, cache, lay, preset, c, inp.block_table.numpy(), inp.seq_lens.numpy())
    ref = brute_force(w, inp, preset, lay, c, cache, q)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-10)
