"""Pins for the oracle's full dequantisation and its continuation-chunk decode.

Each check ties the oracle to something other than its own formula:
  * attention written in the original basis over the dequantised keys and
    values equals the oracle's rotated-basis decode (the two differ only by
    the orthonormal rotation, so a wrong inverse rotation, norm or value
    reconstruction breaks the equality);
  * with norm correction the dequantised key keeps the input key's length up
    to the fp16 rounding of the stored norm ([vLLM-TQ] "norm correction 的折叠");
  * the mean relative squared error of the keys lies close to the codebook's
    closed-form distortion d * E[(x - c)^2] (pinned in the codebook tests);
  * FP8 keys come back as the nearest e4m3 value of the input (half a unit in
    the last place of a 3-bit mantissa);
  * values lie within half a quantisation step of the input plus the fp16
    rounding of scale and zero ([vLLM-TQ] "V 的 min/max 均匀量化");
  * the continuation decode equals causal attention written with an explicit
    mask over the dequantised sequence.
"""

import math

import numpy as np
import pytest

from oracle import decode as od
from oracle import dequant as dq
from oracle import numerics
from test_oracle_decode import build

# d * E[(x - c)^2] for N(0, 1/d), the codebook tests' closed-form values
DISTORTION = {4: 0.0095010, 3: 0.0345478}


def _dequant(name, **over):
    w, inp, preset, lay, c, cache, ks, vs = build(name, **over)
    kh, vh = dq.dequantize(cache, lay, preset, c, inp.block_table.numpy(), inp.seq_lens.numpy(),
                           inp.max_seq_len)
    return w, inp, preset, lay, c, cache, ks, vs, kh, vh


@pytest.mark.parametrize("name,over", [("tiny", {}), ("gqa_small", {}), ("k3v4_small", {}), ("k8v4_small", {}),
                                       ("gqa_small", {"preset": "3bit_nc"})])
def test_original_basis_attention_equals_decode(name, over):
    w, inp, preset, lay, c, cache, _, _, kh, vh = _dequant(name, **over)
    q = inp.q.double().numpy()
    ref = od.decode(q, cache, lay, preset, c, inp.block_table.numpy(), inp.seq_lens.numpy())
    group = w.n_q // w.n_kv
    for b in range(w.batch):
        length = int(inp.seq_lens[b])
        for h in range(w.n_q):
            keys = kh[b, :length, h // group]
            vals = vh[b, :length, h // group]
            s = keys @ q[b, h] / math.sqrt(w.d)
            e = np.exp(s - s.max())
            np.testing.assert_allclose((e / e.sum()) @ vals, ref[b, h], rtol=0, atol=1e-10)


@pytest.mark.parametrize("name", ["gqa_small", "k3v4_small", "long_small"])
def test_key_length_kept_by_norm_correction(name):
    w, inp, _, _, _, _, ks, _, kh, _ = _dequant(name)
    for b in range(w.batch):
        length = int(inp.seq_lens[b])
        ratio = np.linalg.norm(kh[b, :length], axis=-1) / np.linalg.norm(ks[b], axis=-1)
        assert np.max(np.abs(ratio - 1.0)) <= 2.0 ** -11 + 1e-9


@pytest.mark.parametrize("name,bits,over", [("gqa_small", 4, {}), ("k3v4_small", 3, {}), ("long_small", 4, {}),
                                            ("gqa_small", 3, {"preset": "3bit_nc"})])
def test_key_error_near_codebook_distortion(name, bits, over):
    w, inp, _, _, _, _, ks, _, kh, _ = _dequant(name, **over)
    err = []
    for b in range(w.batch):
        length = int(inp.seq_lens[b])
        k = ks[b]
        err.append((((k - kh[b, :length]) ** 2).sum(-1) / (k * k).sum(-1)).ravel())
    mean = np.concatenate(err).mean()
    # a unit vector's rotated coordinates have slightly lighter tails than
    # N(0, 1/d), so the error sits a little below the Gaussian distortion
    assert 0.90 * DISTORTION[bits] <= mean <= 1.05 * DISTORTION[bits]


def test_fp8_keys_are_nearest_e4m3():
    w, inp, _, _, _, _, ks, _, kh, _ = _dequant("k8v4_small")
    table = numerics.e4m3_decode_table()
    finite = np.unique(table[np.isfinite(table)])
    for b in range(w.batch):
        length = int(inp.seq_lens[b])
        got = kh[b, :length]
        assert np.all(np.isin(got, finite))
        k = ks[b]
        # half an ulp of a 3-bit mantissa; below 2^-6 the subnormal step 2^-9
        half_ulp = np.where(np.abs(k) >= 2.0 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(k), 1e-30))) - 4),
                            2.0 ** -10)
        assert np.all(np.abs(got - k) <= half_ulp * (1 + 1e-12))


@pytest.mark.parametrize("name,over", [("gqa_small", {}), ("k8v4_small", {}),
                                       ("gqa_small", {"preset": "3bit_nc"})])
def test_values_within_half_step(name, over):
    w, inp, preset, _, _, _, _, vs, _, vh = _dequant(name, **over)
    top = 2 ** preset.value_bits - 1
    for b in range(w.batch):
        length = int(inp.seq_lens[b])
        v = vs[b]
        mn, mx = v.min(-1, keepdims=True), v.max(-1, keepdims=True)
        s = np.maximum((mx - mn) / top, 1e-8)
        tol = s / 2 * (1 + 1e-5) + top * s * 2.0 ** -11 + np.abs(mn) * 2.0 ** -11 + 1e-7
        assert np.all(np.abs(vh[b, :length] - v) <= tol)


def test_rows_past_the_length_are_zero():
    w, inp, _, _, _, _, _, _, kh, vh = _dequant("tiny")
    assert kh.shape == (2, 128, 1, 128)
    assert np.all(kh[0, 37:] == 0) and np.all(vh[0, 37:] == 0)
    assert np.all(np.any(kh[0, :37] != 0, axis=-1))
    w, inp, preset, lay, c, cache, _, _ = build("tiny")
    lens = inp.seq_lens.numpy().copy()
    lens[1] = 0
    kh, vh = dq.dequantize(cache, lay, preset, c, inp.block_table.numpy(), lens, 128)
    assert np.all(kh[1] == 0) and np.all(vh[1] == 0) and np.any(kh[0] != 0)


@pytest.mark.parametrize("name", ["gqa_small", "k8v4_small"])
def test_continuation_equals_masked_causal_attention(name):
    w, inp, preset, lay, c, cache, _, _, kh, vh = _dequant(name)
    b = int(np.argmax(inp.seq_lens.numpy()))
    length = int(inp.seq_lens[b])
    q_len = 23
    cached = length - q_len
    rng = np.random.default_rng(5)
    qc = rng.standard_normal((q_len, w.n_q, w.d))
    got = od.continuation_decode(qc, cache, lay, preset, c, inp.block_table.numpy()[b], cached)
    group = w.n_q // w.n_kv
    # row i of the mask admits positions 0 .. cached + i
    mask = np.arange(length)[None, :] <= cached + np.arange(q_len)[:, None]
    for h in range(w.n_q):
        s = qc[:, h] @ kh[b, :length, h // group].T / math.sqrt(w.d)
        s = np.where(mask, s, -np.inf)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        ref = (p / p.sum(axis=1, keepdims=True)) @ vh[b, :length, h // group]
        np.testing.assert_allclose(got[:, h], ref, rtol=0, atol=1e-10)
