"""Pins for the oracle's TurboQuant_prod (Lloyd-Max code + 1-bit QJL residual) keys.

The estimator's defining property is unbiasedness over the random matrix S;
it is pinned statistically (seeded S, a tolerance of 5 standard errors) and
through the closed form of the expectation it rests on. The Lloyd-Max part is
pinned against brute-force nearest centroids, the bit formats by round trips
and worked examples.
"""

import math

import numpy as np
import pytest

from oracle import codebook as cb
from oracle import qjl
from oracle import rotation


def _key_query(seed, d=128):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal(d)
    k[3] *= 6
    q = rng.standard_normal(d)
    return k.astype(np.float16).astype(np.float64), q.astype(np.float16).astype(np.float64)


def _cb(bits=2, d=128):
    c = cb.codebook(d, bits)
    return c, cb.midpoints_fp32(c)


def test_sign_expectation_closed_form():
    # E over s ~ N(0, I) of sign(<s, r>) <s, y> = sqrt(2 / pi) <r, y> / ||r||:
    # the identity that makes the QJL term unbiased
    rng = np.random.default_rng(7)
    d, n = 16, 400_000
    r, y = rng.standard_normal(d), rng.standard_normal(d)
    s = rng.standard_normal((n, d))
    samples = np.sign(s @ r) * (s @ y)
    want = math.sqrt(2 / math.pi) * (r @ y) / np.linalg.norm(r)
    se = samples.std() / math.sqrt(n)
    assert abs(samples.mean() - want) < 5 * se


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_estimate_is_unbiased_over_S(seed):
    d = 128
    k, q = _key_query(seed)
    c, m = _cb()
    trials = 3000
    rng = np.random.default_rng(100 + seed)
    est = np.empty(trials)
    for t in range(trials):
        S = rng.standard_normal((d, d))
        info = qjl.prod_quantize(k[None], S, c, m, 2)
        signs = 2.0 * info["sign_bits"].astype(np.float64) - 1.0
        est[t] = qjl.prod_estimate(q[None], S, c, info["idx"], signs, info["norm"], info["rnorm"])[0, 0]
    truth = q @ k
    se = est.std() / math.sqrt(trials)
    assert abs(est.mean() - truth) < 5 * se
    # the Lloyd-Max part alone is biased for this key (its error is not zero
    # mean over S: it does not depend on S at all), which is what the QJL term fixes
    mse_only = np.linalg.norm(k) * (rotation.rotate(q) @ c.astype(np.float64)[info["idx"][0]])
    assert abs(mse_only - truth) > 5 * se


def test_lloyd_max_part_is_the_nearest_centroid():
    c, m = _cb()
    rng = np.random.default_rng(5)
    k = rng.standard_normal((200, 128)).astype(np.float16).astype(np.float64)
    info = qjl.prod_quantize(k, rng.standard_normal((128, 128)), c, m, 2)
    y = info["y"].astype(np.float32).astype(np.float64)
    dist = np.abs(y[:, :, None] - c.astype(np.float64)[None, None, :])
    sd = np.sort(dist, axis=-1)
    tie = np.isclose(sd[..., 0], sd[..., 1], rtol=0, atol=1e-9)
    assert np.array_equal(info["idx"][~tie], dist.argmin(axis=-1)[~tie])


def test_residual_norm_and_pythagoras():
    # ||y||^2 = 1 (up to the 1e-8 in the normalisation) = ||x~||^2 + 2<x~, r> + ||r||^2
    c, m = _cb()
    rng = np.random.default_rng(6)
    k = rng.standard_normal((50, 128))
    info = qjl.prod_quantize(k, rng.standard_normal((128, 128)), c, m, 2)
    xt = c.astype(np.float64)[info["idx"]]
    r = info["residual"]
    lhs = (info["y"] ** 2).sum(-1)
    rhs = (xt ** 2).sum(-1) + 2 * (xt * r).sum(-1) + info["rnorm"] ** 2
    assert np.allclose(lhs, rhs, rtol=0, atol=1e-12)
    assert np.allclose(lhs, 1.0, rtol=0, atol=1e-6)


def test_sign_packing_examples_and_round_trip():
    bits = np.zeros((1, 16), dtype=np.uint8)
    bits[0, [0, 3, 9, 15]] = 1
    assert qjl.pack_signs(bits).tolist() == [[0b00001001, 0b10000010]]
    rng = np.random.default_rng(8)
    b = rng.integers(0, 2, size=(7, 128))
    assert np.array_equal(qjl.unpack_signs(qjl.pack_signs(b), 128), 2.0 * b - 1.0)


def test_sign_of_zero_projection_is_plus():
    c, m = _cb()
    d = 128
    S = np.zeros((d, d))                            # every projection is exactly 0
    info = qjl.prod_quantize(np.ones((1, d)), S, c, m, 2)
    assert np.all(info["sign_bits"] == 1)


def test_paged_store_and_scores_match_the_estimator():
    # the paged forms are only byte placement: scores read back from the cache
    # equal the estimator on fp16 norms, for ragged lengths and a permuted table
    d, n_kv, n_q, bs = 128, 2, 4, 16
    c, m = _cb()
    rng = np.random.default_rng(9)
    S = rng.standard_normal((d, d))
    lens = [37, 16, 0]
    nblk = [(x + bs - 1) // bs for x in lens]
    perm = rng.permutation(sum(nblk))
    table = np.full((3, max(nblk)), -1)
    at = 0
    for b, nb in enumerate(nblk):
        table[b, :nb] = perm[at: at + nb]
        at += nb
    lay = qjl.prod_tile_layout(d, bs, n_kv, 2)
    assert lay.slot_bytes == 52 and lay.tile_bytes == 832
    cache = np.zeros(sum(nblk) * lay.block_bytes, dtype=np.uint8)
    keys = []
    for b, L in enumerate(lens):
        k = rng.standard_normal((L, n_kv, d)).astype(np.float16).astype(np.float64)
        pos = np.arange(L)
        qjl.prod_store(k, table[b, pos // bs] * bs + pos % bs, S, cache, lay, c, m)
        keys.append(k)
    q = rng.standard_normal((3, n_q, d)).astype(np.float16).astype(np.float64)
    got = qjl.prod_scores(q, S, cache, lay, c, table, lens, 40)
    for b, L in enumerate(lens):
        assert np.all(got[b, :, L:] == 0)
        for h in range(n_q):
            kv = h // (n_q // n_kv)
            if L == 0:
                continue
            info = qjl.prod_quantize(keys[b][:, kv], S, c, m, 2)
            signs = 2.0 * info["sign_bits"] - 1.0
            from oracle import numerics
            n16 = numerics.fp16_value(info["norm_bits"])
            r16 = numerics.fp16_value(info["rnorm_bits"])
            want = qjl.prod_estimate(q[b, h][None], S, c, info["idx"], signs, n16, r16)[0] / math.sqrt(d)
            assert np.allclose(got[b, h, :L], want, rtol=0, atol=1e-12)
