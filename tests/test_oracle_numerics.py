"""Pins for the oracle's number formats and fixed-precision value quantiser."""

import struct

import numpy as np
import pytest
import torch

from oracle import numerics


def f32(x: float) -> float:
    """Round a Python float to IEEE single precision (struct round trip)."""
    return struct.unpack("<f", struct.pack("<f", x))[0]


def test_fp16_round_to_nearest_even():
    one = 1.0
    ulp = 2.0 ** -10
    assert numerics.fp16_value(numerics.fp16_bits(one + ulp / 2)) == 1.0          # tie -> even
    assert numerics.fp16_value(numerics.fp16_bits(one + 3 * ulp / 2)) == 1 + 2 * ulp
    assert numerics.fp16_value(numerics.fp16_bits(65504.0)) == 65504.0
    rng = np.random.default_rng(0)
    x = rng.standard_normal(20000) * 30
    ref = torch.tensor(x).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(numerics.fp16_bits(x), ref)


def test_e4m3_table_and_encoder():
    t = numerics.e4m3_decode_table()
    assert t[0x7E] == 448.0 and t[0xFE] == -448.0
    assert t[0x08] == 2.0 ** -6 and t[0x01] == 2.0 ** -9
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    codes = np.arange(256, dtype=np.uint8)
    finite = ~np.isnan(t)
    # every finite code round-trips (the two zeros map to the sign-preserving code)
    assert np.array_equal(numerics.e4m3_encode(t[finite]), codes[finite])
    rng = np.random.default_rng(1)
    # float32-exact inputs: torch rounds float64 through float32 first
    x = (rng.standard_normal(50000) * 40).astype(np.float32).astype(np.float64)
    x = x[np.abs(x) < 448]
    ref = torch.tensor(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(numerics.e4m3_encode(x), ref)
    assert numerics.e4m3_encode(np.array([1e6, -1e6])).tolist() == [0x7E, 0xFE]
    # halfway between 1.0 (mantissa 0) and 1.125 (mantissa 1) goes to the even one
    assert numerics.e4m3_encode(np.array([1.0625]))[0] == 0x38


@pytest.mark.parametrize("bits", [3, 4])
def test_value_quant_matches_single_precision_steps(bits):
    rng = np.random.default_rng(2)
    v = (rng.standard_normal((40, 128)) * 3).astype(np.float16).astype(np.float64)
    q, s, mn = numerics.value_quant_fp32(v, bits)
    levels = 2 ** bits - 1
    for r in range(v.shape[0]):
        lo, hi = f32(min(v[r])), f32(max(v[r]))
        sr = f32(f32(hi - lo) / levels)
        sr = sr if sr > f32(1e-8) else f32(1e-8)
        assert s[r] == np.float32(sr) and mn[r] == np.float32(lo)
        for i in range(128):
            t = f32(f32(f32(v[r, i]) - lo) / sr) + 0.5
            t = f32(t)
            assert q[r, i] == min(max(int(t), 0), levels)


@pytest.mark.parametrize("bits", [3, 4])
def test_value_quant_invariants(bits):
    rng = np.random.default_rng(5)
    v = (rng.standard_normal((200, 128)) * 2).astype(np.float16).astype(np.float64)
    q, s, mn = numerics.value_quant_fp32(v, bits)
    levels = 2 ** bits - 1
    assert np.all(q[np.arange(200), v.argmin(1)] == 0)
    assert np.all(q[np.arange(200), v.argmax(1)] == levels)
    s16 = numerics.fp16_value(numerics.fp16_bits(s))
    z16 = numerics.fp16_value(numerics.fp16_bits(mn))
    vhat = s16[:, None] * q + z16[:, None]
    fp16_slack = (np.abs(s16 - s) * levels + np.abs(z16 - mn))[:, None]
    assert np.all(np.abs(vhat - v) <= s[:, None] / 2 * (1 + 1e-6) + fp16_slack + 1e-12)


def test_value_quant_constant_vector():
    v = np.full((1, 128), 0.3125)
    q, s, mn = numerics.value_quant_fp32(v, 4)
    assert np.all(q == 0) and s[0] == np.float32(1e-8) and mn[0] == np.float32(0.3125)
    vhat = numerics.fp16_value(numerics.fp16_bits(s))[0] * q + numerics.fp16_value(numerics.fp16_bits(mn))[0]
    assert np.all(vhat == 0.3125)
