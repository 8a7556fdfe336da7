"""Pins for the oracle's Lloyd-Max codebook against values fixed outside it.

* the pages' printed codebook at d = 128 (golden fixture);
* textbook Lloyd-Max quantisers of the unit Gaussian (J. Max, "Quantizing for
  minimum distortion", IRE Trans. Inf. Theory 6(1), 1960, Table I);
* the 1-bit closed form +-sigma sqrt(2/pi);
* conditional means and distortion by independent numerical integration
  (scipy.integrate.quad), not by the oracle's own closed form.
"""

import json
import math
import os

import numpy as np
import pytest
from scipy import integrate

from oracle import codebook as cb

pytestmark = pytest.mark.filterwarnings("ignore::scipy.integrate.IntegrationWarning")


def _pdf(x, sigma):
    return math.exp(-0.5 * (x / sigma) ** 2) / (sigma * math.sqrt(2 * math.pi))


def _cell_mean(a, b, sigma):
    m0 = integrate.quad(lambda x: _pdf(x, sigma), a, b, epsabs=0, epsrel=1e-13, limit=200)[0]
    m1 = integrate.quad(lambda x: x * _pdf(x, sigma), a, b, epsabs=0, epsrel=1e-13, limit=200)[0]
    return m1 / m0


@pytest.mark.parametrize("bits", [3, 4])
def test_matches_printed_codebook(golden_dir, bits):
    g = json.load(open(os.path.join(golden_dir, "codebook_d128.json")))
    c = cb.codebook(128, bits)
    pos = c[len(c) // 2:]
    printed = np.array(g["positive_half"][str(bits)])
    assert np.max(np.abs(pos - printed)) <= g["printed_precision"]


# Max (1960), unit variance, positive half of the output levels and the MSE.
MAX_TABLE = {
    2: ([0.4528, 1.510], 0.1175),
    3: ([0.2451, 0.7560, 1.344, 2.152], 0.03455),
    4: ([0.1284, 0.3881, 0.6568, 0.9424, 1.256, 1.618, 2.069, 2.733], 0.009497),
}


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_matches_textbook_gaussian_quantiser(bits):
    c, _ = cb.lloyd_max_gaussian(bits, 1.0)
    levels, _ = MAX_TABLE[bits]
    np.testing.assert_allclose(c[len(c) // 2:], levels, rtol=0, atol=1.5e-3)


def test_one_bit_closed_form():
    sigma = 1 / math.sqrt(64)
    c, _ = cb.lloyd_max_gaussian(1, sigma)
    expect = sigma * math.sqrt(2 / math.pi)
    assert abs(c[1] - expect) < 1e-14 and abs(c[0] + expect) < 1e-14


@pytest.mark.parametrize("d,bits", [(128, 3), (128, 4), (64, 4), (256, 3)])
def test_antisymmetric_and_sorted(d, bits):
    c = cb.codebook(d, bits)
    assert c.dtype == np.float32
    assert np.all(np.diff(c) > 0)
    assert np.array_equal(c, -c[::-1])


@pytest.mark.parametrize("bits", [3, 4])
def test_centroids_are_conditional_means(bits):
    d = 128
    sigma = 1 / math.sqrt(d)
    c = cb.codebook(d, bits).astype(np.float64)
    edges = [-math.inf] + list((c[:-1] + c[1:]) / 2) + [math.inf]
    for i in range(len(c)):
        a, b = edges[i], edges[i + 1]
        a = -12 * sigma if a == -math.inf else a
        b = 12 * sigma if b == math.inf else b
        assert abs(_cell_mean(a, b, sigma) - c[i]) < 1e-6


@pytest.mark.parametrize("bits", [3, 4])
def test_distortion_against_textbook_and_high_rate(golden_dir, bits):
    d = 128
    sigma = 1 / math.sqrt(d)
    c = cb.codebook(d, bits).astype(np.float64)
    edges = [-12 * sigma] + list((c[:-1] + c[1:]) / 2) + [12 * sigma]
    mse = sum(integrate.quad(lambda x, ci=c[i]: (x - ci) ** 2 * _pdf(x, sigma),
                             edges[i], edges[i + 1], epsabs=0, epsrel=1e-12, limit=200)[0]
              for i in range(len(c)))
    unit_vector_nmse = d * mse            # d coordinates of variance 1/d
    _, textbook = MAX_TABLE[bits]
    assert abs(unit_vector_nmse - textbook) / textbook < 2e-3
    hr = json.load(open(os.path.join(golden_dir, "distortion.json")))["nmse_high_rate"][str(bits)]
    assert unit_vector_nmse < hr          # the high-rate formula is an upper estimate here
    assert unit_vector_nmse > 0.75 * hr


def test_midpoints_fp32_rule():
    c = cb.codebook(128, 4)
    m = cb.midpoints_fp32(c)
    assert m.dtype == np.float32 and len(m) == 15
    # fp32 arithmetic, done independently with numpy float32 ops
    expect = (c[:-1] + c[1:]) / np.float32(2)
    assert np.array_equal(m, expect)
    assert m[7] == 0.0
    assert np.all(m > c[:-1]) and np.all(m < c[1:])


def test_spacing_remarks(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "distortion.json")))
    c4 = cb.codebook(128, 4).astype(np.float64)
    c3 = cb.codebook(128, 3).astype(np.float64)
    # "centre spacing" read as the gap between the two innermost positive levels
    assert abs((c4[9] - c4[8]) - g["spacing_4bit"]["centre"]) < 1e-3
    assert abs((c4[15] - c4[14]) - g["spacing_4bit"]["tail"]) < 1.5e-3
    assert abs((c3[5] - c3[4]) - g["spacing_3bit"]["centre"]) < 1.5e-3
    assert abs((c3[7] - c3[6]) - g["spacing_3bit"]["tail"]) < 1.5e-3
