"""Pins of the Lloyd-Max N(0,1) codebook.

Closed form at 1 bit (+-sqrt(2/pi)); Max's published Gaussian tables (J. Max,
"Quantizing for minimum distortion", IRE Trans. Inf. Theory, 1960, Table I) at
2, 3 and 4 bits; the centroid condition and the distortion by numerical
quadrature (independent of the closed forms the oracle uses); Monte Carlo on
N(0,1) samples against the distortion.
"""
import math

import numpy as np
import pytest
from scipy.integrate import quad
from scipy.stats import norm

from oracle.codebook import codebook, distortion, lloyd_max_gaussian, quantize_unit

MAX_TABLE = {
    2: ([0.4528, 1.5104], 0.1175),
    3: ([0.2451, 0.7560, 1.3440, 2.1520], 0.03455),
    4: ([0.1284, 0.3881, 0.6568, 0.9424, 1.2562, 1.6180, 2.0690, 2.7326], 0.009497),
}


def test_one_bit_closed_form():
    c = lloyd_max_gaussian(1)
    assert c[1] == pytest.approx(math.sqrt(2 / math.pi), abs=1e-14)
    assert distortion(c) == pytest.approx(1 - 2 / math.pi, abs=1e-14)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_max_table(bits):
    levels, d = MAX_TABLE[bits]
    c = lloyd_max_gaussian(bits)
    n = len(c)
    assert np.all(np.diff(c) > 0)
    np.testing.assert_allclose(c[n // 2:], levels, atol=1.5e-4)
    np.testing.assert_allclose(c, -c[::-1], atol=0)
    # the table prints 4 significant digits
    assert distortion(c) == pytest.approx(d, rel=1e-3)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_centroid_condition_by_quadrature(bits):
    c = lloyd_max_gaussian(bits)
    t = np.concatenate(([-np.inf], 0.5 * (c[:-1] + c[1:]), [np.inf]))
    for i in range(len(c)):
        mass = quad(norm.pdf, t[i], t[i + 1], epsabs=1e-13, epsrel=1e-12)[0]
        mean = quad(lambda x: x * norm.pdf(x), t[i], t[i + 1],
                    epsabs=1e-13, epsrel=1e-12)[0] / mass
        assert c[i] == pytest.approx(mean, abs=1e-9)


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_distortion_by_quadrature(bits):
    c = lloyd_max_gaussian(bits)
    t = np.concatenate(([-np.inf], 0.5 * (c[:-1] + c[1:]), [np.inf]))
    d = sum(quad(lambda x, ci=ci: (x - ci) ** 2 * norm.pdf(x), t[i], t[i + 1],
                 epsabs=1e-15, epsrel=1e-13)[0] for i, ci in enumerate(c))
    assert distortion(c) == pytest.approx(d, rel=1e-10)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_thresholds_are_fp32_midpoints(bits):
    lv, lv32, thr = codebook(bits)
    assert thr.dtype == np.float32 and lv32.dtype == np.float32
    mids = 0.5 * (lv[:-1] + lv[1:])
    assert np.all(np.abs(thr.astype(np.float64) - mids) <= np.spacing(np.float32(np.abs(mids) + 1e-30)))
    assert thr[len(thr) // 2] == 0.0


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_unit_scale_mse_matches_distortion(bits):
    """Quantize -> dequantize MSE on N(0,1) equals the codebook's distortion."""
    lv, _, thr = codebook(bits)
    rng = np.random.default_rng(1234 + bits)
    n = 2_000_000
    x = rng.standard_normal(n).astype(np.float32)
    err = (x.astype(np.float64) - lv[quantize_unit(x, thr)]) ** 2
    mse = err.mean()
    sigma = err.std() / math.sqrt(n)
    assert abs(mse - distortion(lv)) < 4 * sigma


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_nearest_level(bits):
    """The threshold rule picks the nearest level (brute force over levels)."""
    lv, lv32, thr = codebook(bits)
    v = np.linspace(-4, 4, 20001).astype(np.float32)
    codes = quantize_unit(v, thr)
    dist = np.abs(v.astype(np.float64)[:, None] - lv[None, :])
    best = np.argmin(dist, axis=1)
    near_tie = np.sort(dist, axis=1)[:, 1] - np.sort(dist, axis=1)[:, 0] < 1e-6
    assert np.all((codes == best) | near_tie)
