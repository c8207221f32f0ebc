"""Pins of the rotation: orthonormal and self-inverse, closed forms, and the
fp32 fast transform against the fp64 matrix product."""
import math

import numpy as np
import pytest

from oracle.wht import fwht_f32, wht_f64


@pytest.mark.parametrize("n", [16, 64, 128, 256])
def test_orthonormal_self_inverse(n):
    eye = np.eye(n)
    h = wht_f64(eye)
    np.testing.assert_allclose(h @ h, eye, atol=1e-12)
    np.testing.assert_allclose(h, h.T, atol=0)
    x = np.random.default_rng(n).standard_normal((8, n))
    np.testing.assert_allclose(np.linalg.norm(wht_f64(x), axis=1),
                               np.linalg.norm(x, axis=1), rtol=1e-12)
    np.testing.assert_allclose(wht_f64(wht_f64(x)), x, atol=1e-12)


@pytest.mark.parametrize("n", [64, 128, 256])
def test_closed_forms(n):
    e0 = np.zeros(n)
    e0[0] = 1
    np.testing.assert_allclose(wht_f64(e0), np.full(n, 1 / math.sqrt(n)), atol=1e-15)
    np.testing.assert_allclose(wht_f64(np.ones(n)), math.sqrt(n) * e0, atol=1e-12)
    # fp32 fast transform: same closed forms
    np.testing.assert_allclose(fwht_f32(e0.astype(np.float32)),
                               np.full(n, 1 / math.sqrt(n)), rtol=1e-7)
    np.testing.assert_allclose(fwht_f32(np.ones(n, np.float32)), math.sqrt(n) * e0,
                               atol=1e-6)
    # row k of the Sylvester matrix: sign of (-1)^popcount(k & j)
    k = 5
    ek = np.zeros(n, np.float32)
    ek[k] = 1
    signs = np.array([(-1) ** bin(k & j).count("1") for j in range(n)])
    np.testing.assert_allclose(fwht_f32(ek), signs / math.sqrt(n), rtol=1e-7)


@pytest.mark.parametrize("n", [64, 128, 256])
def test_fast_f32_matches_f64(n):
    x = np.random.default_rng(3).standard_normal((1000, n)).astype(np.float32)
    y32 = fwht_f32(x).astype(np.float64)
    y64 = wht_f64(x.astype(np.float64))
    scale = np.abs(x).max(axis=1, keepdims=True)
    # log2(n) add stages + one multiply: a few fp32 ulps of the row scale
    assert np.max(np.abs(y32 - y64) / scale) < (math.log2(n) + 2) * 2 ** -23 * math.sqrt(n)
