"""Pins of the E4M3 / BF16 encoders: torch's float8_e4m3fn and bfloat16 casts
(library special cases) plus hand-checked points of the E4M3 definition."""
import numpy as np
import pytest
import torch

from oracle.numformats import (bf16_decode, bf16_encode, e2m1_decode, e2m1_encode,
                               e4m3_decode, e4m3_encode)


def test_e4m3_decode_all_codes_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.nanmax(ours) == 448.0
    assert ours[1] == 2.0 ** -9


def test_e4m3_roundtrip_all_finite():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    assert np.array_equal(e4m3_encode(e4m3_decode(codes)), codes)


def test_e4m3_encode_vs_torch_in_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(300_000) * np.exp(rng.uniform(-12, 6, 300_000)),
        rng.uniform(-448, 448, 100_000),
    ]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e4m3_encode(x), ref)


def test_e4m3_midpoints_round_to_even():
    vals = e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = 0.5 * (vals[:-1] + vals[1:])
    got = e4m3_encode(mids)
    lower = np.arange(0x7E, dtype=np.uint8)
    expect = np.where(lower % 2 == 0, lower, lower + 1).astype(np.uint8)
    assert np.array_equal(got, expect)


@pytest.mark.parametrize("x,code", [
    (448.0, 0x7E), (464.0, 0x7E), (1e9, 0x7E), (np.inf, 0x7E), (-500.0, 0xFE),
    (2.0 ** -9, 0x01), (2.0 ** -10, 0x00), (0.75 * 2.0 ** -9, 0x01),
    (0.5, 0x30), (1.0, 0x38), (0.36596, 0x2C), (0.0, 0x00), (-0.0, 0x80),
])
def test_e4m3_points(x, code):
    assert int(e4m3_encode(np.float32(x))) == code


def test_bf16_vs_torch():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(500_000) * np.exp(rng.uniform(-30, 30, 500_000))).astype(np.float32)
    # exact ties: low half 0x8000 with even and odd kept parts
    ties = (np.arange(1000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    x = np.concatenate([x, ties, np.array([0.0, -0.0, 1.0, 3.0e38], np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.uint16).numpy()
    assert np.array_equal(bf16_encode(x), ref)
    assert np.array_equal(bf16_decode(bf16_encode(x)),
                          torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_e2m1_decode_table():
    """E2M1: sign bit 3, exponent bits 2-1 (bias 1), mantissa bit 0; exponent 0
    is subnormal (0, 0.5).  Written out by hand."""
    want = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    got = e2m1_decode(np.arange(16, dtype=np.uint8))
    assert list(got[:8]) == want
    assert list(-got[8:]) == want


def test_e2m1_roundtrip_all_codes():
    codes = np.arange(16, dtype=np.uint8)
    assert np.array_equal(e2m1_encode(e2m1_decode(codes)), codes)   # -0.0 -> 0x8 too


@pytest.mark.parametrize("x,code", [
    (0.25, 0x0), (0.75, 0x2), (1.25, 0x2), (1.75, 0x4), (2.5, 0x4), (3.5, 0x6), (5.0, 0x6),
    (0.26, 0x1), (0.74, 0x1), (1.26, 0x3), (4.99, 0x6), (5.01, 0x7), (6.0, 0x7), (1e9, 0x7),
    (-0.25, 0x8), (-0.3, 0x9), (-5.01, 0xF), (0.0, 0x0), (-0.0, 0x8), (1e-30, 0x0)])
def test_e2m1_points(x, code):
    """Midpoints go to the even code; beyond 6 saturates; sign from the sign bit."""
    assert int(e2m1_encode(np.float32(x))) == code
