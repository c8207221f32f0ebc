"""Pins of the oracle's cache write.

* Hand-worked groups (tests/golden/turbo_groups.txt, derived by hand from the
  format descriptions of "spark_runtime/kv_cache.rs"), NVFP4 included.
* "Turbo4 ~2x lower MSE than NVFP4 at the same bit rate" ("spark_runtime/
  kv_cache.rs", KvCacheDtype::Turbo4): the direction and a loose band.
* Packing: brute-force round trips and an independent big-integer packing.
* Layout: the [num_blocks, block_size, num_kv_heads, head_dim] layout of the
  "metrale_model_layers/.../kv_cache_bf16k_turbov.rs" invariants read back
  with numpy's row-major reshape; slot -> (slot // bs, slot % bs) from
  "combs_models/kv.rs" PagedKVCache::attention.
* Strided input rows (key_stride / value_stride) equal contiguous rows.
"""
import os

import numpy as np
import pytest

import oracle.formats as F
from oracle.cache_write import (cache_write, pack_codes, quantize_nvfp4, quantize_rotated,
                                quantize_rows, unpack_codes)
from oracle.codebook import codebook
from oracle.numformats import bf16_encode
from oracle.wht import fwht_f32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "turbo_groups.txt")


def load_golden():
    cases = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, fmt, inputs, scales, data = [p.strip() for p in line.split("|")]
        cases.append((name, fmt, inputs, bytes.fromhex(scales), bytes.fromhex(data)))
    return cases


@pytest.mark.parametrize("case", load_golden(), ids=lambda c: c[0])
def test_hand_worked_groups(case):
    name, fmt, inputs, scales, data = case
    if inputs == "half_levels":
        lv32 = codebook(F.CODE_BITS[fmt])[1]
        y = np.float32(0.5) * lv32[np.arange(16) % len(lv32)]
    else:
        y = np.array([float(v) for v in inputs.split()], np.float32)
    assert y.shape == (16,)
    if fmt == "nvfp4":
        enc, sc = quantize_nvfp4(y[None, :])
    else:
        enc, sc = quantize_rotated(fmt, y[None, :])
    if fmt == "turbo8":
        got_data = enc[0].tobytes()
        got_scale = sc.astype("<u2").tobytes()
    else:
        got_data = pack_codes(enc[0], F.CODE_BITS[fmt]).tobytes()
        got_scale = sc.tobytes()
    assert got_scale == scales
    assert got_data == data


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_pack_roundtrip_exhaustive(bits):
    n = 1 << bits
    # every ordered pair of codes at every position inside an 8-code window
    codes = np.array([[a, b] + [0] * 6 for a in range(n) for b in range(n)], np.uint8)
    for shift in range(7):
        c = np.roll(codes, shift, axis=1)
        assert np.array_equal(unpack_codes(pack_codes(c, bits), bits, 8), c)
    rng = np.random.default_rng(bits)
    c = rng.integers(0, n, size=(50, 256), dtype=np.uint8)
    assert np.array_equal(unpack_codes(pack_codes(c, bits), bits, 256), c)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_pack_matches_integer_stream(bits):
    rng = np.random.default_rng(10 + bits)
    for _ in range(200):
        c = rng.integers(0, 1 << bits, size=64, dtype=np.uint8)
        big = sum(int(v) << (bits * i) for i, v in enumerate(c))
        assert pack_codes(c, bits).tobytes() == big.to_bytes(64 * bits // 8, "little")


def test_rows_are_rotated_then_grouped():
    x = np.random.default_rng(5).standard_normal((10, 128)).astype(np.float32)
    for side in ("turbo2", "turbo3", "turbo4", "turbo8"):
        a = quantize_rows(side, x)
        b = quantize_rotated(side, fwht_f32(x))
        assert all(np.array_equal(u, v) for u, v in zip(a, b))


@pytest.mark.parametrize("side", ["bf16", "fp8", "turbo4", "turbo3", "turbo2", "turbo8"])
def test_layout_and_slots(side):
    bs, nkv, hd, nblocks = 16, 2, 64, 5
    stride = F.block_bytes(side, bs, nkv, hd) + 32   # padded stride is allowed
    rng = np.random.default_rng(7)
    slots = np.array([17, 3, -1, 79, 40], np.int64)
    x = rng.standard_normal((5, nkv, hd)).astype(np.float32)
    cache = np.zeros(nblocks * stride, np.uint8)
    cache_write(side, x, cache, slots, nkv, hd, bs, stride, scale=0.05)
    dsec = F.data_section_bytes(side, bs, nkv, hd)
    ssec = F.block_bytes(side, bs, nkv, hd) - dsec
    blocks = cache.reshape(nblocks, stride)
    written = np.zeros((nblocks, bs), bool)
    for t, slot in enumerate(slots):
        if slot < 0:
            continue
        b, o = divmod(int(slot), bs)
        written[b, o] = True
        enc, sc = quantize_rows(side, x[t], scale=0.05)
        if side == "bf16":
            view = blocks[:, :dsec].copy().view("<u2").reshape(nblocks, bs, nkv, hd)
            assert np.array_equal(view[b, o], enc)
        elif side in ("fp8", "turbo8"):
            view = blocks[:, :dsec].reshape(nblocks, bs, nkv, hd)
            assert np.array_equal(view[b, o], enc)
        else:
            bits = F.CODE_BITS[side]
            codes = unpack_codes(blocks[:, :dsec], bits, bs * nkv * hd)
            assert np.array_equal(codes.reshape(nblocks, bs, nkv, hd)[b, o], enc)
        if side == "turbo8":
            sview = blocks[:, dsec:dsec + ssec].copy().view("<u2").reshape(nblocks, bs, nkv, hd // 16)
            assert np.array_equal(sview[b, o], sc)
        elif side not in ("bf16", "fp8"):
            sview = blocks[:, dsec:dsec + ssec].reshape(nblocks, bs, nkv, hd // 16)
            assert np.array_equal(sview[b, o], sc)
    # untouched rows and the padding stay zero
    assert not blocks[:, F.block_bytes(side, bs, nkv, hd):].any()
    if side == "bf16":
        view = blocks[:, :dsec].copy().view("<u2").reshape(nblocks, bs, nkv, hd)
        assert not view[~written].any()


def test_strided_rows_equal_contiguous():
    nq, nkv, hd, t = 4, 2, 64, 9
    row = (nq + 2 * nkv) * hd + 64
    rng = np.random.default_rng(9)
    fused = rng.standard_normal((t, row)).astype(np.float32)
    k_view = fused[:, nq * hd:(nq + nkv) * hd].reshape(t, nkv, hd)
    slots = np.arange(t, dtype=np.int64) * 3
    stride = F.block_bytes("turbo3", 16, nkv, hd)
    a = np.zeros(4 * stride, np.uint8)
    b = np.zeros(4 * stride, np.uint8)
    cache_write("turbo3", k_view, a, slots, nkv, hd, 16, stride)
    cache_write("turbo3", fused.reshape(-1)[nq * hd:], b, slots, nkv, hd, 16, stride,
                row_stride=row)
    assert np.array_equal(a, b)


def test_bf16_side_is_rne():
    x = np.random.default_rng(2).standard_normal((3, 64)).astype(np.float32)
    enc, _ = quantize_rows("bf16", x)
    assert np.array_equal(enc, bf16_encode(x))


def test_full_pipeline_mse_report():
    """Reported, not pinned: the group scale amax/c_max stretches each group to
    the outer level, so the pipeline's MSE is not the unit-scale distortion."""
    x = np.random.default_rng(4).standard_normal((4096, 128)).astype(np.float32)
    from oracle.decode import dequantize_rows
    from oracle.cache_write import encode_rows_bytes
    from oracle.wht import wht_f64
    for side in ("turbo2", "turbo3", "turbo4", "turbo8"):
        d, s = encode_rows_bytes(side, x)
        back = wht_f64(dequantize_rows(side, d, s, 128))
        mse = np.mean((back - x) ** 2)
        assert mse < {"turbo2": 0.2, "turbo3": 0.06, "turbo4": 0.02, "turbo8": 0.002}[side]


def test_turbo4_beats_nvfp4_mse():
    """KvCacheDtype::Turbo4's doc claims ~2x lower MSE than NVFP4 at the same
    bit rate.  With the readings here (NVFP4 scale amax/6, Turbo4 scale
    amax/c_max after the WHT) the ratio on N(0,1) rows, with and without
    outlier channels, is ~1.55: Turbo4 is better, by less than the page's
    round number.  Pinned: the direction and a band around the measured ratio."""
    from oracle.decode import dequantize_rows
    from oracle.cache_write import encode_rows_bytes
    from oracle.wht import wht_f64
    rng = np.random.default_rng(5)
    gauss = rng.standard_normal((4096, 128)).astype(np.float32)
    out = (gauss * np.where(rng.random(128) < 0.02, 10.0, 1.0)).astype(np.float32)
    for x in (gauss, out):
        mse = {}
        for side in ("turbo4", "nvfp4"):
            d, sc = encode_rows_bytes(side, x)
            back = dequantize_rows(side, d, sc, 128)
            if side == "turbo4":
                back = wht_f64(back)
            mse[side] = np.mean((back - x) ** 2) / np.mean(x.astype(np.float64) ** 2)
        ratio = mse["nvfp4"] / mse["turbo4"]
        assert 1.3 < ratio < 2.5, ratio


def test_nvfp4_is_not_rotated_and_dequantizes_to_e2m1_grid():
    """NVFP4 stores x itself (is_wht_rotated lists the Turbo sides only): a
    row whose groups are already on the E2M1 grid times a power of two comes
    back exactly."""
    from oracle.decode import dequantize_rows
    from oracle.cache_write import encode_rows_bytes
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -6, -4, -3, -2, -1.5, -1, -0.5, 0], np.float32)
    x = np.concatenate([grid * 0.25, grid * 8.0])[None, :]
    d, sc = encode_rows_bytes("nvfp4", x)
    assert np.array_equal(dequantize_rows("nvfp4", d, sc, 32), x.astype(np.float64))
