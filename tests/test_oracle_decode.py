"""Pins of the oracle's paged decode.

* BF16 K/V: equals an independent naive softmax-attention loop in fp64
  ("combs_models/kv.rs", attend, one query, repeat_kv head mapping) to 1e-12.
* Special cases: seq_len 1 -> v_0; q = 0 -> mean of the attended V rows;
  window 1 -> the newest V row; seq_len 0 -> zeros.
* Rotated-basis identity: scores of WHT(q) against the stored (rotated)
  rows, and the output rotated back once, equal the plain definition.
"""
import math

import numpy as np
import pytest

import oracle.formats as F
from oracle.cache_write import cache_write
from oracle.decode import gather_side, paged_decode
from oracle.wht import wht_f64


def build(fmt, lens, nq=4, nkv=2, hd=64, bs=16, seed=0, k_scale=0.05, v_scale=0.05):
    rng = np.random.default_rng(seed)
    nblocks = sum(-(-n // bs) for n in lens) + 3
    perm = rng.permutation(nblocks)
    mb = max(1, max(-(-n // bs) for n in lens))
    tables = np.zeros((len(lens), mb), np.int64)
    ks, vs, cur = [], [], 0
    kside, vside = F.kv_pair(fmt)
    kstride = F.block_bytes(kside, bs, nkv, hd)
    vstride = F.block_bytes(vside, bs, nkv, hd)
    kc = np.zeros(nblocks * kstride, np.uint8)
    vc = np.zeros(nblocks * vstride, np.uint8)
    for s, n in enumerate(lens):
        nb = -(-n // bs)
        tables[s, :nb] = perm[cur:cur + nb]
        cur += nb
        k = rng.standard_normal((n, nkv, hd)).astype(np.float32)
        v = rng.standard_normal((n, nkv, hd)).astype(np.float32)
        pos = np.arange(n)
        slots = tables[s, pos // bs] * bs + pos % bs
        cache_write(kside, k, kc, slots, nkv, hd, bs, kstride, scale=k_scale)
        cache_write(vside, v, vc, slots, nkv, hd, bs, vstride, scale=v_scale)
    q = rng.standard_normal((len(lens), nq, hd))
    return dict(q=q, k_cache=kc, v_cache=vc, block_tables=tables,
                seq_lens=np.array(lens), nkv=nkv, hd=hd, block_size=bs,
                k_block_stride=kstride, v_block_stride=vstride, fmt=fmt,
                k_scale=k_scale, v_scale=v_scale)


def naive(q, k, v, scale):
    """Plain loops: softmax(q.k * scale) . v for one head."""
    n = len(k)
    s = [scale * sum(float(q[d]) * float(k[t][d]) for d in range(len(q))) for t in range(n)]
    m = max(s)
    w = [math.exp(x - m) for x in s]
    z = sum(w)
    return [sum(w[t] * float(v[t][d]) for t in range(n)) / z for d in range(len(q))]


def test_bf16_equals_naive_loop():
    a = build("bf16", [5, 23])
    out = paged_decode(**a)
    for s, n in enumerate(a["seq_lens"]):
        pos = np.arange(n)
        blocks = a["block_tables"][s, pos // 16]
        k = gather_side(a["k_cache"], "bf16", blocks, pos % 16, 2, 64, 16, a["k_block_stride"])
        v = gather_side(a["v_cache"], "bf16", blocks, pos % 16, 2, 64, 16, a["v_block_stride"])
        for j in range(4):
            ref = naive(a["q"][s, j], k[:, j // 2], v[:, j // 2], 1 / 8)
            np.testing.assert_allclose(out[s, j], ref, atol=1e-12, rtol=0)


@pytest.mark.parametrize("fmt", ["bf16", "turbo4", "fp8k_turbo2v", "turbo8"])
def test_special_cases(fmt):
    a = build(fmt, [1, 40, 0])
    out = paged_decode(**a)
    kside, vside = F.kv_pair(fmt)
    b0 = a["block_tables"][0, 0]
    v0 = gather_side(a["v_cache"], vside, [b0], [0], 2, 64, 16, a["v_block_stride"], 0.05)
    for j in range(4):
        np.testing.assert_allclose(out[0, j], v0[0, j // 2], atol=1e-12)
    assert not out[2].any()
    a0 = dict(a, q=np.zeros_like(a["q"]))
    out0 = paged_decode(**a0)
    pos = np.arange(40)
    blocks = a["block_tables"][1, pos // 16]
    v = gather_side(a["v_cache"], vside, blocks, pos % 16, 2, 64, 16, a["v_block_stride"], 0.05)
    for j in range(4):
        np.testing.assert_allclose(out0[1, j], v[:, j // 2].mean(axis=0), atol=1e-12)
    out_w1 = paged_decode(**a, window=1)
    for j in range(4):
        np.testing.assert_allclose(out_w1[1, j], v[39, j // 2], atol=1e-12)


def test_window_equals_truncated_sequence():
    a = build("turbo4k_turbo3v", [45, 33])
    w = paged_decode(**a, window=20)
    # same as attending over only the last 20 positions: drop the others by
    # re-running with a table shifted so the window is the whole sequence
    for s, n in enumerate(a["seq_lens"]):
        pos = np.arange(n - 20, n)
        blocks = a["block_tables"][s, pos // 16]
        k = gather_side(a["k_cache"], "turbo4", blocks, pos % 16, 2, 64, 16, a["k_block_stride"])
        v = gather_side(a["v_cache"], "turbo3", blocks, pos % 16, 2, 64, 16, a["v_block_stride"])
        for j in range(4):
            ref = naive(a["q"][s, j], k[:, j // 2], v[:, j // 2], 1 / 8)
            np.testing.assert_allclose(w[s, j], ref, atol=1e-12)


@pytest.mark.parametrize("fmt", ["turbo4", "turbo4k_turbo3v", "turbo2", "turbo8"])
def test_rotated_basis_identity(fmt):
    a = build(fmt, [30, 50], nq=8, nkv=2)
    out = paged_decode(**a)
    kside, vside = F.kv_pair(fmt)
    for s, n in enumerate(a["seq_lens"]):
        pos = np.arange(n)
        blocks = a["block_tables"][s, pos // 16]
        kr = gather_side(a["k_cache"], kside, blocks, pos % 16, 2, 64, 16,
                         a["k_block_stride"], to_original_basis=False)
        vr = gather_side(a["v_cache"], vside, blocks, pos % 16, 2, 64, 16,
                         a["v_block_stride"], to_original_basis=False)
        for j in range(8):
            qr = wht_f64(a["q"][s, j])
            sc = (kr[:, j // 4] @ qr) / 8
            p = np.exp(sc - sc.max())
            p /= p.sum()
            o = wht_f64(p @ vr[:, j // 4])
            np.testing.assert_allclose(out[s, j], o, atol=1e-12)


def test_sparse_v_drops_small_weights_only():
    a = build("bf16k_turbo4v", [64])
    dense = paged_decode(**a)
    sparse = paged_decode(**a, sparse_v_threshold=1e-3)
    huge = paged_decode(**a, sparse_v_threshold=1.0)
    assert np.max(np.abs(dense - sparse)) < 0.05
    assert not huge.any()


def test_attend_on_given_rows():
    """attend() on K/V rows equals the naive loop, and the paged decode of a
    BF16 cache that holds the same (bf16-exact) rows, window included."""
    from oracle.decode import attend
    from oracle.numformats import bf16_decode, bf16_encode
    rng = np.random.default_rng(5)
    n, nq, nkv, hd, bs = 37, 6, 3, 64, 16
    k = bf16_decode(bf16_encode(rng.standard_normal((n, nkv, hd)).astype(np.float32)))
    v = bf16_decode(bf16_encode(rng.standard_normal((n, nkv, hd)).astype(np.float32)))
    q = rng.standard_normal((nq, hd))
    got = attend(q, k, v)
    for j in range(nq):
        ref = naive(q[j], k[:, j // 2], v[:, j // 2], 1 / 8)
        np.testing.assert_allclose(got[j], ref, atol=1e-12, rtol=0)
    nb = -(-n // bs)
    stride = F.block_bytes("bf16", bs, nkv, hd)
    kc = np.zeros(nb * stride, np.uint8)
    vc = np.zeros(nb * stride, np.uint8)
    slots = np.arange(n)
    cache_write("bf16", k.astype(np.float32), kc, slots, nkv, hd, bs, stride)
    cache_write("bf16", v.astype(np.float32), vc, slots, nkv, hd, bs, stride)
    tables = np.arange(nb)[None, :]
    for window in (0, 5):
        pd = paged_decode(q[None], kc, vc, tables, np.array([n]), nkv, hd, bs, stride, stride,
                          "bf16", window=window)
        lo = n - window if window else 0
        np.testing.assert_array_equal(pd[0], attend(q, k[lo:], v[lo:]))
    assert not attend(q, k[:0], v[:0]).any()
