"""Pins of the chunked-prefill oracle (oracle/prefill.py).

* A chunk of one query per sequence is the decode of that sequence: the
  prefill oracle equals the already pinned decode oracle, every format.
* Causality: rewriting the cache rows after a query's position leaves that
  query's output unchanged (and changes the last query's).
* Window: a windowed query equals the decode of its sequence truncated at
  the query's position, with the same window.
* An independent scalar loop (positions one by one, running max and sum) on
  BF16-exact K/V gives the same output.
"""
import math

import numpy as np
import pytest

import oracle


def _case(fmt, lens, chunks, nq=4, nkv=2, hd=64, bs=16, seed=0):
    rng = np.random.default_rng(seed)
    nblk = [-(-n // bs) for n in lens]
    num_blocks = sum(nblk) + 2
    perm = rng.permutation(num_blocks).astype(np.int32)
    mb = max(nblk)
    tables = np.full((len(lens), mb), -1, np.int32)
    cur = 0
    for s, nb in enumerate(nblk):
        tables[s, :nb] = perm[cur:cur + nb]
        cur += nb
    kside, vside = oracle.kv_pair(fmt)
    kst = oracle.block_bytes(kside, bs, nkv, hd)
    vst = oracle.block_bytes(vside, bs, nkv, hd)
    kc = np.zeros(num_blocks * kst, np.uint8)
    vc = np.zeros(num_blocks * vst, np.uint8)
    total = sum(lens)
    k = rng.standard_normal((total, nkv, hd)).astype(np.float32)
    v = rng.standard_normal((total, nkv, hd)).astype(np.float32)
    slots = np.concatenate([tables[s, np.arange(n) // bs].astype(np.int64) * bs + np.arange(n) % bs
                            for s, n in enumerate(lens)])
    ks = float(np.abs(k).max()) / 448.0
    vs = float(np.abs(v).max()) / 448.0
    oracle.cache_write(kside, k, kc, slots, nkv, hd, bs, kst, scale=ks)
    oracle.cache_write(vside, v, vc, slots, nkv, hd, bs, vst, scale=vs)
    cu = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int64)
    q = rng.standard_normal((int(cu[-1]), nq, hd)).astype(np.float32)
    return dict(fmt=fmt, lens=lens, cu=cu, q=q, kc=kc, vc=vc, tables=tables, nkv=nkv, hd=hd,
                bs=bs, kst=kst, vst=vst, ks=ks, vs=vs, k=k, v=v)


def _prefill(c, window=0, kc=None):
    return oracle.paged_prefill(c["q"], c["cu"], c["kc"] if kc is None else kc, c["vc"],
                                c["tables"], c["lens"], c["nkv"], c["hd"], c["bs"], c["kst"],
                                c["vst"], c["fmt"], k_scale=c["ks"], v_scale=c["vs"],
                                window=window)


@pytest.mark.parametrize("hd", [64, 256])
@pytest.mark.parametrize("fmt", ["bf16", "fp8", "turbo4", "turbo4k_turbo3v", "nvfp4", "turbo8"])
def test_chunk_of_one_is_decode(fmt, hd):
    c = _case(fmt, [37, 50, 16], [1, 1, 1], hd=hd)
    got = _prefill(c)
    ref = oracle.paged_decode(c["q"], c["kc"], c["vc"], c["tables"], c["lens"], c["nkv"], c["hd"],
                              c["bs"], c["kst"], c["vst"], fmt, k_scale=c["ks"], v_scale=c["vs"])
    assert np.allclose(got, ref, rtol=0, atol=1e-12)


def test_causal_rows_after_a_query_do_not_matter():
    c = _case("turbo4", [40], [8], seed=3)
    base = _prefill(c)
    # rewrite the cache rows of positions 36..39 (the last 4 queries' own rows)
    kc2 = c["kc"].copy()
    bs, nkv, hd = c["bs"], c["nkv"], c["hd"]
    blk = c["tables"][0, 36 // bs]
    rng = np.random.default_rng(9)
    new = rng.standard_normal((4, nkv, hd)).astype(np.float32) * 3
    slots = np.array([blk * bs + (p % bs) for p in range(36, 40)], np.int64)
    oracle.cache_write("turbo4", new, kc2, slots, nkv, hd, bs, c["kst"])
    got = _prefill(c, kc=kc2)
    assert np.array_equal(got[:4], base[:4])          # queries at positions 32..35
    assert not np.allclose(got[7], base[7])           # the last query sees position 39


@pytest.mark.parametrize("window", [1, 5, 20])
def test_window_is_truncated_decode(window):
    c = _case("bf16k_turbo4v", [45], [12], seed=4)
    got = _prefill(c, window=window)
    for i in range(12):
        p = 45 - 12 + i
        ref = oracle.paged_decode(c["q"][i:i + 1], c["kc"], c["vc"], c["tables"], [p + 1],
                                  c["nkv"], c["hd"], c["bs"], c["kst"], c["vst"], c["fmt"],
                                  window=window)
        assert np.allclose(got[i], ref[0], rtol=0, atol=1e-12)


def test_scalar_loop_bf16():
    """Positions one at a time with a running max and sum (the online form of
    softmax), on BF16-exact values so the cache holds the inputs exactly."""
    c = _case("bf16", [21, 9], [5, 9], nq=4, nkv=2, hd=64, seed=5)
    k = oracle.bf16_decode(oracle.bf16_encode(c["k"])).astype(np.float64)
    v = oracle.bf16_decode(oracle.bf16_encode(c["v"])).astype(np.float64)
    got = _prefill(c)
    scale = 1.0 / math.sqrt(64)
    starts = np.concatenate([[0], np.cumsum(c["lens"])])
    for s, L in enumerate(c["lens"]):
        C = int(c["cu"][s + 1] - c["cu"][s])
        for i in range(C):
            p = L - C + i
            for j in range(4):
                h = j // 2
                m, den, acc = -math.inf, 0.0, np.zeros(64)
                for t in range(p + 1):
                    sc = float(np.dot(k[starts[s] + t, h], c["q"][c["cu"][s] + i, j])) * scale
                    m_new = max(m, sc)
                    f = math.exp(m - m_new) if m > -math.inf else 0.0
                    w = math.exp(sc - m_new)
                    den = den * f + w
                    acc = acc * f + w * v[starts[s] + t, h]
                    m = m_new
                assert np.allclose(got[c["cu"][s] + i, j], acc / den, rtol=0, atol=1e-12)
