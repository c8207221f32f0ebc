"""GPU chunked prefill vs the oracle on identical cache bytes (the oracle
writes the cache; the same bytes are uploaded): max-abs <= 2e-3, mean-abs
<= 2e-4, the decode's bound.

Every catalogue format; head_dim 64/128/256; GQA ratios 1, 2, 3, 4, 8;
ragged chunks (a whole sequence, a single query, an empty chunk, a chunk
longer than its sequence whose first queries attend nothing, chunks spanning
several 64-row tiles); windows; block sizes 8/16/32; bf16 q and output;
head_dim 256 (64-row tiles, 32-position steps) at GQA 1, 4 and 8."""
import numpy as np
import pytest
import torch

import oracle
from kvq_cases import ALL_FORMATS, assert_decode_close, decode_case
from quantized_paged_kv_reshape_gb300 import ops

pytestmark = pytest.mark.gpu

LENS = [37, 50, 1, 300, 129, 16, 3]
CHUNKS = [5, 50, 1, 64, 129, 0, 5]


def _prefill_case(fmt, lens, chunks, nq, nkv, hd, bs=16, seed=0):
    c = decode_case(fmt, lens, nq, nkv, hd, bs=bs, seed=seed)
    rng = np.random.default_rng(seed + 99)
    cu = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    q = rng.standard_normal((int(cu[-1]), nq, hd)).astype(np.float32)
    c.update(cu=cu, qp=q, chunks=list(chunks))
    return c


def _oracle(c, window=0, q=None):
    return oracle.paged_prefill(c["qp"] if q is None else q, c["cu"], c["kc"], c["vc"], c["tables"],
                                c["lens"], c["nkv"], c["hd"], c["bs"], c["kst"], c["vst"],
                                c["fmt"], k_scale=c["k_scale"], v_scale=c["v_scale"],
                                window=window)


def _gpu(c, window=0, q_dtype=torch.float32, out_dtype=torch.float32):
    dev = "cuda"
    kpool = torch.from_numpy(c["kc"].reshape(c["num_blocks"], c["kst"])).to(dev)
    vpool = torch.from_numpy(c["vc"].reshape(c["num_blocks"], c["vst"])).to(dev)
    q = torch.from_numpy(c["qp"]).to(dev).to(q_dtype)
    out = ops.paged_prefill(q, torch.from_numpy(c["cu"]).to(dev), max(c["chunks"]), kpool, vpool,
                            torch.from_numpy(c["tables"]).to(dev),
                            torch.from_numpy(c["lens"]).to(dev), c["fmt"], c["nkv"], c["bs"],
                            out_dtype=out_dtype, k_scale=c["k_scale"], v_scale=c["v_scale"],
                            sliding_window=window)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("fmt", ALL_FORMATS)
@pytest.mark.parametrize("hd,nq,nkv", [(64, 4, 2), (128, 8, 2), (256, 4, 2), (128, 16, 2)])
def test_prefill_parity(fmt, hd, nq, nkv):
    c = _prefill_case(fmt, LENS, CHUNKS, nq, nkv, hd, seed=hd + nq)
    got = _gpu(c)
    ref = _oracle(c)
    assert_decode_close(got, ref)
    # queries of the 5-query chunk over a 3-token sequence at p < 0 are zero
    s = len(LENS) - 1
    assert not got[c["cu"][s]:c["cu"][s] + 2].any()


@pytest.mark.parametrize("nq,nkv", [(2, 2), (6, 2), (8, 8)])
def test_prefill_gqa_ratios(nq, nkv):
    c = _prefill_case("turbo4", [120, 33], [70, 33], nq, nkv, 128, seed=nq)
    assert_decode_close(_gpu(c), _oracle(c))


@pytest.mark.parametrize("fmt", ["bf16", "turbo4k_turbo3v", "fp8k_turbo2v", "turbo8"])
@pytest.mark.parametrize("window", [1, 17, 100])
def test_prefill_window(fmt, window):
    c = _prefill_case(fmt, LENS, CHUNKS, 8, 2, 128, seed=window)
    assert_decode_close(_gpu(c, window=window), _oracle(c, window=window))


@pytest.mark.parametrize("fmt", ["bf16", "turbo2", "turbo8", "turbo4k_turbo3v", "fp8k_turbo2v"])
@pytest.mark.parametrize("nq,nkv,window", [(2, 2, 0), (16, 2, 0), (8, 4, 33)])
def test_prefill_hd256(fmt, nq, nkv, window):
    """head_dim 256 runs 64-row tiles with 32-position steps: GQA 1 (64
    queries per tile), GQA 8 (8 per tile), a window cutting steps."""
    c = _prefill_case(fmt, [300, 77, 40], [200, 77, 9], nq, nkv, 256, seed=nq + window)
    assert_decode_close(_gpu(c, window=window), _oracle(c, window=window))


@pytest.mark.parametrize("bs", [8, 32])
def test_prefill_block_sizes(bs):
    c = _prefill_case("bf16k_turbo4v", [70, 9, 257], [70, 9, 100], 8, 2, 128, bs=bs, seed=bs)
    assert_decode_close(_gpu(c), _oracle(c))


def test_prefill_bf16_io():
    c = _prefill_case("turbo4", [90, 40], [90, 20], 8, 2, 128, seed=7)
    qb = torch.from_numpy(c["qp"]).to(torch.bfloat16).float().numpy()
    got = _gpu(c, q_dtype=torch.bfloat16, out_dtype=torch.bfloat16)
    ref = _oracle(c, q=qb)
    # bf16 output rounding (half an ulp, ~2e-3 relative) on top of the bound
    err = np.abs(got - ref)
    assert err.max() <= 2e-3 + 4e-3 * np.abs(ref).max()
    assert err.mean() <= 2e-3


def test_prefill_chunk_of_one_is_decode():
    """One query per sequence at the newest position: the decode's result."""
    c = _prefill_case("turbo4", LENS[:5], [1] * 5, 8, 2, 128, seed=3)
    dev = "cuda"
    kpool = torch.from_numpy(c["kc"].reshape(c["num_blocks"], c["kst"])).to(dev)
    vpool = torch.from_numpy(c["vc"].reshape(c["num_blocks"], c["vst"])).to(dev)
    dec = ops.paged_decode(torch.from_numpy(c["qp"]).to(dev), kpool, vpool,
                           torch.from_numpy(c["tables"]).to(dev),
                           torch.from_numpy(c["lens"][:5]).to(dev), "turbo4", 2, 16)
    torch.cuda.synchronize()
    got = _gpu(c)
    assert np.abs(got - dec.cpu().numpy()).max() <= 2e-3


def test_prefill_graph_replay():
    """The prefill captures into a CUDA graph: after the query buffer is
    refilled, each replay matches the oracle for the new queries."""
    c = _prefill_case("turbo4", [300, 77], [64, 20], 8, 2, 128, seed=41)
    dev = "cuda"
    kpool = torch.from_numpy(c["kc"].reshape(c["num_blocks"], c["kst"])).to(dev)
    vpool = torch.from_numpy(c["vc"].reshape(c["num_blocks"], c["vst"])).to(dev)
    q = torch.from_numpy(c["qp"]).to(dev)
    cu = torch.from_numpy(c["cu"]).to(dev)
    tables = torch.from_numpy(c["tables"]).to(dev)
    lens = torch.from_numpy(c["lens"]).to(dev)
    out = torch.empty_like(q)

    def call():
        ops.paged_prefill(q, cu, max(c["chunks"]), kpool, vpool, tables, lens, c["fmt"], c["nkv"],
                          c["bs"], out=out, k_scale=c["k_scale"], v_scale=c["v_scale"])

    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    torch.cuda.synchronize()
    rng = np.random.default_rng(43)
    for qn in (rng.standard_normal(c["qp"].shape).astype(np.float32), c["qp"]):
        q.copy_(torch.from_numpy(qn))
        g.replay()
        torch.cuda.synchronize()
        assert_decode_close(out.cpu().numpy().astype(np.float64), _oracle(c, q=qn))
