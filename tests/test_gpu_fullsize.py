"""Full-size parity at the benchmark workloads, sampled.

Each case fills the whole paged cache with one cache-write launch and runs
one decode launch over the whole batch, at the workload's full size (the
same calls bench.py times).  The sampled sequences' K/V are drawn on the
host (seeded, exact oracle inputs); every other sequence is drawn on the
device with the same distribution.  Checked against the oracle:
  * the cache bytes of every block of the sampled sequences (bit-exact);
  * the decode output of the sampled sequences (all their query heads),
    with the oracle reading the oracle-written bytes (max-abs 2e-3,
    mean-abs 2e-4).
Workloads: llama8b (32 x 4096, bf16 / fp8 / turbo4), ragged (64 x
U[512, 16384], bf16k_turbo3v / fp8k_turbo2v), longctx (4 x 131072, 64q/8kv,
turbo4k_turbo3v, window 0 and 4096), gemma_write (8192-token scattered write
from a fused QKV row, every written byte compared; decode 16 x 8192 turbo2 /
turbo8)."""
import numpy as np
import pytest
import torch

import oracle
from kvq_cases import assert_decode_close, bf16_round
from quantized_paged_kv_reshape_gb300 import ops
from quantized_paged_kv_reshape_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _fill(w, fmt, sampled, dev=DEV):
    """Write the whole cache; returns pools, host rows of sampled seqs, scales."""
    nkv, hd, bs = w.num_kv_heads, w.head_dim, w.block_size
    tables = W.block_tables(w)
    lens = [int(x) for x in w.seq_lens]
    starts = np.concatenate([[0], np.cumsum(lens)])
    total = int(starts[-1])
    g = torch.Generator(device=dev)
    g.manual_seed(77)
    tdt = torch.bfloat16 if w.in_dtype == "bf16" else torch.float32
    rnd = bf16_round if w.in_dtype == "bf16" else (lambda a: a)
    rows = {}
    kv = []
    for side in (0, 1):
        ch = torch.from_numpy(W.channel_scales(w, side)).to(dev)
        x = (torch.randn((total, nkv, hd), generator=g, device=dev) * ch).to(tdt)
        for s in sampled:
            hrow = rnd(W.kv_rows(w, side, lens[s], seed_offset=s))
            rows[(s, side)] = hrow
            x[starts[s]:starts[s + 1]] = torch.from_numpy(hrow).to(dev).to(tdt)
        kv.append(x)
    k_scale = float(kv[0].float().abs().amax()) / 448.0
    v_scale = float(kv[1].float().abs().amax()) / 448.0
    kpool = ops.alloc_pool(w.num_blocks, fmt, 0, bs, nkv, hd, device=dev)
    vpool = ops.alloc_pool(w.num_blocks, fmt, 1, bs, nkv, hd, device=dev)
    slots = torch.from_numpy(W.slot_mapping_for_sequences(w, tables)).to(dev)
    ops.cache_write(kv[0].view(total, -1), kv[1].view(total, -1), kpool, vpool, slots, fmt, nkv,
                    hd, bs, k_scale=k_scale, v_scale=v_scale)
    torch.cuda.synchronize()
    return dict(tables=tables, lens=lens, kpool=kpool, vpool=vpool, rows=rows,
                k_scale=k_scale, v_scale=v_scale)


def _check(w, fmt, sampled, windows=(0,)):
    st = _fill(w, fmt, sampled)
    nkv, hd, bs, nq = w.num_kv_heads, w.head_dim, w.block_size, w.num_q_heads
    kside, vside = oracle.kv_pair(fmt)
    kst, vst = st["kpool"].stride(0), st["vpool"].stride(0)
    # oracle images of the sampled sequences' blocks
    kc = np.zeros(w.num_blocks * kst, np.uint8)
    vc = np.zeros(w.num_blocks * vst, np.uint8)
    kg = st["kpool"].cpu().numpy().reshape(-1)
    vg = st["vpool"].cpu().numpy().reshape(-1)
    for s in sampled:
        n = st["lens"][s]
        pos = np.arange(n)
        slots = st["tables"][s, pos // bs].astype(np.int64) * bs + pos % bs
        oracle.cache_write(kside, st["rows"][(s, 0)], kc, slots, nkv, hd, bs, kst, scale=st["k_scale"])
        oracle.cache_write(vside, st["rows"][(s, 1)], vc, slots, nkv, hd, bs, vst, scale=st["v_scale"])
        for b in st["tables"][s, : -(-n // bs)]:
            assert np.array_equal(kc[b * kst:(b + 1) * kst], kg[b * kst:(b + 1) * kst]), f"K block {b}"
            assert np.array_equal(vc[b * vst:(b + 1) * vst], vg[b * vst:(b + 1) * vst]), f"V block {b}"
    if w.in_dtype == "bf16":
        q = bf16_round(W.q_rows(w))
        qd = torch.from_numpy(q).to(DEV).to(torch.bfloat16)
    else:
        q = W.q_rows(w)
        qd = torch.from_numpy(q).to(DEV)
    tab_d = torch.from_numpy(st["tables"]).to(DEV)
    lens_d = torch.from_numpy(np.asarray(st["lens"], np.int32)).to(DEV)
    for win in windows:
        out = ops.paged_decode(qd, st["kpool"], st["vpool"], tab_d, lens_d, fmt, nkv, bs,
                               k_scale=st["k_scale"], v_scale=st["v_scale"], sliding_window=win)
        torch.cuda.synchronize()
        got = out.cpu().numpy().astype(np.float64)
        for s in sampled:
            sub_tab = st["tables"][s:s + 1]
            ref = oracle.paged_decode(q[s:s + 1], kc, vc, sub_tab, [st["lens"][s]], nkv, hd, bs,
                                      kst, vst, fmt, k_scale=st["k_scale"],
                                      v_scale=st["v_scale"], window=win)
            assert_decode_close(got[s:s + 1], ref)


@pytest.mark.parametrize("fmt", ["bf16", "fp8", "turbo4"])
def test_llama8b_full(fmt):
    _check(W.make("llama8b"), fmt, sampled=[0, 21])


@pytest.mark.parametrize("fmt", ["bf16k_turbo3v", "fp8k_turbo2v"])
def test_ragged_full(fmt):
    w = W.make("ragged")
    order = np.argsort(w.seq_lens)
    _check(w, fmt, sampled=[int(order[0]), int(order[-1])])   # shortest and longest


def test_longctx_full():
    _check(W.make("longctx"), "turbo4k_turbo3v", sampled=[2], windows=(4096, 0))


def test_tiny_full():
    w = W.make("tiny")
    _check(w, "bf16k_turbo4v", sampled=[0, 1])


@pytest.mark.parametrize("fmt", ["turbo2", "turbo8"])
def test_gemma_write_and_decode_full(fmt):
    w = W.make("gemma_write")
    nq, nkv, hd, bs = w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size
    # 8192-token write from a fused QKV row (stride 16384 elements), slots
    # scattered over the whole pool: every written byte is compared.
    fused = bf16_round(W.fused_qkv(w.write_tokens, w.write_row_elems, nq, nkv, hd))
    slots = W.scattered_slots(w.write_tokens, w.num_blocks, bs)
    kside, vside = oracle.kv_pair(fmt)
    kpool = ops.alloc_pool(w.num_blocks, fmt, 0, bs, nkv, hd, device=DEV)
    vpool = ops.alloc_pool(w.num_blocks, fmt, 1, bs, nkv, hd, device=DEV)
    fd = torch.from_numpy(fused).to(DEV).to(torch.bfloat16)
    ops.cache_write(fd[:, nq * hd:], fd[:, (nq + nkv) * hd:], kpool, vpool,
                    torch.from_numpy(slots).to(DEV), fmt, nkv, hd, bs,
                    key_stride=w.write_row_elems, value_stride=w.write_row_elems)
    torch.cuda.synchronize()
    kc = np.zeros(kpool.numel(), np.uint8)
    vc = np.zeros(vpool.numel(), np.uint8)
    flat = fused.reshape(-1)
    oracle.cache_write(kside, flat[nq * hd:], kc, slots, nkv, hd, bs, kpool.stride(0),
                       row_stride=w.write_row_elems)
    oracle.cache_write(vside, flat[(nq + nkv) * hd:], vc, slots, nkv, hd, bs, vpool.stride(0),
                       row_stride=w.write_row_elems)
    assert np.array_equal(kc, kpool.cpu().numpy().reshape(-1))
    assert np.array_equal(vc, vpool.cpu().numpy().reshape(-1))
    # decode over 16 x 8192 with 32 query heads
    _check(w, fmt, sampled=[5])


@pytest.mark.parametrize("name,fmt", [("prefill", "bf16"), ("prefill", "fp8"), ("prefill", "turbo4"),
                                      ("prefill_hd256", "bf16"), ("prefill_hd256", "turbo2"),
                                      ("prefill_hd256", "turbo8")])
def test_prefill_full(name, fmt):
    """The chunked-prefill workloads at full size (8 x 4096 positions, the
    last 512 of every sequence the chunk, the launches bench.py times; head_dim
    128 and the Gemma-shaped head_dim 256): queries of two sampled sequences
    against the oracle, the first 8 and the last 8 of each chunk (the first
    ones through the oracle's causal reading of a shorter sequence)."""
    w = W.make(name)
    nq, nkv, hd, bs, C = w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, w.chunk
    sampled = [0, 5]
    st = _fill(w, fmt, sampled)
    kside, vside = oracle.kv_pair(fmt)
    kst, vst = st["kpool"].stride(0), st["vpool"].stride(0)
    kc = np.zeros(w.num_blocks * kst, np.uint8)
    vc = np.zeros(w.num_blocks * vst, np.uint8)
    for s in sampled:
        n = st["lens"][s]
        pos = np.arange(n)
        slots = st["tables"][s, pos // bs].astype(np.int64) * bs + pos % bs
        oracle.cache_write(kside, st["rows"][(s, 0)], kc, slots, nkv, hd, bs, kst, scale=st["k_scale"])
        oracle.cache_write(vside, st["rows"][(s, 1)], vc, slots, nkv, hd, bs, vst, scale=st["v_scale"])
    ns = len(st["lens"])
    rng = np.random.default_rng(123)
    q = bf16_round(rng.standard_normal((ns * C, nq, hd)).astype(np.float32))
    cu = (np.arange(ns + 1) * C).astype(np.int32)
    out = ops.paged_prefill(torch.from_numpy(q).to(DEV).to(torch.bfloat16), torch.from_numpy(cu).to(DEV), C,
                            st["kpool"], st["vpool"], torch.from_numpy(st["tables"]).to(DEV),
                            torch.from_numpy(np.asarray(st["lens"], np.int32)).to(DEV), fmt, nkv, bs,
                            k_scale=st["k_scale"], v_scale=st["v_scale"])
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    k = 8
    for s in sampled:
        L = st["lens"][s]
        tab = st["tables"][s:s + 1]
        for first, Ls in ((C - k, L), (0, L - C + k)):   # last k queries, first k queries
            qs = q[s * C + first:s * C + first + k]
            ref = oracle.paged_prefill(qs, np.array([0, k]), kc, vc, tab, [Ls], nkv, hd, bs, kst, vst,
                                       fmt, k_scale=st["k_scale"], v_scale=st["v_scale"])
            assert_decode_close(got[s * C + first:s * C + first + k], ref)
