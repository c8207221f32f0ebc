"""The seeded synthetic workloads (CPU): each has the shapes, formats and
value structure its configuration states, block tables hand out every
physical block at most once, slot mappings address the right page and
offset, and every draw is reproducible from its seed."""
import numpy as np
import pytest

from quantized_paged_kv_reshape_gb300 import workloads as W

SHAPES = {  # name: (num_seqs, nq, nkv, hd, block_size, formats)
    "tiny": (2, 4, 2, 64, 16, ("bf16k_turbo4v",)),
    "llama8b": (32, 32, 8, 128, 16, ("bf16", "fp8", "turbo4")),
    "ragged": (64, 32, 8, 128, 16, ("bf16k_turbo3v", "fp8k_turbo2v")),
    "longctx": (4, 64, 8, 128, 16, ("turbo4k_turbo3v",)),
    "gemma_write": (16, 32, 16, 256, 16, ("turbo2", "turbo8")),
    "prefill": (8, 32, 8, 128, 16, ("bf16", "fp8", "turbo4")),
    "prefill_hd256": (8, 32, 16, 256, 16, ("bf16", "turbo2", "turbo8")),
}


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_shapes_and_formats(name):
    w = W.make(name)
    ns, nq, nkv, hd, bs, fmts = SHAPES[name]
    assert (w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size) == \
        (ns, nq, nkv, hd, bs)
    assert tuple(w.formats) == fmts
    assert len(w.seq_lens) == ns and w.seq_lens.dtype == np.int32


def test_lengths_and_windows():
    assert list(W.make("tiny").seq_lens) == [37, 50]
    assert set(W.make("llama8b").seq_lens) == {4096}
    r = W.make("ragged").seq_lens
    assert r.min() >= 512 and r.max() <= 16384 and len(set(r)) > 32
    lc = W.make("longctx")
    assert set(lc.seq_lens) == {131072} and tuple(lc.windows) == (0, 4096)
    g = W.make("gemma_write")
    assert set(g.seq_lens) == {8192} and g.write_tokens == 8192
    assert g.write_row_elems == (32 + 16 + 16) * 256
    assert W.make("prefill").chunk == 512 and W.make("prefill_hd256").chunk == 512


@pytest.mark.parametrize("name", ["tiny", "llama8b", "ragged"])
def test_block_tables_are_disjoint_permutation_slices(name):
    w = W.make(name, seed=3)
    tab = W.block_tables(w)
    used = tab[tab >= 0]
    assert len(np.unique(used)) == len(used) == w.blocks_needed
    assert used.max() < w.num_blocks
    for s, n in enumerate(w.seq_lens):
        nb = -(-int(n) // w.block_size)
        assert (tab[s, :nb] >= 0).all() and (tab[s, nb:] == -1).all()
    assert np.array_equal(tab, W.block_tables(W.make(name, seed=3)))
    assert not np.array_equal(tab, W.block_tables(W.make(name, seed=4)))


def test_slot_mapping_addresses_page_and_offset():
    w = W.make("tiny", seed=1)
    tab = W.block_tables(w)
    slots = W.slot_mapping_for_sequences(w, tab)
    assert len(slots) == int(w.seq_lens.sum()) and len(np.unique(slots)) == len(slots)
    start = 0
    for s, n in enumerate(w.seq_lens):
        for p in (0, 15, 16, int(n) - 1):
            sl = slots[start + p]
            assert sl // w.block_size == tab[s, p // w.block_size]
            assert sl % w.block_size == p % w.block_size
        start += int(n)


def test_channel_scales_structure():
    w = W.make("llama8b")
    sc = W.channel_scales(w, 0).astype(np.float64)
    assert sc.shape == (8, 128)
    # 1% of the 1024 channels (10) carry the x10 outlier factor on top of a
    # lognormal(0, 0.5) scale
    base = W.channel_scales(W.make("llama8b", outlier_frac=0.0), 0).astype(np.float64)
    ratio = sc / base
    assert np.sum(np.isclose(ratio, 10.0)) == 10
    assert np.sum(np.isclose(ratio, 1.0)) == 1024 - 10
    logs = np.log(base).ravel()
    assert abs(logs.mean()) < 0.1 and abs(logs.std() - 0.5) < 0.05
    # tiny: two outlier channels per head, x8, unit scale elsewhere
    t = W.channel_scales(W.make("tiny"), 1)
    assert (np.sum(np.isclose(t, 8.0), axis=1) == 2).all()
    assert (np.sum(np.isclose(t, 1.0), axis=1) == 62).all()
    # gemma_write: plain N(0,1), no channel structure
    assert np.all(W.channel_scales(W.make("gemma_write"), 0) == 1.0)


def test_draws_are_seeded():
    w = W.make("tiny", seed=5)
    a = W.kv_rows(w, 0, 37, seed_offset=1)
    assert np.array_equal(a, W.kv_rows(W.make("tiny", seed=5), 0, 37, seed_offset=1))
    assert not np.array_equal(a, W.kv_rows(w, 1, 37, seed_offset=1))
    assert not np.array_equal(a, W.kv_rows(w, 0, 37, seed_offset=2))
    assert np.array_equal(W.q_rows(w), W.q_rows(W.make("tiny", seed=5)))
    s = W.scattered_slots(100, 20, 16, seed=2)
    assert len(np.unique(s)) == 100 and s.max() < 20 * 16
