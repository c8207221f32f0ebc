"""Seeded synthetic inputs for the five cache workloads.

This module only draws numbers and lays out shapes, block tables and slot
mappings; it contains none of the cache formats' arithmetic.  It is the one
module both the CUDA path's tests/bench and the CPU oracle's tests draw from.

Workloads (sizes follow the quantized-KV-cache pages' use cases):

* ``tiny``: 2 sequences of 37 and 50 tokens, 4 query / 2 KV heads, head_dim
  64, block_size 16, 12 physical blocks handed out by a seeded permutation;
  Q, K, V fp32 N(0,1) with 2 outlier channels per head scaled x8; format
  bf16k_turbo4v.
* ``llama8b``: 32 sequences x 4096 context, 32 query / 8 KV heads, head_dim
  128, block_size 16; K, V bf16 N(0,1) * sigma_c with sigma_c ~
  lognormal(0, 0.5) per channel (channel = (kv head, dim), fixed over
  tokens) and 1% of the channels scaled x10; Q bf16 N(0,1); formats bf16,
  fp8 (per-tensor scale), turbo4.
* ``ragged``: 64 sequences with lengths uniform on [512, 16384], otherwise
  as ``llama8b``; formats bf16k_turbo3v, fp8k_turbo2v.
* ``longctx``: 4 sequences x 131072, 64 query / 8 KV heads, head_dim 128;
  K, V bf16 N(0,1) with 1% channels x10; sliding window 0 or 4096; format
  turbo4k_turbo3v.
* ``gemma_write``: cache write of 8192 tokens, 16 KV heads, head_dim 256,
  K and V read from a fused QKV row of (32+16+16)*256 elements (so the
  per-token stride is 16384 elements, not the 4096-element row), slots from
  a seeded random permutation of the pool; then decode over 16 sequences x
  8192 with 32 query heads; K, V, Q N(0,1) bf16; formats turbo2 and turbo8.

* ``prefill``: chunked prefill, Llama-3-8B-shaped: 8 sequences x 4096
  positions whose last 512 are the new chunk (written, then attended
  causally), 32 query / 8 KV heads, head_dim 128, llama8b's value
  distribution; formats bf16, fp8, turbo4.
* ``prefill_hd256``: the same chunked prefill, Gemma-shaped: 32 query / 16 KV
  heads, head_dim 256, K and V N(0,1) bf16 as gemma_write; formats bf16,
  turbo2, turbo8.

Block tables are seeded permutations of the physical block ids, sliced per
sequence, so no two sequences share a block.
"""

from dataclasses import dataclass, field

import numpy as np


@dataclass
class Workload:
    name: str
    num_seqs: int
    seq_lens: np.ndarray          # int32 [num_seqs]
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    formats: tuple
    in_dtype: str                 # "f32" or "bf16": dtype of Q/K/V activations
    windows: tuple = (0,)
    outlier_mult: float = 10.0
    outlier_frac: float = 0.01
    outliers_per_head: int = 0    # if > 0, a fixed count per head instead of a fraction
    lognormal_sigma: float = 0.0  # 0 => unit channel scale
    extra_blocks: int = 0         # spare physical blocks beyond what the seqs need
    write_tokens: int = 0         # tokens written by the write step (gemma_write)
    write_row_elems: int = 0      # elements in one fused QKV row (key/value stride)
    chunk: int = 0                # chunked prefill: new query tokens per sequence
    seed: int = 0
    notes: dict = field(default_factory=dict)

    @property
    def max_blocks_per_seq(self):
        return int(-(-int(self.seq_lens.max()) // self.block_size)) if self.num_seqs else 0

    @property
    def blocks_needed(self):
        return int(sum(-(-int(n) // self.block_size) for n in self.seq_lens))

    @property
    def num_blocks(self):
        return self.blocks_needed + self.extra_blocks


def make(name, seed=0, **over):
    """Workload spec by name; keyword overrides shrink or vary it."""
    rng = np.random.default_rng(seed)
    if name == "tiny":
        w = Workload("tiny", 2, np.array([37, 50], np.int32), 4, 2, 64, 16,
                     ("bf16k_turbo4v",), "f32", outlier_mult=8.0,
                     outliers_per_head=2, extra_blocks=12 - 7)
    elif name == "llama8b":
        w = Workload("llama8b", 32, np.full(32, 4096, np.int32), 32, 8, 128, 16,
                     ("bf16", "fp8", "turbo4"), "bf16", lognormal_sigma=0.5)
    elif name == "ragged":
        lens = rng.integers(512, 16384, size=64, endpoint=True).astype(np.int32)
        w = Workload("ragged", 64, lens, 32, 8, 128, 16,
                     ("bf16k_turbo3v", "fp8k_turbo2v"), "bf16", lognormal_sigma=0.5)
    elif name == "longctx":
        w = Workload("longctx", 4, np.full(4, 131072, np.int32), 64, 8, 128, 16,
                     ("turbo4k_turbo3v",), "bf16", windows=(0, 4096))
    elif name == "gemma_write":
        w = Workload("gemma_write", 16, np.full(16, 8192, np.int32), 32, 16, 256, 16,
                     ("turbo2", "turbo8"), "bf16", outlier_frac=0.0,
                     write_tokens=8192, write_row_elems=(32 + 16 + 16) * 256)
    elif name == "prefill":
        w = Workload("prefill", 8, np.full(8, 4096, np.int32), 32, 8, 128, 16,
                     ("bf16", "fp8", "turbo4"), "bf16", lognormal_sigma=0.5, chunk=512)
    elif name == "prefill_hd256":
        w = Workload("prefill_hd256", 8, np.full(8, 4096, np.int32), 32, 16, 256, 16,
                     ("bf16", "turbo2", "turbo8"), "bf16", outlier_frac=0.0, chunk=512)
    else:
        raise KeyError(name)
    w.seed = seed
    for k, v in over.items():
        setattr(w, k, v)
    if "seq_lens" in over or "num_seqs" in over:
        w.seq_lens = np.asarray(w.seq_lens, np.int32)[: w.num_seqs]
    return w


def block_tables(w, seed=None):
    """int32 [num_seqs, max_blocks_per_seq] tables; unused entries are -1."""
    rng = np.random.default_rng((w.seed if seed is None else seed) + 1000)
    perm = rng.permutation(w.num_blocks).astype(np.int32)
    mb = max(w.max_blocks_per_seq, 1)
    tab = np.full((w.num_seqs, mb), -1, np.int32)
    cur = 0
    for s, n in enumerate(w.seq_lens):
        nb = -(-int(n) // w.block_size)
        tab[s, :nb] = perm[cur:cur + nb]
        cur += nb
    return tab


def channel_scales(w, side, seed=None):
    """fp32 [num_kv_heads, head_dim] per-channel multipliers for K (side 0) or V (1)."""
    rng = np.random.default_rng((w.seed if seed is None else seed) * 7 + 11 + side)
    nkv, hd = w.num_kv_heads, w.head_dim
    sc = np.ones((nkv, hd), np.float64)
    if w.lognormal_sigma > 0:
        sc *= rng.lognormal(0.0, w.lognormal_sigma, size=(nkv, hd))
    if w.outliers_per_head > 0:
        for h in range(nkv):
            idx = rng.choice(hd, size=w.outliers_per_head, replace=False)
            sc[h, idx] *= w.outlier_mult
    elif w.outlier_frac > 0:
        n_out = max(1, int(round(w.outlier_frac * nkv * hd)))
        idx = rng.choice(nkv * hd, size=n_out, replace=False)
        sc.reshape(-1)[idx] *= w.outlier_mult
    return sc.astype(np.float32)


def kv_rows(w, side, n_tokens, seed_offset=0, seed=None):
    """fp32 [n_tokens, nkv, hd] activations for K (side 0) or V (side 1).

    ``seed_offset`` selects an independent stream (e.g. one per sequence), so
    a sample of the workload can be drawn without drawing all of it.
    """
    base = w.seed if seed is None else seed
    rng = np.random.default_rng([base, side, seed_offset])
    x = rng.standard_normal((n_tokens, w.num_kv_heads, w.head_dim), dtype=np.float32)
    return x * channel_scales(w, side, seed)[None]


def q_rows(w, seed_offset=0, seed=None):
    """fp32 [num_seqs, nq, hd] queries, N(0,1)."""
    base = w.seed if seed is None else seed
    rng = np.random.default_rng([base, 7, seed_offset])
    q = rng.standard_normal((w.num_seqs, w.num_q_heads, w.head_dim), dtype=np.float32)
    if w.outliers_per_head > 0:  # the tiny workload scales Q's outlier channels too
        sc = channel_scales(w, 2, seed)
        rep = w.num_q_heads // w.num_kv_heads
        q = q * np.repeat(sc, rep, axis=0)[None]
    return q


def slot_mapping_for_sequences(w, tables):
    """int64 [sum(seq_lens)] slots of every position of every sequence, in order."""
    out = []
    for s, n in enumerate(w.seq_lens):
        pos = np.arange(int(n), dtype=np.int64)
        out.append(tables[s, pos // w.block_size].astype(np.int64) * w.block_size
                   + pos % w.block_size)
    return np.concatenate(out) if out else np.zeros(0, np.int64)


def scattered_slots(num_tokens, num_blocks, block_size, seed=0):
    """int64 [num_tokens] distinct slots drawn at random from the whole pool."""
    rng = np.random.default_rng(seed + 2000)
    return rng.permutation(num_blocks * block_size)[:num_tokens].astype(np.int64)


def fused_qkv(num_tokens, row_elems, nq, nkv, hd, seed=0):
    """fp32 [num_tokens, row_elems] fused QKV rows, N(0,1).

    K of token t, head h starts at element t*row_elems + nq*hd + h*hd and V
    at t*row_elems + (nq+nkv)*hd + h*hd.
    """
    rng = np.random.default_rng([seed, 9])
    assert row_elems >= (nq + 2 * nkv) * hd
    return rng.standard_normal((num_tokens, row_elems), dtype=np.float32)


# ------------------------------------------------------------ sharding over ranks
#
# Weak scaling over `world` GPUs: the job decodes a batch `world` times the
# workload's, and the sequences, which share nothing, are dealt out round
# robin (rank r owns global sequences r, r + world, ...).  Each rank holds the
# pages of its own sequences; no data crosses ranks.

def global_lengths(name, world=1, seed=0):
    """int32 lengths of the `world`-times batch of workload `name` (world 1:
    the workload's own batch)."""
    base = make(name, seed=seed)
    if world == 1:
        return base.seq_lens.copy()
    if name == "ragged":
        rng = np.random.default_rng([seed, world])
        return rng.integers(512, 16384, size=base.num_seqs * world,
                            endpoint=True).astype(np.int32)
    return np.tile(base.seq_lens, world).astype(np.int32)


def shard_sequences(num_seqs, world, rank):
    """Global indices of the sequences rank `rank` of `world` owns."""
    if not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    return np.arange(rank, num_seqs, world, dtype=np.int64)


def rank_workload(name, world=1, rank=0, seed=0):
    """The sub-workload of rank `rank`: its sequences of the `world`-times
    batch, with their lengths; ``notes['global_seqs']`` lists their global
    indices.  For world 1 this is the workload itself."""
    lens = global_lengths(name, world, seed)
    idx = shard_sequences(lens.size, world, rank)
    if world == 1:
        w = make(name, seed=seed)
    else:
        w = make(name, seed=seed, num_seqs=int(idx.size), seq_lens=lens[idx])
    w.notes["global_seqs"] = idx
    w.notes["world"] = world
    return w
