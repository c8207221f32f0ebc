"""Chunked-prefill attention over the quantized paged cache (oracle side).

A chunk of C new query tokens per sequence attends, causally, to the paged
cache that already holds them ("combs_models/kv.rs", ``attend`` with its
causal mask for several query rows and ``repeat_kv``; the cache write of the
chunk comes first, as in the page's write-then-attend step).  Readings
(the pages only name chunked prefill over the quantized cache as the next
step): sequence s holds L = seq_lens[s] positions in the cache; its C =
cu_q[s+1] - cu_q[s] query rows are the last C positions, so query i sits at
position p = L - C + i and attends to positions [lo, p] with lo = max(0,
p + 1 - W) for a window W > 0, else 0.  Everything else - dequantization
of the stored bytes, the rotation back to the original basis, GQA, scale,
softmax - is the decode oracle's plain definition, in fp64.

Pins (tests/test_oracle_prefill.py): a chunk of one query equals the decode
oracle; cache rows after a query's position do not change its output; a
windowed query equals the decode of the truncated sequence with the same
window; an independent scalar loop on BF16-exact K/V.
"""

import math

import numpy as np

from . import formats as F
from .decode import gather_side


def paged_prefill(q, cu_q, k_cache, v_cache, block_tables, seq_lens, nkv, hd,
                  block_size, k_block_stride, v_block_stride, fmt, sm_scale=None,
                  k_scale=None, v_scale=None, window=0):
    """fp64 output [total_q, nq, hd]; q is [total_q, nq, hd], rows of sequence s
    at cu_q[s] .. cu_q[s+1] - 1."""
    q = np.asarray(q, dtype=np.float64)
    total_q, nq, _ = q.shape
    rep = nq // nkv
    k_side, v_side = F.kv_pair(fmt)
    if sm_scale is None or sm_scale == 0:
        sm_scale = 1.0 / math.sqrt(hd)
    block_tables = np.asarray(block_tables, dtype=np.int64)
    out = np.zeros((total_q, nq, hd), dtype=np.float64)
    for s in range(len(seq_lens)):
        L = int(seq_lens[s])
        q0, q1 = int(cu_q[s]), int(cu_q[s + 1])
        C = q1 - q0
        if C == 0 or L == 0:
            continue
        pos = np.arange(L, dtype=np.int64)
        blocks = block_tables[s, pos // block_size]
        offs = pos % block_size
        k = gather_side(k_cache, k_side, blocks, offs, nkv, hd, block_size, k_block_stride, k_scale)
        v = gather_side(v_cache, v_side, blocks, offs, nkv, hd, block_size, v_block_stride, v_scale)
        for i in range(C):
            p = L - C + i
            if p < 0:
                continue   # a query without a cached position attends nothing
            lo = max(0, p + 1 - window) if window > 0 else 0
            for j in range(nq):
                kh = j // rep
                scores = (k[lo:p + 1, kh, :] @ q[q0 + i, j]) * sm_scale
                w = np.exp(scores - scores.max())
                out[q0 + i, j] = (w / w.sum()) @ v[lo:p + 1, kh, :]
    return out
