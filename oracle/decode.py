"""Paged decode attention over the quantized cache (oracle side).

The plain definition, in fp64:

1. For sequence s with L = seq_lens[s] and window W, the attended positions
   are p in [lo, L) with lo = max(0, L - W) when W > 0, else 0 (reading
   adopted: the last W positions including the newest; the decode launcher of
   "metrale_model_layers/.../kv_cache_bf16k_turbov.rs" only passes
   ``sliding_window``).  Position p lives in block
   block_tables[s, p // block_size] at offset p % block_size
   ("combs_models/kv.rs", ``PagedKVCache::attention`` / ``gather_window``).
2. Each stored K/V row is dequantized from the cache bytes to fp64:
   bf16 -> its value; fp8 -> E4M3 value * per-tensor scale; turbo{2,3,4} ->
   level[code] * E4M3 group scale; turbo8 -> E4M3 value * BF16 group scale;
   nvfp4 -> E2M1 value * E4M3 group scale (not rotated).
   Rows stored in the Walsh-Hadamard basis ("spark_runtime/kv_cache.rs",
   ``is_wht_rotated``) are rotated back with the fp64 WHT (its own inverse),
   so attention below runs on K and V in the original basis; the kernel's
   rotated-basis shortcut (WHT(Q) before the scores, inverse WHT after P.V)
   is not used here.
3. "combs_models/kv.rs", ``attend`` with one query (no causal mask) and
   ``repeat_kv``: query head j reads kv head j // (nq / nkv);
   scores = (q . k) * sm_scale, P = softmax over the attended positions,
   out = P . V.  sm_scale defaults to 1/sqrt(head_dim).
4. L = 0 (nothing to attend) gives a zero output row (reading adopted).
5. Sparse-V (the decode launcher's doc comment: skip a position's V when its
   attention weight is at most the threshold, 1e-3 by default): terms with
   normalised weight <= threshold are dropped from P.V while the softmax
   denominator is kept (reading adopted).  Threshold 0 disables it.

Pins: tests/test_oracle_decode.py (an independent naive attention loop on
BF16-exact K/V, seq_len 1 -> v_0, q = 0 -> mean of V, window 1 -> last V,
and the rotated-basis identity checked against this plain definition;
``attend`` on given K/V equals the paged decode of a BF16 cache holding the
same bf16-exact rows, and the naive loop directly).
"""

import math

import numpy as np

from . import formats as F
from .codebook import codebook
from .numformats import bf16_decode, e2m1_decode, e4m3_decode
from .cache_write import unpack_codes
from .wht import wht_f64


def dequantize_rows(side, data, scales, hd, scale=None):
    """fp64 values [R, hd] (in the stored basis) from per-row byte images."""
    data = np.asarray(data, dtype=np.uint8)
    r = data.shape[0]
    if side == F.BF16:
        bits = data.reshape(r, hd, 2).astype(np.uint16)
        return bf16_decode(bits[..., 0] | (bits[..., 1] << 8)).astype(np.float64)
    if side == F.FP8:
        return e4m3_decode(data) * float(np.float32(scale))
    ng = hd // F.GROUP
    if side == F.TURBO8:
        sb = np.asarray(scales, np.uint8).reshape(r, ng, 2).astype(np.uint16)
        s = bf16_decode(sb[..., 0] | (sb[..., 1] << 8)).astype(np.float64)
        vals = e4m3_decode(data).reshape(r, ng, F.GROUP)
        return (vals * s[..., None]).reshape(r, hd)
    bits = F.CODE_BITS[side]
    codes = unpack_codes(data, bits, hd)
    s = e4m3_decode(np.asarray(scales, np.uint8).reshape(r, ng))
    if side == F.NVFP4:
        vals = e2m1_decode(codes).reshape(r, ng, F.GROUP)
    else:
        lv64, _, _ = codebook(bits)
        vals = lv64[codes].reshape(r, ng, F.GROUP)
    return (vals * s[..., None]).reshape(r, hd)


def gather_side(cache, side, blocks, offsets, nkv, hd, block_size,
                block_stride_bytes, scale=None, to_original_basis=True):
    """Dequantized rows [n, nkv, hd] (fp64) of positions (blocks[i], offsets[i])."""
    blocks = np.asarray(blocks, dtype=np.int64)
    offsets = np.asarray(offsets, dtype=np.int64)
    n = blocks.size
    dsec = F.data_section_bytes(side, block_size, nkv, hd)
    data_row = dsec // (block_size * nkv)
    scale_row = F.scale_section_bytes(side, block_size, nkv, hd) // (block_size * nkv)
    row = (offsets[:, None] * nkv + np.arange(nkv)[None, :]).reshape(-1)
    base = np.repeat(blocks * block_stride_bytes, nkv)
    d_idx = (base + row * data_row)[:, None] + np.arange(data_row)[None, :]
    data = cache[d_idx]
    scl = None
    if scale_row:
        s_idx = (base + dsec + row * scale_row)[:, None] + np.arange(scale_row)[None, :]
        scl = cache[s_idx]
    vals = dequantize_rows(side, data, scl, hd, scale)
    if to_original_basis and F.is_wht_rotated(side):
        vals = wht_f64(vals)
    return vals.reshape(n, nkv, hd)


def attended_positions(seq_len, window):
    """Positions a one-token decode attends to."""
    lo = max(0, seq_len - window) if window > 0 else 0
    return np.arange(lo, seq_len, dtype=np.int64)


def attend(q, k, v, sm_scale=None, sparse_v_threshold=0.0):
    """fp64 output [nq, hd] of one query per head over given K/V rows.

    "combs_models/kv.rs", ``attend`` for one query (no mask) with
    ``repeat_kv``: q [nq, hd], k and v [n, nkv, hd] (the attended positions,
    in the original basis); query head j reads kv head j // (nq / nkv).
    scores = (q . k) * sm_scale, P = softmax over the n positions, out = P.V;
    sparse-V drops terms whose normalised weight is <= the threshold (the
    denominator kept).  n = 0 gives zeros.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    nq, hd = q.shape
    nkv = k.shape[1]
    rep = nq // nkv
    if sm_scale is None or sm_scale == 0:
        sm_scale = 1.0 / math.sqrt(hd)
    out = np.zeros((nq, hd), dtype=np.float64)
    if k.shape[0] == 0:
        return out
    for j in range(nq):
        kh = j // rep
        scores = (k[:, kh, :] @ q[j]) * sm_scale
        w = np.exp(scores - scores.max())
        p = w / w.sum()
        if sparse_v_threshold > 0:
            p = np.where(p <= sparse_v_threshold, 0.0, p)
        out[j] = p @ v[:, kh, :]
    return out


def paged_decode(q, k_cache, v_cache, block_tables, seq_lens, nkv, hd,
                 block_size, k_block_stride, v_block_stride, fmt,
                 sm_scale=None, k_scale=None, v_scale=None, window=0,
                 sparse_v_threshold=0.0):
    """fp64 output [num_seqs, nq, hd] of one-query-per-sequence attention."""
    q = np.asarray(q, dtype=np.float64)
    nseq, nq, _ = q.shape
    k_side, v_side = F.kv_pair(fmt)
    block_tables = np.asarray(block_tables, dtype=np.int64)
    out = np.zeros((nseq, nq, hd), dtype=np.float64)
    for s in range(nseq):
        pos = attended_positions(int(seq_lens[s]), window)
        if pos.size == 0:
            continue
        blocks = block_tables[s, pos // block_size]
        offs = pos % block_size
        k = gather_side(k_cache, k_side, blocks, offs, nkv, hd, block_size,
                        k_block_stride, k_scale)
        v = gather_side(v_cache, v_side, blocks, offs, nkv, hd, block_size,
                        v_block_stride, v_scale)
        out[s] = attend(q[s], k, v, sm_scale, sparse_v_threshold)
    return out
