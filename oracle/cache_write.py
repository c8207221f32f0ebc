"""Quantized paged cache write (oracle side).

What it computes, per (token t, kv head h) row x of head_dim elements:

* ``bf16``   : x rounded to BF16 (RNE), 2 bytes little-endian per element.
* ``fp8``    : E4M3(x / s) with the caller's per-tensor scale s (fp32 divide).
* ``turbo{2,3,4}``: y = WHT(x) (fp32, fixed butterfly order, see ``wht``);
  per 16-element group g: ratio = amax_g / c_max (fp32 divide, c_max the
  largest fp32 codebook level), scale byte = E4M3(ratio), s = its value;
  per element: v = y / s (fp32 divide), code = number of fp32 thresholds
  <= v.  A group whose scale byte decodes to 0 stores code 2**(b-1) (the
  smallest positive level) for every element; it dequantizes to 0.
* ``turbo8`` : y = WHT(x); s = BF16(amax_g / 448) per group; data byte =
  E4M3(y / s) (fp32 divide); a zero scale stores data byte 0x00.
* ``nvfp4``  : no rotation; per 16-element group g of x: scale byte =
  E4M3(amax_g / 6) (fp32 divide, 6 = the largest E2M1 magnitude), s = its
  value; per element: code = E2M1(x / s) (fp32 divide, RNE, saturating);
  a group whose scale byte decodes to 0 stores code 0 (dequantizes to 0).
  Packed and laid out exactly like turbo4 ("spark_runtime/kv_cache.rs",
  ``block_bytes_dims``: "Same byte layout, different codebook (E2M1 vs
  Lloyd-Max)").

Layout of one block of one side ("metrale_model_layers/.../
kv_cache_bf16k_turbov.rs", module invariants; "spark_runtime/kv_cache.rs",
``block_bytes_dims`` and the ``*_data_bytes`` / ``*_scale_bytes`` helpers):
element e = (slot_in_block * nkv + h) * hd + d.  The code section holds the
codes of e = 0.. packed LSB-first into a little-endian bit stream (4-bit: low
nibble = even e; 2-bit: bits 2(e%4); 3-bit: bits 3e.. of the stream, 8 codes
per 3 bytes); the scale section follows it at ``data_section_bytes`` and
holds scale g = e // 16 (one byte, or two little-endian bytes for turbo8).

The row is addressed by ``slot_mapping[t]``: block = slot // block_size,
offset = slot % block_size ("combs_models/kv.rs", ``PagedKVCache::attention``:
the page id is the table entry at pos / page_size, the slot pos % page_size).
A negative slot skips the row (reading adopted; the pages are silent).

Inputs are read through per-token element strides ``key_stride`` /
``value_stride``: row (t, h) starts at element t*stride + h*hd (the page's
launcher passes both strides, so K/V may be views of a fused QKV buffer).

Pins: tests/test_oracle_write.py (hand-worked 16-element groups in
tests/golden/turbo_groups.txt, brute-force packing round trips, an
independent big-integer packing of 3-bit codes, the unit-scale MSE against
the closed-form distortion, and the byte arithmetic of the section sizes).
"""

import numpy as np

from . import formats as F
from .codebook import codebook, quantize_unit
from .numformats import (bf16_encode, e4m3_decode, e4m3_encode, bf16_decode, e2m1_encode,
                         E2M1_MAX)
from .wht import fwht_f32


def quantize_rotated(side, y):
    """Group-quantize rows ``y`` [R, hd] that are already in the rotated basis.

    turbo{2,3,4} -> (uint8 codes [R, hd], uint8 E4M3 scale bytes [R, hd/16])
    turbo8       -> (uint8 E4M3 data [R, hd], uint16 BF16 scales [R, hd/16])
    """
    y = np.asarray(y, dtype=np.float32)
    r, hd = y.shape
    g = y.reshape(r, hd // F.GROUP, F.GROUP)
    amax = np.max(np.abs(g), axis=-1)
    if side == F.TURBO8:
        s_bits = bf16_encode(amax / np.float32(448.0))
        s = bf16_decode(s_bits)[..., None]
        with np.errstate(divide="ignore", invalid="ignore"):
            v = g / s
        data = e4m3_encode(v)
        data = np.where(s == 0, np.uint8(0), data).astype(np.uint8)
        return data.reshape(r, hd), s_bits
    bits = F.CODE_BITS[side]
    _, lv32, thr = codebook(bits)
    c_max = lv32[-1]
    s_byte = e4m3_encode(amax / c_max)
    s = e4m3_decode(s_byte).astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        v = g / s
    codes = quantize_unit(v, thr)
    codes = np.where(s == 0, np.uint8(1 << (bits - 1)), codes).astype(np.uint8)
    return codes.reshape(r, hd), s_byte


def quantize_nvfp4(x):
    """NVFP4 rows x [R, hd] (original basis): (uint8 E2M1 codes [R, hd],
    uint8 E4M3 scale bytes [R, hd/16])."""
    x = np.asarray(x, dtype=np.float32)
    r, hd = x.shape
    g = x.reshape(r, hd // F.GROUP, F.GROUP)
    amax = np.max(np.abs(g), axis=-1)
    s_byte = e4m3_encode(amax / np.float32(E2M1_MAX))
    s = e4m3_decode(s_byte).astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        v = g / s
    codes = np.where(s == 0, np.uint8(0), e2m1_encode(v)).astype(np.uint8)
    return codes.reshape(r, hd), s_byte


def quantize_rows(side, x, scale=None):
    """Encode rows ``x`` [R, hd] (fp32) of one side.

    Returns (codes or raw, group_scales):
      bf16  -> (uint16 [R, hd], None)
      fp8   -> (uint8 [R, hd], None)
      turbo -> (uint8 codes [R, hd], uint8 scale bytes [R, hd/16])
      turbo8-> (uint8 E4M3 data [R, hd], uint16 BF16 scales [R, hd/16])
    """
    x = np.asarray(x, dtype=np.float32)
    if side == F.BF16:
        return bf16_encode(x), None
    if side == F.FP8:
        s = np.float32(scale)
        return e4m3_encode(x / s), None
    if side == F.NVFP4:
        return quantize_nvfp4(x)
    return quantize_rotated(side, fwht_f32(x))


def pack_codes(codes, bits):
    """Pack uint8 codes [..., n] (n*bits % 8 == 0) LSB-first into bytes."""
    codes = np.asarray(codes, dtype=np.uint8)
    lead, n = codes.shape[:-1], codes.shape[-1]
    shifts = np.arange(bits, dtype=np.uint8)
    bitplane = (codes[..., :, None] >> shifts) & 1          # [..., n, bits]
    stream = bitplane.reshape(lead + (n * bits,))
    return np.packbits(stream, axis=-1, bitorder="little")


def unpack_codes(packed, bits, n):
    """Inverse of ``pack_codes``: the first n codes of the bit stream."""
    packed = np.asarray(packed, dtype=np.uint8)
    lead = packed.shape[:-1]
    stream = np.unpackbits(packed, axis=-1, bitorder="little")[..., : n * bits]
    planes = stream.reshape(lead + (n, bits)).astype(np.uint8)
    weights = (1 << np.arange(bits)).astype(np.uint8)
    return np.sum(planes * weights, axis=-1).astype(np.uint8)


def encode_rows_bytes(side, x, scale=None):
    """Per-row byte images: (data bytes [R, data_row], scale bytes [R, scale_row])."""
    enc, sc = quantize_rows(side, x, scale)
    r = enc.shape[0]
    if side == F.BF16:
        data = enc.astype("<u2").view(np.uint8).reshape(r, -1)
        return data, np.zeros((r, 0), np.uint8)
    if side == F.FP8:
        return enc, np.zeros((r, 0), np.uint8)
    if side == F.TURBO8:
        return enc, sc.astype("<u2").view(np.uint8).reshape(r, -1)
    return pack_codes(enc, F.CODE_BITS[side]), sc


def cache_write(side, rows, cache, slot_mapping, nkv, hd, block_size,
                block_stride_bytes, scale=None, row_stride=None):
    """Scatter the rows of one side into ``cache`` (uint8 [num_blocks*stride]).

    ``rows``: fp32 or bf16-valued fp32 array.  If ``row_stride`` is given,
    ``rows`` is a flat element array and row (t, h) starts at
    t*row_stride + h*hd; otherwise ``rows`` is [T, nkv, hd].
    Modifies ``cache`` in place and returns it.
    """
    slot_mapping = np.asarray(slot_mapping, dtype=np.int64)
    t_count = slot_mapping.shape[0]
    if row_stride is None:
        x = np.asarray(rows, dtype=np.float32).reshape(t_count, nkv, hd)
    else:
        flat = np.asarray(rows, dtype=np.float32).reshape(-1)
        idx = (np.arange(t_count)[:, None, None] * row_stride
               + np.arange(nkv)[None, :, None] * hd
               + np.arange(hd)[None, None, :])
        x = flat[idx]
    keep = slot_mapping >= 0
    x = x[keep]
    slots = slot_mapping[keep]
    if slots.size == 0:
        return cache
    data, scl = encode_rows_bytes(side, x.reshape(-1, hd), scale)
    data_row = data.shape[1]
    scale_row = scl.shape[1]
    dsec = F.data_section_bytes(side, block_size, nkv, hd)
    block = slots // block_size
    off = slots % block_size
    # Row (token i, head h) sits at row index off*nkv + h inside its block.
    row = (off[:, None] * nkv + np.arange(nkv)[None, :]).reshape(-1)
    base = np.repeat(block * block_stride_bytes, nkv)
    d_idx = (base + row * data_row)[:, None] + np.arange(data_row)[None, :]
    cache[d_idx] = data
    if scale_row:
        s_idx = (base + dsec + row * scale_row)[:, None] + np.arange(scale_row)[None, :]
        cache[s_idx] = scl
    return cache
