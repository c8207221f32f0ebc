"""FP8 E4M3 and BF16 encoders / decoders written from the format definitions.

"spark_runtime/kv_cache.rs": ``Fp8`` is "FP8 E4M3 with per-tensor scale", the
Turbo2/3/4 group scales are FP8 (one byte per 16 elements) and the Turbo8
group scales are BF16 (two bytes).  The pages fix the formats, not the
rounding; the reading used here is round-to-nearest-even, saturating to the
largest finite value (448 for E4M3) and keeping subnormals.

E4M3 (OCP FP8, "fn" variant): 1 sign bit, 4 exponent bits (bias 7), 3
mantissa bits; no infinities; S.1111.111 is NaN; largest finite 448;
subnormals m/8 * 2^-6.

Encoding here is literally "pick the nearest representable value": every
finite E4M3 magnitude is enumerated from the decoder and the input magnitude
is matched to the closest one, ties to the one with the even code.  Nothing
bit-twiddles, so the encoder is checkable by eye against the definition.

BF16: the upper 16 bits of an IEEE fp32 pattern.  Encoding rounds the fp32
value to the nearest bf16, ties to even mantissa.

E2M1 (the 4-bit element of NVFP4, "spark_runtime/kv_cache.rs" ``Nvfp4``:
"E2M1 packed nibbles"): 1 sign bit (bit 3), 2 exponent bits (bias 1), 1
mantissa bit; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 for codes 0..7; no
infinities or NaN.  Encoding is again "pick the nearest representable
magnitude", ties to the even code, saturating at 6, sign from the sign bit of
the input (the pages name the format only; RNE-saturate is the reading).

Pins (tests/test_oracle_numformats.py): all 256 E4M3 codes against torch's
float8_e4m3fn view (a library special case); encoding against torch's RNE
cast inside the finite range; hand-checked saturation, subnormal and tie
cases; BF16 against torch's bfloat16 cast; the 16 E2M1 codes and their
midpoint ties by hand, and the E2M1 encoder against torch's float4_e2m1fn_x2
where that dtype exists.
"""

import numpy as np

E4M3_MAX = 448.0


def e4m3_decode(codes):
    """fp64 values of uint8 E4M3 codes (NaN for S.1111.111)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = c & 0x7
    normal = (1.0 + man / 8.0) * np.power(2.0, exp - 7.0)
    sub = (man / 8.0) * 2.0 ** -6
    mag = np.where(exp == 0, sub, normal)
    mag = np.where((exp == 15) & (man == 7), np.nan, mag)
    return sign * mag


# All finite non-negative magnitudes, ascending, with their codes 0x00..0x7E.
_POS_CODES = np.arange(0x7F, dtype=np.uint8)
_POS_VALUES = e4m3_decode(_POS_CODES)
assert np.all(np.diff(_POS_VALUES) > 0)


def e4m3_encode(x):
    """uint8 E4M3 codes of fp32/fp64 values: RNE, saturating, subnormals kept.

    NaN maps to 0x7F.  The sign of zero is kept (-0.0 -> 0x80).
    """
    x = np.asarray(x, dtype=np.float64)
    mag = np.abs(x)
    mag_sat = np.minimum(mag, E4M3_MAX)
    # Neighbours: largest representable <= mag, smallest representable >= mag.
    hi_idx = np.searchsorted(_POS_VALUES, mag_sat, side="left")
    hi_idx = np.minimum(hi_idx, len(_POS_VALUES) - 1)
    lo_idx = np.where(_POS_VALUES[hi_idx] == mag_sat, hi_idx,
                      np.maximum(hi_idx - 1, 0))
    lo_v = _POS_VALUES[lo_idx]
    hi_v = _POS_VALUES[hi_idx]
    d_lo = mag_sat - lo_v
    d_hi = hi_v - mag_sat
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi_idx % 2 == 0) & (hi_idx != lo_idx))
    idx = np.where(pick_hi, hi_idx, lo_idx)
    code = _POS_CODES[idx].astype(np.uint8)
    code = np.where(np.signbit(x), code | np.uint8(0x80), code).astype(np.uint8)
    code = np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)
    return code


def bf16_encode(x):
    """uint16 BF16 patterns of fp32 values, round to nearest even."""
    x = np.asarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    upper = bits >> 16
    lower = bits & 0xFFFF
    # Round up when the dropped half is above 0x8000, or exactly 0x8000 and the
    # kept part is odd (ties to even).
    round_up = (lower > 0x8000) | ((lower == 0x8000) & ((upper & 1) == 1))
    out = (upper + round_up.astype(np.uint64)) & 0xFFFF
    nan = np.isnan(x)
    out = np.where(nan, (upper | 0x40) & 0xFFFF, out)  # keep NaN a quiet NaN
    return out.astype(np.uint16)


def bf16_decode(bits):
    """fp32 values of uint16 BF16 patterns (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


E2M1_MAX = 6.0


def e2m1_decode(codes):
    """fp64 values of 4-bit E2M1 codes (uint8 holding 0..15)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64) & 0xF
    sign = np.where(c & 0x8, -1.0, 1.0)
    exp = (c >> 1) & 0x3
    man = c & 0x1
    mag = np.where(exp == 0, man * 0.5, (1.0 + man / 2.0) * np.power(2.0, exp - 1.0))
    return sign * mag


_E2M1_POS_CODES = np.arange(8, dtype=np.uint8)
_E2M1_POS_VALUES = e2m1_decode(_E2M1_POS_CODES)
assert np.all(np.diff(_E2M1_POS_VALUES) > 0)


def e2m1_encode(x):
    """4-bit E2M1 codes (uint8 0..15) of fp32/fp64 values: RNE, saturating.

    The sign bit follows the input's sign bit (-0.0 and negatives that round
    to zero give 0x8).  NaN is not expected (the callers divide finite values
    by nonzero scales) and maps to 0x7.
    """
    x = np.asarray(x, dtype=np.float64)
    mag = np.minimum(np.abs(x), E2M1_MAX)
    hi_idx = np.searchsorted(_E2M1_POS_VALUES, mag, side="left")
    hi_idx = np.minimum(hi_idx, len(_E2M1_POS_VALUES) - 1)
    lo_idx = np.where(_E2M1_POS_VALUES[hi_idx] == mag, hi_idx, np.maximum(hi_idx - 1, 0))
    d_lo = mag - _E2M1_POS_VALUES[lo_idx]
    d_hi = _E2M1_POS_VALUES[hi_idx] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi_idx % 2 == 0) & (hi_idx != lo_idx))
    code = np.where(pick_hi, hi_idx, lo_idx).astype(np.uint8)
    code = np.where(np.signbit(x), code | np.uint8(0x8), code).astype(np.uint8)
    code = np.where(np.isnan(x), np.uint8(0x7), code).astype(np.uint8)
    return code
