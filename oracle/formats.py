"""Format catalogue and per-block byte arithmetic (oracle side).

Follows "spark_runtime/kv_cache.rs", ``enum KvCacheDtype`` (variant list and
their one-line storage descriptions), ``kv_pair``, ``is_wht_rotated``,
``is_asymmetric``, ``FromStr`` (accepted spellings) and
``KvCacheConfig::block_bytes_dims`` / the ``turbo*_data_bytes`` /
``turbo*_scale_bytes`` section helpers.

A *side* format is what one pool (K or V) stores; a combined format names the
pair.  Byte counts per block of E = block_size * num_kv_heads * head_dim
elements, as the page's ``block_bytes_dims`` states them:

  bf16   2E               fp8    E
  turbo4 E/2  + E/16      turbo3 3E/8 + E/16
  turbo2 E/4  + E/16      turbo8 E    + 2*E/16   (BF16 group scales)
  nvfp4  E/2  + E/16      (same layout as turbo4, E2M1 codebook)

Pinned by tests/test_oracle_formats.py against the page's own numbers
(spelled-out byte counts, the spellings of ``FromStr``).
"""

GROUP = 16  # NVFP4_GROUP_SIZE: one scale per 16 consecutive elements

# Side formats.
BF16, FP8, NVFP4, TURBO4, TURBO3, TURBO2, TURBO8 = (
    "bf16", "fp8", "nvfp4", "turbo4", "turbo3", "turbo2", "turbo8")
SIDE_FORMATS = (BF16, FP8, NVFP4, TURBO4, TURBO3, TURBO2, TURBO8)

# Combined formats in the page's enum order, with their (K, V) pair.
FORMATS = {
    "bf16": (BF16, BF16),
    "fp8": (FP8, FP8),
    "nvfp4": (NVFP4, NVFP4),
    "turbo4": (TURBO4, TURBO4),
    "turbo3": (TURBO3, TURBO3),
    "turbo2": (TURBO2, TURBO2),
    "turbo8": (TURBO8, TURBO8),
    "turbo4k_turbo3v": (TURBO4, TURBO3),
    "turbo4k_turbo8v": (TURBO4, TURBO8),
    "turbo3k_turbo8v": (TURBO3, TURBO8),
    "bf16k_turbo4v": (BF16, TURBO4),
    "bf16k_turbo3v": (BF16, TURBO3),
    "fp8k_turbo4v": (FP8, TURBO4),
    "fp8k_turbo3v": (FP8, TURBO3),
    "bf16k_turbo2v": (BF16, TURBO2),
    "fp8k_turbo2v": (FP8, TURBO2),
}

# Short aliases accepted by the page's FromStr.
_ALIASES = {
    "turbo4k3v": "turbo4k_turbo3v", "turbo4k8v": "turbo4k_turbo8v",
    "turbo3k8v": "turbo3k_turbo8v", "bf16k4v": "bf16k_turbo4v",
    "bf16k3v": "bf16k_turbo3v", "fp8k4v": "fp8k_turbo4v",
    "fp8k3v": "fp8k_turbo3v", "bf16k2v": "bf16k_turbo2v",
    "fp8k2v": "fp8k_turbo2v",
}

# Bits per stored code for the codebook sides.
CODE_BITS = {TURBO4: 4, TURBO3: 3, TURBO2: 2, NVFP4: 4}


def format_from_string(s):
    """Parse a ``--kv-cache-dtype`` spelling; raises ValueError if unknown."""
    if s in FORMATS:
        return s
    if s in _ALIASES:
        return _ALIASES[s]
    raise ValueError(f"unsupported kv cache format {s!r}")


def format_name(fmt):
    """Canonical spelling (the long form for the asymmetric pairs)."""
    return format_from_string(fmt)


def kv_pair(fmt):
    """(K side format, V side format)."""
    return FORMATS[format_from_string(fmt)]


def is_wht_rotated(side):
    """True where the side is stored in the Walsh-Hadamard basis."""
    return side in (TURBO2, TURBO3, TURBO4, TURBO8)


def is_asymmetric(fmt):
    k, v = kv_pair(fmt)
    return k != v


def data_section_bytes(side, block_size, nkv, hd):
    """Bytes of the code (or raw data) section of one block of one side."""
    e = block_size * nkv * hd
    if side == BF16:
        return 2 * e
    if side in (FP8, TURBO8):
        return e
    if side in (NVFP4, TURBO4):
        return e // 2
    if side == TURBO3:
        return e * 3 // 8
    if side == TURBO2:
        return e // 4
    raise ValueError(side)


def scale_section_bytes(side, block_size, nkv, hd):
    """Bytes of the per-group scale section (0 for raw sides)."""
    e = block_size * nkv * hd
    if side in (BF16, FP8):
        return 0
    if side == TURBO8:
        return 2 * (e // GROUP)
    return e // GROUP


def block_bytes(side, block_size, nkv, hd):
    """Bytes per block of one side (K or V, not both)."""
    return (data_section_bytes(side, block_size, nkv, hd)
            + scale_section_bytes(side, block_size, nkv, hd))
