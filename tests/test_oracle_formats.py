"""Pins of the oracle's format catalogue against what the pages print.

"spark_runtime/kv_cache.rs": the KvCacheDtype doc comments (bytes per element,
"22% smaller than turbo4", "6.4x compression vs bf16", BF16 Turbo8 scales
costing "~6% extra cache memory"), FromStr's accepted spellings, kv_pair and
is_wht_rotated.  "metrale_model_layers/.../kv_cache_bf16k_turbov.rs":
Turbo2V is "2.5 bits per V element", Turbo3V "3/8 byte per element" plus one
FP8 scale per 16 elements.
"""
import pytest

import oracle.formats as F

BS, NKV, HD = 16, 8, 128
E = BS * NKV * HD


def bits_per_elem(side):
    return 8.0 * F.block_bytes(side, BS, NKV, HD) / E


def test_printed_bytes_per_element():
    assert bits_per_elem("bf16") == 16.0          # "2 bytes per element"
    assert bits_per_elem("fp8") == 8.0            # "1 byte per element"
    assert bits_per_elem("nvfp4") == 4.5          # "0.5 bytes data + per-group FP8 scale"
    assert bits_per_elem("turbo4") == bits_per_elem("nvfp4")  # "Same byte layout as NVFP4"
    assert bits_per_elem("turbo2") == 2.5         # "2.5 bits per V element"
    assert F.data_section_bytes("turbo3", BS, NKV, HD) * 8 == 3 * E  # "3/8 byte per element"


def test_printed_ratios():
    # "22% smaller than turbo4"
    assert round(100 * (1 - bits_per_elem("turbo3") / bits_per_elem("turbo4"))) == 22
    # "6.4x compression vs bf16"
    assert bits_per_elem("bf16") / bits_per_elem("turbo2") == pytest.approx(6.4)
    # BF16 scales instead of FP8 ones: "~6% extra cache memory"
    fp8_scaled = 8 + 8 / 16
    assert round(100 * (bits_per_elem("turbo8") / fp8_scaled - 1)) == 6


def test_page_sizes_llama_block():
    # One block of 16 tokens x 8 heads x 128 dims.
    assert F.block_bytes("turbo4", BS, NKV, HD) == 8192 + 1024
    assert F.block_bytes("turbo3", BS, NKV, HD) == 6144 + 1024
    assert F.block_bytes("turbo2", BS, NKV, HD) == 4096 + 1024
    assert F.block_bytes("bf16", BS, NKV, HD) == 32768
    assert F.block_bytes("turbo8", BS, NKV, HD) == 16384 + 2048


SPELLINGS = {
    "bf16": ("bf16", "bf16"), "fp8": ("fp8", "fp8"), "nvfp4": ("nvfp4", "nvfp4"),
    "turbo4": ("turbo4", "turbo4"), "turbo3": ("turbo3", "turbo3"),
    "turbo2": ("turbo2", "turbo2"), "turbo8": ("turbo8", "turbo8"),
    "turbo4k_turbo3v": ("turbo4", "turbo3"), "turbo4k3v": ("turbo4", "turbo3"),
    "turbo4k_turbo8v": ("turbo4", "turbo8"), "turbo4k8v": ("turbo4", "turbo8"),
    "turbo3k_turbo8v": ("turbo3", "turbo8"), "turbo3k8v": ("turbo3", "turbo8"),
    "bf16k_turbo4v": ("bf16", "turbo4"), "bf16k4v": ("bf16", "turbo4"),
    "bf16k_turbo3v": ("bf16", "turbo3"), "bf16k3v": ("bf16", "turbo3"),
    "fp8k_turbo4v": ("fp8", "turbo4"), "fp8k4v": ("fp8", "turbo4"),
    "fp8k_turbo3v": ("fp8", "turbo3"), "fp8k3v": ("fp8", "turbo3"),
    "bf16k_turbo2v": ("bf16", "turbo2"), "bf16k2v": ("bf16", "turbo2"),
    "fp8k_turbo2v": ("fp8", "turbo2"), "fp8k2v": ("fp8", "turbo2"),
}


@pytest.mark.parametrize("name", sorted(SPELLINGS))
def test_spellings_and_pairs(name):
    assert F.kv_pair(name) == SPELLINGS[name]


def test_unknown_spelling():
    with pytest.raises(ValueError):
        F.format_from_string("int4")


def test_rotated_sides():
    assert {s for s in F.SIDE_FORMATS if F.is_wht_rotated(s)} == {
        "turbo2", "turbo3", "turbo4", "turbo8"}
    assert sum(F.is_asymmetric(f) for f in F.FORMATS) == 9
