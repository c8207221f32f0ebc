"""The bench's algorithmic units (the numerators of its rooflines) on the
CPU, against the per-configuration byte counts worked out from the formats'
sizes: cache bytes per decode layer, bytes per write, FLOPs per prefill."""
import os
import sys

import numpy as np
import pytest

from quantized_paged_kv_reshape_gb300 import _abi as A
from quantized_paged_kv_reshape_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()
    A.lib()


@pytest.mark.parametrize("fmt,expected", [
    ("bf16", 536_870_912),      # 32 x 4096 tokens x 8 heads x (256 + 256) B
    ("fp8", 268_435_456),       # ... x (128 + 128) B
    ("turbo4", 150_994_944),    # ... x (72 + 72) B: 64 B codes + 8 B scales per side
])
def test_llama8b_decode_bytes(fmt, expected):
    assert bench.algorithmic_decode_bytes(fmt, np.full(32, 4096), 8, 128, 16) == expected


def test_longctx_and_gemma_decode_bytes():
    lens = np.full(4, 131072)
    # Turbo4 K (72 B) + Turbo3 V (48 B codes + 8 B scales) per token-head
    assert bench.algorithmic_decode_bytes("turbo4k_turbo3v", lens, 8, 128, 16) == 536_870_912
    assert bench.algorithmic_decode_bytes("turbo4k_turbo3v", lens, 8, 128, 16, 4096) == 16_777_216
    g = np.full(16, 8192)
    # head_dim 256: Turbo2 64 + 16 B, Turbo8 256 + 32 B per side
    assert bench.algorithmic_decode_bytes("turbo2", g, 16, 256, 16) == 335_544_320
    assert bench.algorithmic_decode_bytes("turbo8", g, 16, 256, 16) == 1_207_959_552


def test_write_bytes():
    # 8192 fused-QKV tokens, 16 heads, head_dim 256, bf16 in: read K and V rows,
    # write both Turbo2 sides, read the int64 slots
    assert bench.write_bytes("turbo2", 8192, 16, 256, 16) == (
        2 * 8192 * 16 * 256 * 2 + 8192 * 16 * 160 + 8 * 8192)
    assert bench.write_bytes("bf16", 32, 8, 128, 16) == 2 * 32 * 8 * 128 * 2 + 32 * 8 * 512 + 8 * 32


def test_prefill_flops():
    # per sequence the 512 queries attend 3584 + i + 1 keys; 4 x 128 FLOP per
    # key and query head, 32 query heads, 8 sequences
    keys = 512 * (4096 - 512) + 512 * 513 // 2
    assert bench.prefill_flops(np.full(8, 4096), 512, 32, 128) == 8 * keys * 4 * 128 * 32
    assert bench.prefill_flops(np.full(8, 4096), 512, 32, 128) == 257_731_592_192
