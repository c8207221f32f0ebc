"""The bench's quality comparison on CPU tensors: maximum and mean absolute
differences and the per-row cosine, against values worked out by hand."""
import math
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_identical_outputs():
    x = torch.randn(3, 4, 8)
    q = bench._compare(x, x)
    assert q["max_abs"] == 0.0 and q["mean_abs"] == 0.0
    assert abs(q["cos_min"] - 1.0) < 1e-6 and abs(q["cos_mean"] - 1.0) < 1e-6


def test_hand_worked_rows():
    ref = torch.tensor([[[1.0, 0.0], [0.0, 2.0]]])   # rows (1, 0) and (0, 2)
    got = torch.tensor([[[1.0, 1.0], [0.0, -2.0]]])  # 45 degrees off; opposite
    q = bench._compare(got, ref)
    assert q["max_abs"] == 4.0                        # |-2 - 2|
    assert q["mean_abs"] == (0 + 1 + 0 + 4) / 4
    assert abs(q["cos_min"] + 1.0) < 1e-6
    assert abs(q["cos_mean"] - (1 / math.sqrt(2) - 1) / 2) < 1e-6


def test_zero_reference_rows_are_skipped():
    ref = torch.tensor([[[0.0, 0.0], [3.0, 4.0]]])   # an empty sequence's zero row
    got = torch.tensor([[[0.0, 0.0], [3.0, 4.0]]])
    q = bench._compare(got, ref)
    assert abs(q["cos_min"] - 1.0) < 1e-6 and abs(q["cos_mean"] - 1.0) < 1e-6


def test_sample_sequences():
    import numpy as np
    assert bench.sample_sequences(np.array([512, 9000, 700, 16384, 512])) == [0, 3]
    assert bench.sample_sequences(np.full(32, 4096)) == [0, 31]
    assert bench.sample_sequences(np.full(4, 131072)) == [0]
    assert bench.sample_sequences(np.array([5])) == [0]


def test_oracle_quality_against_hand_worked_attention():
    """One sequence of two positions, one kv head and one query head: the
    oracle's attention of q = 0 is the mean of the V rows; a GPU row equal to
    it scores 0 / cosine 1, one off by 0.5 in a dim scores that, and a window
    of 1 attends the newest row only."""
    import numpy as np
    k = np.zeros((2, 1, 2))
    v = np.array([[[1.0, 0.0]], [[3.0, 2.0]]])
    q = np.zeros((1, 2))
    exact = np.array([[2.0, 1.0]])
    off = np.array([[2.5, 1.0]])
    r = bench.oracle_quality([("llama8b", "bf16", 0, 7, q, k, v, exact, off)])
    e, s = r["llama8b:bf16"]["exact"], r["llama8b:bf16"]["sparse_v"]
    assert e["max_abs"] == 0.0 and abs(e["cos_min"] - 1.0) < 1e-12
    assert s["max_abs"] == 0.5 and s["mean_abs"] == 0.25
    assert r["llama8b:bf16"]["seqs"] == [7]
    w = bench.oracle_quality([("longctx", "turbo4", 1, 0, q, k, v, np.array([[3.0, 2.0]]),
                               np.array([[3.0, 2.0]]))])
    assert w["longctx:turbo4@window1"]["exact"]["max_abs"] == 0.0
