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
