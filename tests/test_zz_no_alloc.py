"""The decode entry point that allocates nothing (kvq_paged_decode_noalloc).

It is for callers that cannot allocate device memory themselves - e.g. a
runtime whose device memory is all owned by its own pool, or a plugin host
that forbids allocations - so the split-K scratch comes from an array built
into the library.  Checked through the C ABI against kvq_paged_decode with a
caller-provided workspace, on two different decodes in a row (the second
one finds the first one's partials in the shared array), and against the
oracle.  This file is collected last so a stop-at-first-failure run has
already run every other test."""
import numpy as np
import pytest
import torch

from kvq_cases import assert_decode_close, decode_case, oracle_decode
from quantized_paged_kv_reshape_gb300 import _abi as A
from quantized_paged_kv_reshape_gb300 import ops

pytestmark = pytest.mark.gpu


def _device_case(c, dev="cuda"):
    return dict(
        kpool=torch.from_numpy(c["kc"].reshape(c["num_blocks"], c["kst"])).to(dev),
        vpool=torch.from_numpy(c["vc"].reshape(c["num_blocks"], c["vst"])).to(dev),
        q=torch.from_numpy(c["q"]).to(dev),
        tables=torch.from_numpy(c["tables"]).to(dev),
        lens=torch.from_numpy(c["lens"]).to(dev))


def _noalloc(c, d, window=0):
    out = torch.full(c["q"].shape, float("nan"), dtype=torch.float32, device="cuda")
    fmt = A.kvq_format_from_string(c["fmt"])
    A.kvq_paged_decode_noalloc(
        d["q"].data_ptr(), A.KVQ_DTYPE_F32, d["q"].stride(0), d["kpool"].data_ptr(),
        d["vpool"].data_ptr(), out.data_ptr(), A.KVQ_DTYPE_F32, d["tables"].data_ptr(),
        d["tables"].shape[1], d["lens"].data_ptr(), c["q"].shape[0], c["num_blocks"],
        c["nq"], c["nkv"], c["hd"], c["bs"], c["kst"], c["vst"], 0.0, c["k_scale"],
        c["v_scale"], window, 0.0, fmt, None, torch.cuda.current_stream().cuda_stream)
    return out


def _with_workspace(c, d, window=0):
    return ops.paged_decode(d["q"], d["kpool"], d["vpool"], d["tables"], d["lens"], c["fmt"],
                            c["nkv"], c["bs"], k_scale=c["k_scale"], v_scale=c["v_scale"],
                            sliding_window=window)


def test_noalloc_matches_workspace_entry_twice():
    cases = [decode_case("turbo4k_turbo3v", [300, 45, 1, 129], 16, 4, 128, seed=21),
             decode_case("fp8k_turbo2v", [77, 500], 8, 2, 256, seed=22)]
    for c in cases:                      # two calls in a row, different shapes
        d = _device_case(c)
        got = _noalloc(c, d).cpu().numpy().astype(np.float64)
        ref = _with_workspace(c, d).cpu().numpy().astype(np.float64)
        torch.cuda.synchronize()
        assert_decode_close(got, ref)
        assert_decode_close(got, oracle_decode(c))


def test_noalloc_rejects_sizes_beyond_the_array():
    # 4096 sequences x 64 query heads x head_dim 256 needs far more than 8 MiB.
    need = A.kvq_decode_workspace_bytes(4096, 64, 8, 256, 16, 64, 0, 0)
    assert need > A.KVQ_NOALLOC_SCRATCH_BYTES
    with pytest.raises(A.KvqError) as e:
        A.kvq_paged_decode_noalloc(
            16, A.KVQ_DTYPE_F32, 64 * 256, 4096, 4096, 64, A.KVQ_DTYPE_F32, 128, 64, 256,
            4096, 8, 64, 8, 256, 16, 1 << 20, 1 << 20, 0.0, 1.0, 1.0, 0, 0.0, 0, None, None)
    assert e.value.status == A.KVQ_ERR_WORKSPACE


def test_noalloc_graph_capture_reuses_the_last_lookup():
    """A call made while its stream is captured reuses the address the last
    uncaptured call on the device looked up; the captured decode replays
    with new queries and matches the workspace entry each time."""
    c = decode_case("turbo4", [200, 33, 64], 8, 2, 128, seed=31)
    d = _device_case(c)
    _noalloc(c, d)                        # an uncaptured call looks the address up
    torch.cuda.synchronize()
    q_static = d["q"].clone()
    d2 = dict(d, q=q_static)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = _noalloc(c, d2)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    for _ in range(2):
        q_static.copy_(torch.from_numpy(rng.standard_normal(c["q"].shape).astype(np.float32)))
        g.replay()
        torch.cuda.synchronize()
        ref = _with_workspace(c, d2).cpu().numpy().astype(np.float64)
        assert_decode_close(out.cpu().numpy().astype(np.float64), ref)


_FIRST_CALL_IN_CAPTURE = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
from quantized_paged_kv_reshape_gb300 import _abi as A
dev = "cuda"
q = torch.zeros((2, 4, 128), device=dev)
pool = torch.zeros((8, 4096), dtype=torch.uint8, device=dev)
out = torch.zeros((2, 4, 128), device=dev)
tables = torch.zeros((2, 4), dtype=torch.int32, device=dev)
lens = torch.ones(2, dtype=torch.int32, device=dev)
s = torch.cuda.Stream()
g = torch.cuda.CUDAGraph()
status = None
try:
    with torch.cuda.graph(g, stream=s):
        A.kvq_paged_decode_noalloc(
            q.data_ptr(), A.KVQ_DTYPE_F32, 4 * 128, pool.data_ptr(), pool.data_ptr(),
            out.data_ptr(), A.KVQ_DTYPE_F32, tables.data_ptr(), 4, lens.data_ptr(), 2, 8, 4, 2,
            128, 16, 4096, 4096, 0.0, 1.0, 1.0, 0, 0.0, A.kvq_format_from_string("turbo4"),
            None, s.cuda_stream)
except A.KvqError as e:
    status = e.status
    print("MESSAGE", str(e))
print("STATUS", status)
"""


def test_noalloc_first_call_during_capture_fails_cleanly():
    """In a process whose first decode without a workspace is made during
    stream capture there is no address to reuse (a lookup could load the
    module, which capture forbids): the call fails with KVQ_ERR_CUDA before
    launching anything."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FIRST_CALL_IN_CAPTURE, root], capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert f"STATUS {A.KVQ_ERR_CUDA}" in r.stdout, r.stdout
    assert "uncaptured call first" in r.stdout, r.stdout
