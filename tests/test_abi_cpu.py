"""CPU checks of the C ABI: the library loads, exports every symbol that
include/kvq.h declares, its catalogue / byte arithmetic / codebook equal the
oracle's, and invalid arguments are rejected on the host before anything is
launched (no GPU needed for any of this)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from quantized_paged_kv_reshape_gb300 import _abi as A
from quantized_paged_kv_reshape_gb300 import build as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "kvq.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()
    A.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_\w+)\s*\(", text)))


def test_exports_every_declared_symbol():
    names = declared_functions()
    assert len(names) >= 12
    handle = ctypes.CDLL(A.LIB_PATH)
    missing = [n for n in names if not hasattr(handle, n)]
    assert not missing


def test_catalogue_matches_oracle():
    for i, name in enumerate(A.FORMAT_NAMES):
        assert A.kvq_format_name(i) == name
        k, v = oracle.kv_pair(name)
        assert A.FORMAT_NAMES[A.kvq_side_format(i, 0)] == k
        assert A.FORMAT_NAMES[A.kvq_side_format(i, 1)] == v
        assert A.kvq_side_is_rotated(i, 0) == int(oracle.is_wht_rotated(k))
        assert A.kvq_side_is_rotated(i, 1) == int(oracle.is_wht_rotated(v))
    for alias, full in [("turbo4k3v", "turbo4k_turbo3v"), ("fp8k2v", "fp8k_turbo2v"),
                        ("bf16k4v", "bf16k_turbo4v"), ("turbo3k8v", "turbo3k_turbo8v")]:
        assert A.kvq_format_from_string(alias) == A.FORMAT_NAMES.index(full)
    with pytest.raises(A.KvqError) as e:
        A.kvq_format_from_string("int4")
    assert e.value.status == A.KVQ_ERR_FORMAT
    assert A.kvq_format_name(99) is None


@pytest.mark.parametrize("bs", [1, 8, 16, 32])
@pytest.mark.parametrize("nkv", [1, 2, 8, 16])
@pytest.mark.parametrize("hd", [64, 128, 256])
def test_block_bytes_match_oracle(bs, nkv, hd):
    for i, name in enumerate(A.FORMAT_NAMES):
        k, v = oracle.kv_pair(name)
        assert A.kvq_block_bytes(i, 0, bs, nkv, hd) == oracle.block_bytes(k, bs, nkv, hd)
        assert A.kvq_block_bytes(i, 1, bs, nkv, hd) == oracle.block_bytes(v, bs, nkv, hd)
        assert A.kvq_data_section_bytes(i, 1, bs, nkv, hd) == oracle.data_section_bytes(v, bs, nkv, hd)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_codebook_bits_equal_oracle(bits):
    lv, th = A.kvq_codebook(bits)
    _, lv32, th32 = oracle.codebook(bits)
    assert np.array_equal(np.array(lv, np.float32).view(np.uint32), lv32.view(np.uint32))
    assert np.array_equal(np.array(th, np.float32).view(np.uint32), th32.view(np.uint32))


def _write(**over):
    args = dict(key=16, value=16, in_dtype=A.KVQ_DTYPE_BF16, k_cache=4096, v_cache=4096,
                slot_mapping=64, num_tokens=4, num_blocks=8, num_kv_heads=2, head_dim=128,
                block_size=16, key_stride=256, value_stride=256, k_block_stride_bytes=8192,
                v_block_stride_bytes=8192, k_scale=1.0, v_scale=1.0, fmt=0, error_flag=None,
                stream=None)
    args.update(over)
    with pytest.raises(A.KvqError) as e:
        A.kvq_cache_write(**args)
    return e.value.status


def test_write_rejects_bad_arguments():
    assert _write(key=None) == A.KVQ_ERR_ARG
    assert _write(head_dim=96) == A.KVQ_ERR_SHAPE
    assert _write(fmt=42) == A.KVQ_ERR_FORMAT
    assert _write(in_dtype=7) == A.KVQ_ERR_FORMAT
    assert _write(k_block_stride_bytes=4096) == A.KVQ_ERR_ARG  # below block bytes
    assert _write(k_cache=4104) == A.KVQ_ERR_ALIGN
    assert _write(v_block_stride_bytes=8200) == A.KVQ_ERR_ALIGN
    assert _write(key_stride=100) == A.KVQ_ERR_ARG
    assert _write(fmt=1, k_scale=0.0) == A.KVQ_ERR_ARG   # fp8 needs a scale
    assert _write(num_tokens=-1) == A.KVQ_ERR_ARG


def _decode(**over):
    args = dict(q=16, q_dtype=A.KVQ_DTYPE_BF16, q_stride=4096, k_cache=4096, v_cache=4096,
                out=64, out_dtype=A.KVQ_DTYPE_F32, block_tables=128, max_blocks_per_seq=4,
                seq_lens=256, num_seqs=2, num_blocks=8, num_q_heads=32, num_kv_heads=8,
                head_dim=128, block_size=16, k_block_stride_bytes=65536,
                v_block_stride_bytes=65536, sm_scale=0.0, k_scale=1.0, v_scale=1.0,
                sliding_window=0, sparse_v_threshold=0.0, workspace=8192,
                workspace_bytes=1 << 30, fmt=0, error_flag=None, stream=None)
    args.update(over)
    with pytest.raises(A.KvqError) as e:
        A.kvq_paged_decode(**args)
    return e.value.status


def test_decode_rejects_bad_arguments():
    assert _decode(num_q_heads=30) == A.KVQ_ERR_SHAPE      # not a multiple
    assert _decode(num_q_heads=128) == A.KVQ_ERR_SHAPE     # ratio 16 > 8
    assert _decode(block_size=64) == A.KVQ_ERR_SHAPE
    assert _decode(head_dim=80) == A.KVQ_ERR_SHAPE
    assert _decode(workspace_bytes=16) == A.KVQ_ERR_WORKSPACE
    assert _decode(workspace=None) == A.KVQ_ERR_ARG
    assert _decode(workspace=8200) == A.KVQ_ERR_ALIGN
    assert _decode(sparse_v_threshold=-1.0) == A.KVQ_ERR_ARG
    assert _decode(q_stride=100) == A.KVQ_ERR_ARG
    assert _decode(fmt=15, k_scale=-1.0) == A.KVQ_ERR_ARG
    assert _decode(sliding_window=-5) == A.KVQ_ERR_ARG


def _prefill(**over):
    args = dict(q=16, q_dtype=A.KVQ_DTYPE_BF16, q_stride=4096, cu_q=32, max_chunk=64,
                k_cache=4096, v_cache=4096, out=64, out_dtype=A.KVQ_DTYPE_F32, block_tables=128,
                max_blocks_per_seq=4, seq_lens=256, num_seqs=2, num_blocks=8, num_q_heads=32,
                num_kv_heads=8, head_dim=128, block_size=16, k_block_stride_bytes=65536,
                v_block_stride_bytes=65536, sm_scale=0.0, k_scale=1.0, v_scale=1.0,
                sliding_window=0, fmt=0, error_flag=None, stream=None)
    args.update(over)
    with pytest.raises(A.KvqError) as e:
        A.kvq_paged_prefill(**args)
    return e.value.status


def test_prefill_rejects_bad_arguments():
    """Host-side validation, before any launch (these calls never reach CUDA)."""
    assert _prefill(num_q_heads=30) == A.KVQ_ERR_SHAPE
    assert _prefill(num_q_heads=128) == A.KVQ_ERR_SHAPE
    assert _prefill(block_size=64) == A.KVQ_ERR_SHAPE
    assert _prefill(head_dim=80) == A.KVQ_ERR_SHAPE
    assert _prefill(cu_q=None) == A.KVQ_ERR_ARG
    assert _prefill(max_chunk=-1) == A.KVQ_ERR_ARG
    assert _prefill(q_stride=100) == A.KVQ_ERR_ARG
    assert _prefill(k_cache=4104) == A.KVQ_ERR_ALIGN
    assert _prefill(k_block_stride_bytes=1024) == A.KVQ_ERR_ARG
    assert _prefill(fmt=1, k_scale=0.0) == A.KVQ_ERR_ARG
    assert _prefill(fmt=42) == A.KVQ_ERR_FORMAT
    assert _prefill(q_dtype=9) == A.KVQ_ERR_FORMAT


def test_prefill_nothing_to_do_is_ok():
    """No sequences or an empty chunk bound: success without a launch."""
    A.kvq_paged_prefill(q=16, q_dtype=A.KVQ_DTYPE_F32, q_stride=4096, cu_q=32, max_chunk=0,
                        k_cache=4096, v_cache=4096, out=64, out_dtype=A.KVQ_DTYPE_F32,
                        block_tables=128, max_blocks_per_seq=4, seq_lens=256, num_seqs=2,
                        num_blocks=8, num_q_heads=32, num_kv_heads=8, head_dim=128,
                        block_size=16, k_block_stride_bytes=65536, v_block_stride_bytes=65536,
                        sm_scale=0.0, k_scale=1.0, v_scale=1.0, sliding_window=0, fmt=0,
                        error_flag=None, stream=None)


def test_workspace_formula():
    """Partials [num_seqs][nq][kmax][hd + 4] fp32, then int32 partial counts
    [num_seqs][nkv] (16-byte padded); kmax >= 2 (a unit cut once) and never
    above floor((slabs - 1) / 16) + 2 for a sequence of `slabs` 16-token slabs."""
    counts = 32 * 8 * 4
    n = A.kvq_decode_workspace_bytes(32, 32, 8, 128, 16, 256, 0, 0)
    row = 32 * 32 * (128 + 4) * 4
    assert n > counts and (n - counts) % row == 0
    assert 2 <= (n - counts) // row <= (256 - 1) // 16 + 2
    # a 40-token window bounds the slabs at 4, hence kmax at 2
    n = A.kvq_decode_workspace_bytes(32, 32, 8, 128, 16, 256, 40, 0)
    assert n == 2 * row + counts
    assert A.kvq_decode_workspace_bytes(32, 32, 8, 128, 24, 256, 0, 0) == 0


def test_decode_path_rejects_what_the_decode_rejects():
    """kvq_decode_path answers -1 for arguments kvq_paged_decode refuses (no
    device work, so it runs without a GPU)."""
    from quantized_paged_kv_reshape_gb300 import _abi as A, ops
    t4 = ops.fmt_id("turbo4")
    assert A.kvq_decode_path(t4, 96, 8, 16) == -1      # head_dim
    assert A.kvq_decode_path(t4, 128, 0, 16) == -1     # num_kv_heads
    assert A.kvq_decode_path(t4, 128, 8, 12) == -1     # block_size
    assert A.kvq_decode_path(99, 128, 8, 16) == -1     # format
    assert A.kvq_decode_path(t4, 128, 8, 16) in (0, 1)
