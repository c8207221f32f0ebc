"""Torch-facing wrappers of the C ABI: pointers, sizes and streams from torch
tensors, nothing else.  Every step of the cache write and the decode runs in
libkvq's CUDA kernels; these functions refuse CPU tensors."""

import torch

from . import _abi as A


def fmt_id(fmt):
    return fmt if isinstance(fmt, int) else A.kvq_format_from_string(fmt)


def _dev_ptr(t, name):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (libkvq has no CPU path)")
    return t.data_ptr()


def _dtype_code(t, name):
    if t.dtype == torch.float32:
        return A.KVQ_DTYPE_F32
    if t.dtype == torch.bfloat16:
        return A.KVQ_DTYPE_BF16
    raise ValueError(f"{name} must be float32 or bfloat16")


def _stream_ptr(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def block_bytes(fmt, side, block_size, num_kv_heads, head_dim):
    return A.kvq_block_bytes(fmt_id(fmt), side, block_size, num_kv_heads, head_dim)


def alloc_pool(num_blocks, fmt, side, block_size, num_kv_heads, head_dim, device="cuda",
               stride=None):
    """uint8 [num_blocks, stride] pool for one side; stride rounded up to 16 bytes."""
    b = block_bytes(fmt, side, block_size, num_kv_heads, head_dim)
    stride = stride or (b + 15) // 16 * 16
    return torch.zeros((num_blocks, stride), dtype=torch.uint8, device=device)


def cache_write(key, value, k_cache, v_cache, slot_mapping, fmt, num_kv_heads, head_dim,
                block_size, key_stride=None, value_stride=None, k_scale=1.0, v_scale=1.0,
                num_blocks=None, error_flag=None, stream=None, num_tokens=None):
    """Write rows of ``key``/``value`` (first element of token 0, head 0 at
    ``key.data_ptr()``) into the pools ``k_cache``/``v_cache`` ([num_blocks,
    stride] uint8) at ``slot_mapping`` (int64)."""
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    n = slot_mapping.numel() if num_tokens is None else num_tokens
    kd = _dtype_code(key, "key")
    if _dtype_code(value, "value") != kd:
        raise ValueError("key and value must share a dtype")
    ks = key_stride if key_stride is not None else key.stride(0)
    vs = value_stride if value_stride is not None else value.stride(0)
    nb = k_cache.shape[0] if num_blocks is None else num_blocks
    A.kvq_cache_write(
        _dev_ptr(key, "key"), _dev_ptr(value, "value"), kd, _dev_ptr(k_cache, "k_cache"),
        _dev_ptr(v_cache, "v_cache"), _dev_ptr(slot_mapping, "slot_mapping"), n, nb,
        num_kv_heads, head_dim, block_size, ks, vs, k_cache.stride(0), v_cache.stride(0),
        float(k_scale), float(v_scale), fmt_id(fmt), _dev_ptr(error_flag, "error_flag"),
        _stream_ptr(stream))


def decode_kernel(fmt, head_dim, num_kv_heads, block_size):
    """Name of the decode kernel paged_decode launches on the current device
    for these arguments ("decode_tma_kernel" or "decode_tc_kernel")."""
    p = A.kvq_decode_path(fmt_id(fmt), head_dim, num_kv_heads, block_size)
    if p < 0:
        raise ValueError("arguments the decode rejects")
    return "decode_tma_kernel" if p == 1 else "decode_tc_kernel"


def decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                           max_blocks_per_seq, sliding_window, fmt):
    return A.kvq_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                        block_size, max_blocks_per_seq, sliding_window,
                                        fmt_id(fmt))


def alloc_workspace(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                    max_blocks_per_seq, sliding_window, fmt, device="cuda"):
    n = decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                               max_blocks_per_seq, sliding_window, fmt)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device)


def paged_decode(q, k_cache, v_cache, block_tables, seq_lens, fmt, num_kv_heads,
                 block_size, out=None, out_dtype=torch.float32, sm_scale=0.0, k_scale=1.0,
                 v_scale=1.0, sliding_window=0, sparse_v_threshold=0.0, workspace=None,
                 num_blocks=None, error_flag=None, stream=None):
    """Decode attention: q [num_seqs, num_q_heads, head_dim] (row stride q.stride(0)),
    block_tables int32 [num_seqs, max_blocks], seq_lens int32 [num_seqs]."""
    num_seqs, nq, hd = q.shape
    if q.stride(2) != 1 or q.stride(1) != hd:
        raise ValueError("q heads must be contiguous [.., num_q_heads, head_dim]")
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise ValueError("block_tables and seq_lens must be int32")
    if not block_tables.is_contiguous():
        raise ValueError("block_tables must be contiguous")
    mb = block_tables.shape[1]
    if out is None:
        out = torch.empty((num_seqs, nq, hd), dtype=out_dtype, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(num_seqs, nq, num_kv_heads, hd, block_size, mb,
                                    sliding_window, fmt, device=q.device)
    nb = k_cache.shape[0] if num_blocks is None else num_blocks
    A.kvq_paged_decode(
        _dev_ptr(q, "q"), _dtype_code(q, "q"), q.stride(0), _dev_ptr(k_cache, "k_cache"),
        _dev_ptr(v_cache, "v_cache"), _dev_ptr(out, "out"), _dtype_code(out, "out"),
        _dev_ptr(block_tables, "block_tables"), mb, _dev_ptr(seq_lens, "seq_lens"), num_seqs,
        nb, nq, num_kv_heads, hd, block_size, k_cache.stride(0), v_cache.stride(0),
        float(sm_scale), float(k_scale), float(v_scale), int(sliding_window),
        float(sparse_v_threshold), _dev_ptr(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), fmt_id(fmt),
        _dev_ptr(error_flag, "error_flag"), _stream_ptr(stream))
    return out


def paged_prefill(q, cu_q, max_chunk, k_cache, v_cache, block_tables, seq_lens, fmt,
                  num_kv_heads, block_size, out=None, out_dtype=torch.float32, sm_scale=0.0,
                  k_scale=1.0, v_scale=1.0, sliding_window=0, num_blocks=None, error_flag=None,
                  stream=None):
    """Chunked-prefill attention: q [total_q, num_q_heads, head_dim] (row stride
    q.stride(0)), cu_q int32 [num_seqs + 1] query offsets per sequence, the last
    cu_q[s+1] - cu_q[s] of sequence s's seq_lens[s] cached positions being its
    queries (causal)."""
    total_q, nq, hd = q.shape
    if q.stride(2) != 1 or q.stride(1) != hd:
        raise ValueError("q heads must be contiguous [.., num_q_heads, head_dim]")
    for t, name in ((block_tables, "block_tables"), (seq_lens, "seq_lens"), (cu_q, "cu_q")):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous int32")
    num_seqs = seq_lens.shape[0]
    mb = block_tables.shape[1]
    if out is None:
        out = torch.empty((total_q, nq, hd), dtype=out_dtype, device=q.device)
    nb = k_cache.shape[0] if num_blocks is None else num_blocks
    A.kvq_paged_prefill(
        _dev_ptr(q, "q"), _dtype_code(q, "q"), q.stride(0), _dev_ptr(cu_q, "cu_q"),
        int(max_chunk), _dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"),
        _dev_ptr(out, "out"), _dtype_code(out, "out"), _dev_ptr(block_tables, "block_tables"),
        mb, _dev_ptr(seq_lens, "seq_lens"), num_seqs, nb, nq, num_kv_heads, hd, block_size,
        k_cache.stride(0), v_cache.stride(0), float(sm_scale), float(k_scale), float(v_scale),
        int(sliding_window), fmt_id(fmt), _dev_ptr(error_flag, "error_flag"),
        _stream_ptr(stream))
    return out
