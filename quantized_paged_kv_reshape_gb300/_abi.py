"""ctypes binding of libkvq.so: the C ABI of include/kvq.h, same names.

Argument marshalling only.  Every function here forwards to the CUDA
library; there is no fallback.  If the library is missing the first call
raises ``KvqLibraryError`` (build it with ``python -m
quantized_paged_kv_reshape_gb300.build`` or ``__graft_entry__.build()``).
"""

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkvq.so")

KVQ_OK, KVQ_ERR_ARG, KVQ_ERR_FORMAT, KVQ_ERR_SHAPE, KVQ_ERR_ALIGN, KVQ_ERR_WORKSPACE, \
    KVQ_ERR_CUDA = range(7)
KVQ_DTYPE_F32, KVQ_DTYPE_BF16 = 0, 1
KVQ_SIDE_K, KVQ_SIDE_V = 0, 1
KVQ_DEVERR_SLOT, KVQ_DEVERR_BLOCK = 1, 2

FORMAT_NAMES = (
    "bf16", "fp8", "nvfp4", "turbo4", "turbo3", "turbo2", "turbo8",
    "turbo4k_turbo3v", "turbo4k_turbo8v", "turbo3k_turbo8v", "bf16k_turbo4v",
    "bf16k_turbo3v", "fp8k_turbo4v", "fp8k_turbo3v", "bf16k_turbo2v", "fp8k_turbo2v",
)


class KvqLibraryError(RuntimeError):
    pass


class KvqError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{message} (status {status})")
        self.status = status


_lib = None

_SIGS = {
    "kvq_format_from_string": (C.c_int, [C.c_char_p, C.POINTER(C.c_int)]),
    "kvq_format_name": (C.c_char_p, [C.c_int]),
    "kvq_side_format": (C.c_int, [C.c_int, C.c_int]),
    "kvq_side_is_rotated": (C.c_int, [C.c_int, C.c_int]),
    "kvq_block_bytes": (C.c_int64, [C.c_int, C.c_int, C.c_int32, C.c_int32, C.c_int32]),
    "kvq_data_section_bytes": (C.c_int64, [C.c_int, C.c_int, C.c_int32, C.c_int32, C.c_int32]),
    "kvq_codebook": (C.c_int, [C.c_int, C.POINTER(C.c_float), C.POINTER(C.c_float)]),
    "kvq_status_string": (C.c_char_p, [C.c_int]),
    "kvq_last_error": (C.c_char_p, []),
    "kvq_cache_write": (C.c_int, [
        C.c_void_p, C.c_void_p, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p,
        C.c_int32, C.c_int64, C.c_int32, C.c_int32, C.c_int32, C.c_int64, C.c_int64,
        C.c_int64, C.c_int64, C.c_float, C.c_float, C.c_int, C.c_void_p, C.c_void_p]),
    "kvq_decode_path": (C.c_int32, [C.c_int, C.c_int32, C.c_int32, C.c_int32]),
    "kvq_decode_workspace_bytes": (C.c_size_t, [
        C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int]),
    "kvq_paged_decode": (C.c_int, [
        C.c_void_p, C.c_int, C.c_int64, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int,
        C.c_void_p, C.c_int32, C.c_void_p, C.c_int32, C.c_int64, C.c_int32, C.c_int32,
        C.c_int32, C.c_int32, C.c_int64, C.c_int64, C.c_float, C.c_float, C.c_float,
        C.c_int32, C.c_float, C.c_void_p, C.c_size_t, C.c_int, C.c_void_p, C.c_void_p]),
    "kvq_paged_decode_noalloc": (C.c_int, [
        C.c_void_p, C.c_int, C.c_int64, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int,
        C.c_void_p, C.c_int32, C.c_void_p, C.c_int32, C.c_int64, C.c_int32, C.c_int32,
        C.c_int32, C.c_int32, C.c_int64, C.c_int64, C.c_float, C.c_float, C.c_float,
        C.c_int32, C.c_float, C.c_int, C.c_void_p, C.c_void_p]),
    "kvq_paged_prefill": (C.c_int, [
        C.c_void_p, C.c_int, C.c_int64, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p,
        C.c_void_p, C.c_int, C.c_void_p, C.c_int32, C.c_void_p, C.c_int32, C.c_int64,
        C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int64, C.c_int64, C.c_float,
        C.c_float, C.c_float, C.c_int32, C.c_int, C.c_void_p, C.c_void_p]),
}

KVQ_NOALLOC_SCRATCH_BYTES = 8 << 20


def lib():
    """The loaded libkvq.so (loads it on first use)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise KvqLibraryError(
                f"{LIB_PATH} is missing: build the CUDA library first "
                "(python -m quantized_paged_kv_reshape_gb300.build)")
        handle = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def check(status):
    if status != KVQ_OK:
        msg = lib().kvq_last_error().decode() or lib().kvq_status_string(status).decode()
        raise KvqError(status, msg)


def kvq_format_from_string(name):
    out = C.c_int(-1)
    check(lib().kvq_format_from_string(name.encode(), C.byref(out)))
    return out.value


def kvq_format_name(fmt):
    r = lib().kvq_format_name(int(fmt))
    return r.decode() if r is not None else None


def kvq_side_format(fmt, side):
    return lib().kvq_side_format(int(fmt), int(side))


def kvq_side_is_rotated(fmt, side):
    return lib().kvq_side_is_rotated(int(fmt), int(side))


def kvq_block_bytes(fmt, side, block_size, num_kv_heads, head_dim):
    return lib().kvq_block_bytes(int(fmt), int(side), block_size, num_kv_heads, head_dim)


def kvq_data_section_bytes(fmt, side, block_size, num_kv_heads, head_dim):
    return lib().kvq_data_section_bytes(int(fmt), int(side), block_size, num_kv_heads, head_dim)


def kvq_codebook(bits):
    """(levels, thresholds) as lists of fp32 values."""
    n = 1 << bits
    lv = (C.c_float * n)()
    th = (C.c_float * (n - 1))()
    check(lib().kvq_codebook(bits, lv, th))
    return list(lv), list(th)


def kvq_cache_write(key, value, in_dtype, k_cache, v_cache, slot_mapping, num_tokens,
                    num_blocks, num_kv_heads, head_dim, block_size, key_stride, value_stride,
                    k_block_stride_bytes, v_block_stride_bytes, k_scale, v_scale, fmt,
                    error_flag, stream):
    """Raw call with integer device addresses; raises KvqError on a bad status."""
    check(lib().kvq_cache_write(
        key, value, in_dtype, k_cache, v_cache, slot_mapping, num_tokens, num_blocks,
        num_kv_heads, head_dim, block_size, key_stride, value_stride, k_block_stride_bytes,
        v_block_stride_bytes, k_scale, v_scale, int(fmt), error_flag, stream))


def kvq_decode_path(fmt, head_dim, num_kv_heads, block_size):
    return lib().kvq_decode_path(int(fmt), head_dim, num_kv_heads, block_size)


def kvq_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                               max_blocks_per_seq, sliding_window, fmt):
    return lib().kvq_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                            block_size, max_blocks_per_seq, sliding_window,
                                            int(fmt))


def kvq_paged_decode(q, q_dtype, q_stride, k_cache, v_cache, out, out_dtype, block_tables,
                     max_blocks_per_seq, seq_lens, num_seqs, num_blocks, num_q_heads,
                     num_kv_heads, head_dim, block_size, k_block_stride_bytes,
                     v_block_stride_bytes, sm_scale, k_scale, v_scale, sliding_window,
                     sparse_v_threshold, workspace, workspace_bytes, fmt, error_flag, stream):
    """Raw call with integer device addresses; raises KvqError on a bad status."""
    check(lib().kvq_paged_decode(
        q, q_dtype, q_stride, k_cache, v_cache, out, out_dtype, block_tables,
        max_blocks_per_seq, seq_lens, num_seqs, num_blocks, num_q_heads, num_kv_heads,
        head_dim, block_size, k_block_stride_bytes, v_block_stride_bytes, sm_scale, k_scale,
        v_scale, sliding_window, sparse_v_threshold, workspace, workspace_bytes, int(fmt),
        error_flag, stream))


def kvq_paged_decode_noalloc(q, q_dtype, q_stride, k_cache, v_cache, out, out_dtype,
                             block_tables, max_blocks_per_seq, seq_lens, num_seqs, num_blocks,
                             num_q_heads, num_kv_heads, head_dim, block_size,
                             k_block_stride_bytes, v_block_stride_bytes, sm_scale, k_scale,
                             v_scale, sliding_window, sparse_v_threshold, fmt, error_flag,
                             stream):
    """Decode without a workspace argument, for callers that cannot allocate
    device memory: the partials and merge counters use a fixed 8 MiB scratch
    array built into the library (shared by all calls; overlapping calls race)."""
    check(lib().kvq_paged_decode_noalloc(
        q, q_dtype, q_stride, k_cache, v_cache, out, out_dtype, block_tables,
        max_blocks_per_seq, seq_lens, num_seqs, num_blocks, num_q_heads, num_kv_heads,
        head_dim, block_size, k_block_stride_bytes, v_block_stride_bytes, sm_scale, k_scale,
        v_scale, sliding_window, sparse_v_threshold, int(fmt), error_flag, stream))


def kvq_paged_prefill(q, q_dtype, q_stride, cu_q, max_chunk, k_cache, v_cache, out, out_dtype,
                      block_tables, max_blocks_per_seq, seq_lens, num_seqs, num_blocks,
                      num_q_heads, num_kv_heads, head_dim, block_size, k_block_stride_bytes,
                      v_block_stride_bytes, sm_scale, k_scale, v_scale, sliding_window, fmt,
                      error_flag, stream):
    """Raw call with integer device addresses; raises KvqError on a bad status."""
    check(lib().kvq_paged_prefill(
        q, q_dtype, q_stride, cu_q, max_chunk, k_cache, v_cache, out, out_dtype, block_tables,
        max_blocks_per_seq, seq_lens, num_seqs, num_blocks, num_q_heads, num_kv_heads,
        head_dim, block_size, k_block_stride_bytes, v_block_stride_bytes, sm_scale, k_scale,
        v_scale, sliding_window, int(fmt), error_flag, stream))
