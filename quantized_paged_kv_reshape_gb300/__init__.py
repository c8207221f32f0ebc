"""GB300 quantized paged KV cache: cache write + split-K paged decode.

The compute lives in libkvq.so (CUDA, sm_103a) behind the C ABI of
include/kvq.h; ``_abi`` binds it with the same names and ``ops`` marshals
torch tensors into it.  ``workloads`` draws seeded synthetic inputs.
"""

from . import _abi  # noqa: F401
from ._abi import (  # noqa: F401
    FORMAT_NAMES, KvqError, KvqLibraryError, kvq_block_bytes, kvq_cache_write,
    kvq_codebook, kvq_data_section_bytes, kvq_decode_workspace_bytes,
    kvq_format_from_string, kvq_format_name, kvq_paged_decode, kvq_side_format,
    kvq_side_is_rotated,
)
