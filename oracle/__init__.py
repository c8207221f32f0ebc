"""CPU oracle for the quantized paged KV cache: test infrastructure only.

Nothing in the product path imports, links or calls this package.  Only the
tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference leg of
``bench.py`` use it.  It shares no code with the CUDA library: every number
format, the codebook, the rotation, the packing and the attention are
re-derived here from the formats' definitions, in numpy, fp64 for attention
and fp32 exactly where the stored byte is decided (the write path fixes its
rounding in fp32, see ``cache_write``).

Source pages (cited in each module by page title and section):

* "spark_runtime/kv_cache.rs" (Atlas): the ``KvCacheDtype`` catalogue, the
  per-block byte arithmetic (``block_bytes_dims``) and the section sizes.
* "metrale_model_layers/layers/ops/kv_cache_bf16k_turbov.rs": the
  ``[num_blocks, block_size, num_kv_heads, head_dim]`` layout, code section
  then scale section, launcher arguments of the write and decode kernels.
* "combs_models/kv.rs" (burn): ``attend`` (scores -> softmax -> P.V with the
  ``repeat_kv`` GQA mapping, causal for several query rows) and the paged
  slot arithmetic.

Parity status per function (what pins it) is listed in each module header.
"""

from .formats import (  # noqa: F401
    FORMATS, SIDE_FORMATS, format_from_string, format_name, kv_pair,
    is_wht_rotated, is_asymmetric, block_bytes, data_section_bytes,
)
from .codebook import lloyd_max_gaussian, codebook, distortion  # noqa: F401
from .numformats import (  # noqa: F401
    e4m3_decode, e4m3_encode, bf16_encode, bf16_decode, e2m1_decode, e2m1_encode,
)
from .wht import fwht_f32, wht_f64  # noqa: F401
from .cache_write import (  # noqa: F401
    quantize_rows, quantize_rotated, quantize_nvfp4, pack_codes, unpack_codes, encode_rows_bytes,
    cache_write,
)
from .decode import attend, dequantize_rows, gather_side, paged_decode  # noqa: F401
from .prefill import paged_prefill  # noqa: F401
