"""GB300-native paged MQA/GQA decode attention.

The computation lives in the CUDA library ``libpaged_decode_attn.so``
(C ABI: ``include/paged_decode_attn.h``); this package is its Python binding
(``PagedDecodeAttention``, ``merge``, ``plan``, ``rope_kv_write``), the in-tree build script and
the seeded synthetic workload generators. Importing the package does not load
the CUDA library; the first call does, and raises if it is missing.
"""
from ._binding import (ABI_VERSION, EXPORTS, PDA_BF16, PDA_EALIAS, PDA_ECUDA, PDA_EDEVICE,
                       PDA_EINVAL, PDA_ENOMEM, PDA_EUNSUPPORTED, PDA_F32, PDA_FP16, PDA_OK,
                       Config, PagedDecodeAttention, PDAError, load_library, make_config, merge,
                       plan, rope_kv_write, copy_blocks, gather_kv, scatter_kv, remap_table)

__all__ = ["ABI_VERSION", "EXPORTS", "PDA_BF16", "PDA_EALIAS", "PDA_ECUDA", "PDA_EDEVICE",
           "PDA_EINVAL", "PDA_ENOMEM", "PDA_EUNSUPPORTED", "PDA_F32", "PDA_FP16", "PDA_OK",
           "Config", "PagedDecodeAttention", "PDAError", "load_library", "make_config", "merge",
           "plan", "rope_kv_write", "copy_blocks", "gather_kv", "scatter_kv", "remap_table"]
