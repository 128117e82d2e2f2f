"""Quantized paged KV store for GB300: Python binding of the C ABI (include/kvq.h).

Every call marshals torch tensors (device memory) and the current CUDA stream
into the C entry point of the same name in libkvq.so; all compute runs in the
library's CUDA kernels.  Importing this package loads libkvq.so and raises if
it is missing: there is no fallback implementation.
"""
from ._binding import (  # noqa: F401
    FORMATS, KVQError, KVQCache, kvq_bytes_per_token, kvq_cache_layout, kvq_calibrate_scales,
    kvq_create_cache, kvq_decode_attention, kvq_decode_attention_fp8q, kvq_decode_attention_noalloc,
    kvq_decode_workspace_size, kvq_dequantize, kvq_destroy_cache, kvq_extend_attention,
    kvq_extend_workspace_size,
    kvq_format_from_name,
    kvq_format_name, kvq_get_device_error, kvq_last_error_string, kvq_layer_head_scales,
    kvq_layer_scales, kvq_quantize_and_store, kvq_quantize_and_store_per_head, kvq_quantize_query,
    library_path, lib)
