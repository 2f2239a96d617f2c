"""TurboQuant-style compressed KV cache for one GB300: encode (append) head
vectors into packed pages and run fused decode attention on them.

The compute lives in ``libtq.so`` (hand-written CUDA for sm_103a, C ABI in
``include/tq.h``); this package is its ctypes binding plus the build script.
"""
from .tq import (  # noqa: F401
    TQ_DEVERR_LENGTH,
    TQ_DEVERR_PAGE_RANGE,
    TQ_DEVERR_SLOT_RANGE,
    TQ_DEVERR_TIMEOUT,
    TQ_KIND_K,
    TQ_KIND_V,
    TQ_STATIC_SCRATCH_BYTES,
    TQError,
    device_codebook,
    kind_codebook,
    load_library,
    tq_decode,
    tq_decode_attn,
    tq_decode_attn_static,
    tq_decode_attn_timed,
    tq_decode_attn_workspace_size,
    tq_encode,
    tq_encode_kv,
    tq_append_window,
    tq_append_window_workspace_size,
    tq_kivi_decode,
    tq_kivi_decode_attn,
    tq_kivi_decode_attn_workspace_size,
    tq_kivi_encode_keys,
    tq_kivi_encode_values,
    tq_kivi_page_layout,
    tq_make_codebook,
    tq_page_layout,
    tq_status_string,
)
