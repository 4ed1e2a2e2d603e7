"""Causal scaled dot-product attention (prefill and KV-cache decode) on one GB300.

Python face of libattn.so (include/attn.h).  The functions take CUDA torch
tensors and call the C ABI; all computation happens in the library's sm_103a
kernels.  Build the library first with ``transformer_causal_attention_gb300.build.build()``.
"""
from ._binding import (  # noqa: F401
    ATTN_BF16,
    ATTN_F32,
    ATTN_ROPE_HALF,
    AttnError,
    LIB_PATH,
    check_wait_timeout,
    decode,
    decode_window,
    decode_workspace_size,
    kv_append,
    prefill_chunk,
    prefill_mla,
    prefill_window,
    device_status,
    launch_count,
    load,
    prefill,
    rope,
    set_wait_limit_ns,
)
