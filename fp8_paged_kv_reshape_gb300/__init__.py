"""FP8 (OCP E4M3) paged KV cache for GB300 (sm_103a).

The compute path is libkvfp8.so (hand-written CUDA, C ABI in include/kvfp8.h);
``binding`` marshals torch tensors into it.  Importing this package requires the
built library and fails loudly without it.
"""
from .binding import (  # noqa: F401
    ABI_FUNCTIONS,
    CACHE_BF16,
    CACHE_E4M3,
    DEV_BAD_BLOCK,
    DEV_BAD_SCALE,
    DEV_BAD_SLOT,
    DEV_TIMEOUT,
    ERR_UNSUPPORTED,
    KvFp8Error,
    LIB,
    LIB_PATH,
    check_scale_host,
    dequant,
    paged_attention_multi,
    paged_attention_multi_mixed,
    paged_attention_multi_workspace_size,
    paged_decode_attention,
    paged_decode_attention_mixed,
    paged_decode_attention_noalloc,
    paged_decode_workspace_size,
    reshape_and_cache,
    reshape_and_cache_mixed,
    rope_reshape_and_cache,
    status_string,
)
