"""Streaming chunk attention over a rolling ring KV cache, for GB300 (sm_103a).

Thin Python binding of ``libsab.so`` (C ABI in ``include/sab.h``): argument
marshalling only.  Every step of the computation runs in the library's CUDA
kernels; PyTorch is used only to own device memory and to name streams.
There is no CPU or PyTorch fallback: every call fails loudly when the library
is missing.
"""

from ._abi import (  # noqa: F401
    DEBUG_INJECT_APPEND_SLOT,
    DEBUG_INJECT_KEY_ROW,
    DEBUG_INJECT_WS_TILE,
    ERR_BOUNDS,
    ERR_TIMEOUT,
    GUARD_BYTE,
    KV_BF16,
    KV_FP8_E4M3,
    KV_INT8K_FP8V,
    KVRing,
    RingDesc,
    RopeDesc,
    SabError,
    block_causal_attention,
    block_causal_attention_backward,
    block_causal_attention_backward_workspace,
    block_causal_attention_workspace,
    chunk_attention,
    chunk_attention_dev,
    chunk_attention_fp8mma,
    chunk_attention_noalloc,
    chunk_counter_add,
    debug_bounds_enabled,
    debug_inject_bounds_error,
    guard_watch_begin,
    guard_watch_end,
    chunk_attention_workspace,
    get_last_device_error,
    kv_ring_append,
    kv_ring_append_dev,
    kv_ring_bytes,
    kv_ring_create,
    kv_ring_destroy,
    kv_ring_get_desc,
    kv_ring_get_state,
    kv_ring_layer_ptrs,
    kv_ring_set_sink,
    kv_ring_set_state,
    kv_ring_slot_of,
    library,
    library_path,
    memory_prefix_attention,
    memory_prefix_attention_backward,
    qk_norm_rope,
    selftest_bounded_wait,
    selftest_split_abort,
    status_string,
    version,
)
