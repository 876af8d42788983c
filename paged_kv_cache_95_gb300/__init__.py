"""GB300-native paged KV-cache attention (decode, split-KV merge, causal chunked prefill).

The compute lives in ``libpagedkv.so`` (hand-written sm_103a CUDA kernels behind
the C ABI of include/pagedkv.h); :mod:`.pagedkv` is its ctypes binding and
:mod:`.workloads` builds the seeded synthetic inputs.
"""
from .pagedkv import (  # noqa: F401
    BLOCK_SIZE,
    HEAD_DIM,
    PKV_DTYPE_BF16,
    PKV_DTYPE_FLOAT32,
    PKV_DTYPE_FP8_E4M3,
    PKV_STATUS_BAD_BLOCK_ID,
    PKV_STATUS_BAD_CONTEXT_LEN,
    PKV_STATUS_BAD_Q_LEN,
    PKV_STATUS_TIMEOUT,
    BlockManager,
    CacheDesc,
    PagedKVError,
    cache_desc,
    kv_copy_blocks,
    kv_reshape_and_cache,
    kv_reshape_and_cache_fp8,
    load_library,
    paged_attention_decode,
    paged_attention_decode_append,
    paged_attention_decode_static_scratch,
    paged_attention_prefill_chunk,
    paged_attention_prefill_workspace_size,
    paged_attention_verify,
    paged_attention_workspace_size,
    status_string,
    version,
)
