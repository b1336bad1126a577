"""Paged KV-cache decode attention for GB300 (sm_103a).

The computation lives in ``libpagedattn.so`` (C ABI in ``include/pagedattn.h``);
``pagedattn`` is its Python binding.
"""
from .pagedattn import (  # noqa: F401
    PA_BFLOAT16,
    PA_FLOAT16,
    PA_FLOAT32,
    PA_ERR_CAPACITY,
    BlockManager,
    PagedAttnError,
    alloc_prefill_workspace,
    alloc_workspace,
    bad_index_count,
    copy_blocks,
    decode,
    decode_append,
    decode_no_alloc,
    decode_partition_tokens,
    decode_workspace_bytes,
    last_error,
    load_library,
    prefill,
    prefill_workspace_bytes,
    no_alloc_scratch_bytes,
    reshape_and_cache,
    testing_prefill_stalled,
    wait_timeout_count,
)
