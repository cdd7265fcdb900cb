"""GB300-native paged KV-cache decode attention.

The compute path is a C-ABI CUDA library (``include/pagedattn.h``) built for
sm_103a; this package holds its thin Python binding plus the host-side pieces
that feed it: the block manager, byte accounting and the seeded workloads.

    from paged_kv_cache_29_gb300 import pa_reshape_and_cache, pa_decode
"""
from ._binding import (  # noqa: F401
    KERNELS,
    PA_DEVERR_BLOCK_ID,
    PA_DEVERR_CONTEXT,
    PA_DEVERR_SLOT,
    PA_DEVERR_TIMEOUT,
    PagedAttentionError,
    pa_copy_blocks,
    pa_decode,
    pa_decode_fp8,
    pa_decode_int8,
    pa_decode_multi,
    pa_decode_noalloc,
    pa_append_decode,
    pa_append_decode_fp8,
    pa_append_decode_int8,
    pa_decode_window,
    pa_decode_workspace_size,
    pa_decode_workspace_size_multi,
    pa_reshape_and_cache,
    pa_reshape_and_cache_fp8,
    pa_reshape_and_cache_int8,
    pa_default_partition_size,
    pa_status_string,
    pa_version,
)

__all__ = ["pa_reshape_and_cache", "pa_reshape_and_cache_int8", "pa_decode_int8", "pa_decode_window", "pa_decode_multi", "pa_reshape_and_cache_fp8", "pa_decode_fp8", "pa_copy_blocks", "pa_decode", "pa_decode_noalloc", "pa_append_decode", "pa_append_decode_fp8", "pa_append_decode_int8", "pa_decode_workspace_size", "pa_decode_workspace_size_multi", "pa_status_string",
           "pa_default_partition_size", "pa_version", "PagedAttentionError", "KERNELS", "block_manager", "workloads",
           "accounting"]
