"""Sub-byte KV-cache quantization and packed-cache decode attention for GB300 (sm_103a).

The compute path is the CUDA library libkvq.so (C ABI in include/kvq.h); this package only
marshals torch tensors into its calls. Importing the package does not load the library; the
first call does, and raises if it is missing.
"""
from .api import (  # noqa: F401
    KVCache, store, decode_attend, append_decode_attend, attend_workspace_bytes, attend_chunk, debug_scores_i32, debug_attend_scores_i32, row_bytes, cache_plane_bytes,
    PagedKVCache, paged_store, paged_decode_attend, paged_append_decode_attend, paged_attend_workspace_bytes,
    paged_attend_chunk, paged_attend_plan_chunk, append_decode_attend_host, append_decode_attend_host_workspace_bytes,
    paged_append_decode_attend_host, paged_append_decode_attend_host_workspace_bytes,
)
from ._lib import KvqError, LAYOUT_IDS, EXPORTS  # noqa: F401
