"""PagedAttention decode on GB300 (sm_103a): a C-ABI CUDA library and its binding.

The compute path is libpaged_kv.so (hand-written CUDA for sm_103a, C ABI in
include/paged_kv.h); this package is its thin Python binding plus the
seeded synthetic-workload generators used by the tests and the benchmark.
"""

from .binding import (  # noqa: F401
    BLOCK_SIZE,
    BlockManager,
    LibraryNotBuilt,
    OutOfBlocks,
    PagedKVError,
    check_copy_pairs,
    copy_blocks,
    describe_device_flags,
    device_status,
    copy_blocks_int8,
    paged_attention_decode,
    paged_attention_decode_int8,
    paged_attention_decode_noalloc,
    paged_attention_decode_sliding,
    paged_attention_plan,
    reshape_and_cache,
    reshape_and_cache_int8,
    sliding_workspace_size,
    resolved_partition,
    version,
    workspace_size,
)
