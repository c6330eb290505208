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
    paged_attention_decode,
    reshape_and_cache,
    resolved_partition,
    version,
    workspace_size,
)
