"""GB300 (sm_103a) paged KV cache: paged attention decode, slot write, copy-on-write
block copy and a host block allocator, behind the C ABI in include/pkv.h.

The compute path is libpkv.so (hand-written CUDA); this package only binds it.
"""
from .native import (  # noqa: F401
    BlockAllocator,
    PkvError,
    paged_attention_decode,
    paged_attention_workspace_size,
    pkv_block_copy,
    pkv_write,
)
