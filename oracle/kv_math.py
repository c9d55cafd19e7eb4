"""Block-count and byte arithmetic of a paged KV cache, written from the pages.

TEST INFRASTRUCTURE ONLY.

* blocks needed by a sequence of ``length`` tokens with ``block`` tokens per
  block, and the unused slots in its last block (chenhuiyu.github.io "A
  complete explanation from first principles", sections "Calculate a
  block-allocation example" and "Logical continuity, physical flexibility");
* KV bytes per token = layers * 2 * KV heads * head dim * bytes per element,
  the 2 being one cache for keys and one for values (x321.org "The serving
  bottleneck is not just FLOPs", section "First understand what the KV cache
  is storing").
"""
from __future__ import annotations


def blocks_needed(length: int, block: int) -> int:
    """Fewest whole blocks whose slots hold ``length`` tokens."""
    if length < 0 or block < 1:
        raise ValueError("length must be >= 0 and block >= 1")
    return -(-length // block)


def unused_slots(length: int, block: int) -> int:
    """Slots allocated but not holding a token (tail waste inside the last block)."""
    return blocks_needed(length, block) * block - length


def allocated_tokens(lengths, block: int):
    """Token capacity each sequence is given when every sequence allocates on its own."""
    return [blocks_needed(n, block) * block for n in lengths]


def slack_tokens(lengths, block: int) -> int:
    """Total unused token slots over independently allocated sequences."""
    return sum(allocated_tokens(lengths, block)) - sum(lengths)


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, bytes_per_elem: int) -> int:
    """Cache bytes one token costs: a key and a value row per KV head per layer."""
    return layers * 2 * kv_heads * head_dim * bytes_per_elem


def kv_bytes_read(seq_lens, kv_heads: int, head_dim: int, bytes_per_elem: int = 2) -> int:
    """Bytes of valid K and V rows one decode over these sequences must read (one layer)."""
    return sum(int(n) for n in seq_lens) * kv_bytes_per_token(1, kv_heads, head_dim, bytes_per_elem)
