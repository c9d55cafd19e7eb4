"""Plain loop restatements of the two cache-mutating operations.

TEST INFRASTRUCTURE ONLY (tests, smoke check, benchmark CPU leg).  No code is
shared with the CUDA path.

* ``write``: appending a token's key and value into the slot the allocator gave
  it.  The pages say the cache grows by one token per decode step and a
  request grows by allocating further blocks (x321.org "The serving bottleneck
  is not just FLOPs", sections "First understand what the KV cache is storing"
  and "PagedAttention borrows an operating-system trick").  The slot encoding
  is a reading of ours: slot = physical_block * block_size + offset, and a
  negative slot means "no token here, skip".
* ``block_copy``: the copy that materialises copy-on-write of a shared block
  (praveentn.live "PagedAttention KV-cache constraint", section "What the
  change bought": blocks of an identical prefix are shared with copy-on-write).
* ``swap_out`` / ``swap_in``: whole blocks to and from a host buffer, the data
  side of swapping blocks out under memory pressure (same page, "What it
  cost").

Arrays are numpy; bf16 values are carried as their uint16 bit patterns, so
every operation here is an exact bit copy.
"""
from __future__ import annotations

import numpy as np


def write(k, v, slot_mapping, k_cache, v_cache, block_size):
    """In place: for each token t with slot s >= 0, cache[s // bs, :, s % bs, :] = kv[t].

    k, v: [T, Hkv, d]; slot_mapping: [T] int64; caches: [NB, Hkv, bs, d].
    Raises IndexError for a slot past the end of the pool.
    """
    num_blocks = k_cache.shape[0]
    for t in range(len(slot_mapping)):
        s = int(slot_mapping[t])
        if s < 0:
            continue
        block, offset = divmod(s, block_size)
        if block >= num_blocks:
            raise IndexError(f"slot {s} is outside a pool of {num_blocks} blocks")
        for h in range(k_cache.shape[1]):
            k_cache[block, h, offset, :] = k[t, h, :]
            v_cache[block, h, offset, :] = v[t, h, :]


def block_copy(k_cache, v_cache, src_dst_pairs):
    """In place: for each (src, dst) pair, every head and slot of block dst := block src."""
    num_blocks = k_cache.shape[0]
    for src, dst in np.asarray(src_dst_pairs).reshape(-1, 2):
        src, dst = int(src), int(dst)
        if not (0 <= src < num_blocks and 0 <= dst < num_blocks):
            raise IndexError(f"pair ({src}, {dst}) is outside a pool of {num_blocks} blocks")
        k_cache[dst] = k_cache[src]
        v_cache[dst] = v_cache[src]


def swap_out(k_cache, v_cache, block_ids):
    """Host copies of the listed blocks: returns (k, v), each [n, Hkv, bs, d]."""
    num_blocks = k_cache.shape[0]
    ids = [int(b) for b in np.asarray(block_ids).reshape(-1)]
    k = np.empty((len(ids),) + k_cache.shape[1:], dtype=k_cache.dtype)
    v = np.empty_like(k)
    for i, b in enumerate(ids):
        if not 0 <= b < num_blocks:
            raise IndexError(f"block {b} is outside a pool of {num_blocks} blocks")
        k[i] = k_cache[b]
        v[i] = v_cache[b]
    return k, v


def swap_in(k, v, block_ids, k_cache, v_cache):
    """In place: block block_ids[i] of the caches := k[i], v[i]."""
    num_blocks = k_cache.shape[0]
    for i, b in enumerate(int(x) for x in np.asarray(block_ids).reshape(-1)):
        if not 0 <= b < num_blocks:
            raise IndexError(f"block {b} is outside a pool of {num_blocks} blocks")
        k_cache[b] = k[i]
        v_cache[b] = v[i]
