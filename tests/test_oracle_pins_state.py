"""Pins of the oracle's swap and prefix-cache restatements (no GPU, no native library).

Every expected value below is written out by hand from the rules the oracle
restates, not computed by the oracle or by the native allocator:

* swap_out / swap_in copy whole blocks between the pool and host buffers
  (praveentn.live "PagedAttention KV-cache constraint", "What it cost": under
  memory pressure blocks are swapped out to host memory and back);
* a swapped-out sequence keeps its length, gives its blocks back like a free
  does (a block another sequence still holds stays resident) and returns with
  fresh private blocks (same page, "What the change bought" for the sharing);
* a full block is found again only by an exact match of every token before
  its end (chenhuiyu.github.io "A complete explanation from first
  principles", "Prefix reuse requires compatible computation"; x321.org "The
  serving bottleneck is not just FLOPs", prefix caching).

Allocator policy readings the expectations rely on: free blocks are a LIFO
stack that hands out block 0 first, released blocks are pushed back in
logical order, and a known block nobody holds is reused (forgotten) only when
the free stack is empty, the one released longest ago first.

A wrong block index, LIFO swapped for FIFO (on the free stack or on the
forgetting order), a cached count off by a block, or a swap that forgets to
give up or take back a block each fails at least one assertion here.
"""
import numpy as np
import pytest

from oracle import cache_ops
from oracle.allocator import AllocError, OracleAllocator

NB, HKV, BS, D = 6, 2, 2, 3


def numbered_pool(offset):
    """cache[b, h, s, x] = offset + 1000 b + 100 h + 10 s + x (distinct per element)."""
    c = np.zeros((NB, HKV, BS, D), dtype=np.uint16)
    for b in range(NB):
        for h in range(HKV):
            for s in range(BS):
                for x in range(D):
                    c[b, h, s, x] = offset + 1000 * b + 100 * h + 10 * s + x
    return c


# ---------------------------------------------------------------- data side of a swap
def test_swap_out_returns_the_listed_blocks_in_list_order():
    kc, vc = numbered_pool(0), numbered_pool(30000)
    k, v = cache_ops.swap_out(kc, vc, [3, 0, 5])
    assert k.shape == (3, HKV, BS, D) and v.shape == (3, HKV, BS, D)
    # host row 0 is block 3, row 1 block 0, row 2 block 5
    assert k[0].reshape(-1).tolist() == [3000, 3001, 3002, 3010, 3011, 3012, 3100, 3101, 3102, 3110, 3111, 3112]
    assert k[1].reshape(-1).tolist() == [0, 1, 2, 10, 11, 12, 100, 101, 102, 110, 111, 112]
    assert k[2].reshape(-1).tolist() == [5000, 5001, 5002, 5010, 5011, 5012, 5100, 5101, 5102, 5110, 5111, 5112]
    assert v[0, 1, 1, 2] == 33112 and v[1, 0, 0, 0] == 30000 and v[2, 0, 1, 1] == 35011
    # the pool itself is not changed
    assert np.array_equal(kc, numbered_pool(0)) and np.array_equal(vc, numbered_pool(30000))


def test_swap_in_writes_host_row_i_into_block_ids_i_only():
    kc, vc = numbered_pool(0), numbered_pool(30000)
    k, v = cache_ops.swap_out(kc, vc, [3, 0, 5])
    cache_ops.swap_in(k, v, [1, 4, 2], kc, vc)  # old block 3 -> 1, old 0 -> 4, old 5 -> 2
    assert kc[1, 0, 0, 0] == 3000 and kc[1, 1, 1, 2] == 3112
    assert kc[4, 0, 0, 0] == 0 and kc[4, 1, 0, 1] == 101
    assert kc[2, 0, 1, 0] == 5010 and vc[2, 1, 1, 2] == 35112
    # blocks not listed keep their own values
    for b in (0, 3, 5):
        assert kc[b, 0, 0, 0] == 1000 * b and vc[b, 1, 1, 1] == 30000 + 1000 * b + 111


def test_swap_rejects_ids_outside_the_pool():
    kc, vc = numbered_pool(0), numbered_pool(30000)
    with pytest.raises(IndexError):
        cache_ops.swap_out(kc, vc, [0, NB])
    k, v = cache_ops.swap_out(kc, vc, [0])
    with pytest.raises(IndexError):
        cache_ops.swap_in(k, v, [-1], kc, vc)


# ---------------------------------------------------------------- allocator side of a swap
def test_swap_out_keeps_shared_blocks_and_swap_in_takes_fresh_ones_lifo():
    a = OracleAllocator(8, 16)
    a.seq_add(1)
    assert a.seq_append(1, 40) == list(range(40))  # blocks 0, 1, 2 (slots 0..39)
    a.seq_fork(1, 2)
    assert a.seq_swap_out(1, 8) == [0, 1, 2]
    assert a.seqs[1]["len"] == 40 and a.num_free() == 5  # sequence 2 still holds all three
    assert [a.refcount[b] for b in (0, 1, 2)] == [1, 1, 1]
    refused = (lambda: a.seq_append(1, 1), lambda: a.seq_fork(1, 3), lambda: a.seq_cow(1),
               lambda: a.block_table([1], 8), lambda: a.seq_swap_out(1, 8))
    for call in refused:
        with pytest.raises(AllocError) as e:
            call()
        assert e.value.kind == "arg"
    a.seq_free(2)
    # the free stack (top last) is now [7, 6, 5, 4, 3, 0, 1, 2]
    assert a.free == [7, 6, 5, 4, 3, 0, 1, 2] and a.num_free() == 8
    with pytest.raises(AllocError) as e:
        a.seq_swap_in(1, 2)  # 40 tokens need 3 blocks
    assert e.value.kind == "range" and a.num_free() == 8
    assert a.seq_swap_in(1, 8) == [2, 1, 0]
    table, lens = a.block_table([1], 4)
    assert table == [[2, 1, 0, -1]] and lens == [40] and a.num_free() == 5
    with pytest.raises(AllocError) as e:
        a.seq_swap_in(1, 8)  # resident again
    assert e.value.kind == "arg"
    assert a.seq_append(1, 1) == [0 * 16 + 8]  # token 40 goes to slot 8 of logical block 2 (physical 0)


def test_swap_in_is_refused_while_the_pool_is_full_and_changes_nothing():
    b = OracleAllocator(2, 16)
    b.seq_add(7)
    assert b.seq_append(7, 20) == list(range(20))  # blocks [0, 1]
    assert b.seq_swap_out(7, 4) == [0, 1] and b.free == [0, 1]
    b.seq_add(8)
    assert b.seq_append(8, 17) == list(range(16, 32)) + [0]  # blocks [1, 0]
    with pytest.raises(AllocError) as e:
        b.seq_swap_in(7, 4)
    assert e.value.kind == "oom" and b.seqs[7]["swapped"] and b.num_free() == 0
    b.seq_free(8)
    assert b.free == [1, 0]
    assert b.seq_swap_in(7, 4) == [0, 1]


def test_swap_in_ends_prefix_tracking():
    a = OracleAllocator(8, 2)
    a.seq_add(0)
    a.seq_append_tokens(0, [5, 6, 7, 8])  # blocks 0, 1 known by their prefixes
    a.seq_swap_out(0, 4)                  # both unheld, still known
    assert len(a.known) == 2 and a.unheld == [0, 1]
    assert a.seq_swap_in(0, 4) == [2, 3]  # fresh blocks from the free stack, not the known ones
    a.seq_add(1)
    assert a.seq_append_tokens(1, [5, 6, 7, 8]) == ([-1, -1, -1, -1], 4)  # the old blocks are found
    assert a.seq_append_tokens(0, [9, 9]) == ([8, 9], 0)  # sequence 0 no longer tracks its tokens
    assert len(a.known) == 2


# ---------------------------------------------------------------- prefix cache
def test_shared_prompt_is_stored_once_in_the_oracle():
    a = OracleAllocator(32, 4)
    prompt = [7, 1, 7, 2, 9, 9, 3, 5, 4, 4, 1]  # 2 full blocks + 3 tokens
    a.seq_add(0)
    assert a.seq_append_tokens(0, prompt) == (list(range(11)), 0)  # blocks 0, 1, 2
    a.seq_add(1)
    # both full blocks are found; the third (now full with the 12th token) is new: block 3
    assert a.seq_append_tokens(1, prompt + [8]) == ([-1] * 8 + [12, 13, 14, 15], 8)
    table, _ = a.block_table([0, 1], 4)
    assert table == [[0, 1, 2, -1], [0, 1, 3, -1]] and a.refcount[0] == 2 and a.refcount[1] == 2
    a.seq_add(2)
    # the second block differs in its last token: only the first is found; block 4 is new
    assert a.seq_append_tokens(2, [7, 1, 7, 2, 9, 9, 3, 6]) == ([-1] * 4 + [16, 17, 18, 19], 4)
    for i in (0, 1, 2):
        a.seq_free(i)
    # known: the prompt's two blocks, sequence 1's third, sequence 2's second; the
    # partial block 2 was never known and went back to the free stack
    assert sorted(a.known.values()) == [0, 1, 3, 4] and a.unheld == [1, 3, 0, 4]
    assert a.free[-1] == 2 and a.num_free() == 32
    a.seq_add(3)
    assert a.seq_append_tokens(3, prompt[:8]) == ([-1] * 8, 8)
    assert a.unheld == [3, 4] and a.refcount[0] == 1 and a.refcount[1] == 1


def test_known_blocks_are_forgotten_oldest_first_and_only_when_the_stack_is_empty():
    a = OracleAllocator(4, 2)
    a.seq_add(0)
    assert a.seq_append_tokens(0, [1, 2, 3, 4]) == ([0, 1, 2, 3], 0)
    a.seq_free(0)
    assert a.unheld == [0, 1] and a.free == [3, 2]
    a.seq_add(1)
    assert a.seq_append(1, 4) == [4, 5, 6, 7]  # blocks 2 and 3 from the stack; the known ones survive
    assert len(a.known) == 2 and a.unheld == [0, 1]
    a.seq_add(2)
    assert a.seq_append(2, 2) == [0, 1]  # stack empty: block 0, released first, is forgotten and reused
    assert list(a.known.values()) == [1] and a.unheld == [1]
    a.seq_add(3)
    with pytest.raises(AllocError) as e:  # (1, 2) must be stored again and no block is free
        a.seq_append_tokens(3, [1, 2, 3, 4])
    assert e.value.kind == "oom" and a.unheld == [1] and a.seqs[3]["len"] == 0
    a.seq_free(1)
    assert a.free == [2, 3]
    # block 1 is known by its whole prefix (1, 2, 3, 4), so it is found although
    # the block before it was forgotten; the first block is stored again in block 3
    assert a.seq_append_tokens(3, [1, 2, 3, 4]) == ([6, 7, -1, -1], 2)
    assert a.block_table([3], 2) == ([[3, 1]], [4]) and a.unheld == []


def test_prefix_match_must_be_exact_and_whole():
    a = OracleAllocator(16, 2)
    a.seq_add(0)
    a.seq_append_tokens(0, [1, 2, 3, 4, 5, 6])
    a.seq_add(1)
    # same second block (3, 4) after a different first block: not a match
    assert a.seq_append_tokens(1, [9, 2, 3, 4]) == ([6, 7, 8, 9], 0)
    a.seq_add(2)
    # a match of the first block only, then the tokens split over two calls
    assert a.seq_append_tokens(2, [1, 2, 3]) == ([-1, -1, 10], 2)
    assert a.seq_append_tokens(2, [4, 5, 6]) == ([11, -1, -1], 2)  # (5, 6) is found after (1, 2, 3, 4)
    assert a.block_table([2], 4)[0] == [[0, 5, 2, -1]]
