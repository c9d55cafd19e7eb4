"""Prefix caching in the host allocator, against the oracle restatement.

The native allocator keys a full block by a 128-bit chained hash of its token
prefix and checks the block's own tokens on a hit; the oracle keys it by the
exact tuple of every token before its end.  Driven with the same calls, the
two must agree bit for bit: every slot (-1 for tokens found stored), cached
count, error kind, table, refcount and free count.  Pins beyond that: a
shared system prompt is stored once; a prefix that differs in one token is
not shared; a block nobody holds is reused by the next matching prompt and
forgotten only when the free stack is empty.
"""
import numpy as np
import pytest

from oracle.allocator import AllocError, OracleAllocator


@pytest.fixture(scope="module")
def native():
    from paged_kv_cache_276_gb300 import build, native
    build.build()
    return native


def _kind(native, code):
    return {native.PKV_ERR_ARG: "arg", native.PKV_ERR_OOM: "oom", native.PKV_ERR_RANGE: "range",
            native.PKV_ERR_SHARED: "shared"}[code]


def test_shared_prompt_is_stored_once(native):
    a = native.BlockAllocator(32, 4)
    prompt = [7, 1, 7, 2, 9, 9, 3, 5, 4, 4, 1]  # 2 full blocks + 3 tokens
    a.seq_add(0)
    s0, c0 = a.seq_append_tokens(0, prompt)
    assert c0 == 0 and (s0 >= 0).all()
    a.seq_add(1)
    s1, c1 = a.seq_append_tokens(1, prompt + [8])
    assert c1 == 8 and (s1[:8] == -1).all() and (s1[8:] >= 0).all()
    t, _ = a.block_table([0, 1], 4)
    assert t[0, :2].tolist() == t[1, :2].tolist() and t[0, 2] != t[1, 2]
    assert a.refcount(int(t[0, 0])) == 2
    a.seq_add(2)
    s2, c2 = a.seq_append_tokens(2, [7, 1, 7, 2, 9, 9, 3, 6])  # second block differs in its last token
    assert c2 == 4 and (s2[:4] == -1).all() and (s2[4:] >= 0).all()
    # nobody holds the prompt any more: still cached, counted free, reused on the next match
    for i in (0, 1, 2):
        a.seq_free(i)
    reg, unheld = a.prefix_cache_stats()  # the prompt's two blocks, sequence 1's third, sequence 2's second
    assert reg == 4 and unheld == 4 and a.num_free() == 32
    a.seq_add(3)
    s3, c3 = a.seq_append_tokens(3, prompt[:8])
    assert c3 == 8 and a.prefix_cache_stats() == (4, 2)
    a.close()


def test_known_blocks_are_forgotten_only_when_the_free_stack_is_empty(native):
    a = native.BlockAllocator(4, 2)
    a.seq_add(0)
    a.seq_append_tokens(0, [1, 2, 3, 4])   # blocks 0, 1, known
    a.seq_free(0)                          # both unheld
    a.seq_add(1)
    a.seq_append(1, 4)                     # takes the two free blocks (2, 3): the known ones survive
    assert a.prefix_cache_stats() == (2, 2)
    a.seq_add(2)
    a.seq_append(2, 2)                     # free stack empty: the block released longest ago goes
    assert a.prefix_cache_stats() == (1, 1)
    a.seq_add(3)
    with pytest.raises(native.PkvError) as e:  # [1, 2] must be stored again and no block is free
        a.seq_append_tokens(3, [1, 2, 3, 4])
    assert e.value.code == native.PKV_ERR_OOM and a.prefix_cache_stats() == (1, 1)
    a.seq_free(1)
    slots, c = a.seq_append_tokens(3, [1, 2, 3, 4])
    # the second block is known by its whole prefix, so it is found although its first block was forgotten
    assert c == 2 and slots[2:].tolist() == [-1, -1] and (slots[:2] >= 0).all()
    a.close()


@pytest.mark.parametrize("seed", [0, 1, 2, 3, 4])
def test_prefix_cache_matches_oracle_bit_exact(native, seed):
    rng = np.random.default_rng(100 + seed)
    NB, bs = [24, 40, 16, 64, 32][seed], [4, 2, 8, 4, 16][seed]
    na, oa = native.BlockAllocator(NB, bs), OracleAllocator(NB, bs)
    prompts = [list(rng.integers(0, 3, size=int(rng.integers(1, 5 * bs)))) for _ in range(3)]
    next_id = 0
    for step in range(500):
        ids = list(oa.seqs)
        op = rng.choice(["add", "tok", "tok", "tok", "plain", "fork", "cow", "free", "free", "swap_out", "swap_in"])
        res_o = res_n = err_o = err_n = None
        if op == "add" or not ids:
            sid = next_id
            next_id += 1
            oa.seq_add(sid)
            na.seq_add(sid)
            op = "tok"
            ids = [sid]
        sid = int(rng.choice(ids))

        def both(fo, fn):
            nonlocal res_o, res_n, err_o, err_n
            try:
                res_o = fo()
            except AllocError as e:
                err_o = e.kind
            try:
                res_n = fn()
            except native.PkvError as e:
                err_n = _kind(native, e.code)

        if op == "tok":
            s = oa.seqs[sid]
            if s["len"] == 0 and rng.random() < 0.7:
                toks = prompts[int(rng.integers(0, 3))] + list(rng.integers(0, 3, size=int(rng.integers(0, 2 * bs))))
            else:
                toks = list(rng.integers(0, 3, size=int(rng.integers(0, 3 * bs))))
            both(lambda: oa.seq_append_tokens(sid, toks),
                 lambda: (lambda r: (r[0].tolist(), r[1]))(na.seq_append_tokens(sid, toks)))
        elif op == "plain":
            n = int(rng.integers(0, 2 * bs))
            both(lambda: oa.seq_append(sid, n), lambda: na.seq_append(sid, n).tolist())
        elif op == "fork":
            child = next_id
            next_id += 1
            both(lambda: oa.seq_fork(sid, child), lambda: na.seq_fork(sid, child))
        elif op == "cow":
            both(lambda: oa.seq_cow(sid, -1), lambda: na.seq_cow(sid, -1))
        elif op == "free":
            both(lambda: oa.seq_free(sid), lambda: na.seq_free(sid))
        elif op == "swap_out":
            both(lambda: oa.seq_swap_out(sid, 256), lambda: na.seq_swap_out(sid, 256).tolist())
        else:
            both(lambda: oa.seq_swap_in(sid, 256), lambda: na.seq_swap_in(sid, 256).tolist())
        assert err_o == err_n, (step, op, err_o, err_n)
        assert res_o == res_n, (step, op, res_o, res_n)
        live = sorted(i for i in oa.seqs if not oa.seqs[i]["swapped"])
        if live:
            t_o, l_o = oa.block_table(live, 256)
            t_n, l_n = na.block_table(live, 256)
            assert t_n.tolist() == t_o and l_n.tolist() == l_o, step
        for i in oa.seqs:
            assert na.seq_len(i) == oa.seqs[i]["len"]
        assert na.num_free() == oa.num_free()
        assert na.prefix_cache_stats() == (len(oa.known), len(oa.unheld))
        for b in range(NB):
            assert na.refcount(b) == oa.refcount[b]
        # invariants: every block is free, held or known-and-unheld, exactly once
        held = {b for i in oa.seqs for b in oa.seqs[i]["blocks"]}
        assert len(oa.free) + len(oa.unheld) + len(held) == NB
        assert not (set(oa.free) & set(oa.unheld)) and not (held & set(oa.unheld))
    na.close()
