"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test checks the oracle against a value the pages print, a closed form, an
invariant, or a library routine that the special case reduces to (torch's
scaled_dot_product_attention on a contiguous cache), chosen so that a dropped
term, a wrong sign or index, a transposed operand, a wrong scale or a wrong
head grouping fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

from conftest import read_golden
from oracle import attention as OA
from oracle import cache_ops, kv_math
from oracle.allocator import AllocError, OracleAllocator


def bf16(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def randn_bf16(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16)


def paged_from_contiguous(K, V, placement, num_blocks, bs, seed=0):
    """Scatter contiguous per-sequence K/V [B][Hkv][L][d] into a random-filled pool.

    placement[i] lists the physical block of each logical block of sequence i.
    Written independently of the oracle: plain slicing assignments.
    """
    Hkv, _, d = K[0].shape
    kc = randn_bf16((num_blocks, Hkv, bs, d), seed + 11) * 7  # junk elsewhere
    vc = randn_bf16((num_blocks, Hkv, bs, d), seed + 12) * 7
    for i in range(len(placement)):
        L = K[i].shape[1]
        for j, phys in enumerate(placement[i]):
            lo, hi = j * bs, min(L, (j + 1) * bs)
            if lo >= hi:
                continue
            kc[phys, :, : hi - lo, :] = K[i][:, lo:hi, :]
            vc[phys, :, : hi - lo, :] = V[i][:, lo:hi, :]
    return kc, vc


def sdpa_ref(q, K, V, scale=None, mask=None):
    """torch SDPA in fp64 on one sequence: q [Hq, R, d], K/V [Hkv, L, d] (GQA by repeat)."""
    Hq, Hkv = q.shape[0], K.shape[0]
    Kr = K.double().repeat_interleave(Hq // Hkv, dim=0)
    Vr = V.double().repeat_interleave(Hq // Hkv, dim=0)
    return torch.nn.functional.scaled_dot_product_attention(
        q.double().unsqueeze(0), Kr.unsqueeze(0), Vr.unsqueeze(0), attn_mask=mask, scale=scale)[0]


# ---------------------------------------------------------------- page values
def test_block_counts_match_pages():
    for length, block, blocks, capacity, unused, used_last, _origin in read_golden("block_counts.txt"):
        length, block = int(length), int(block)
        assert kv_math.blocks_needed(length, block) == int(blocks)
        assert kv_math.blocks_needed(length, block) * block == int(capacity)
        assert kv_math.unused_slots(length, block) == int(unused)
        # the allocator oracle hands out the same count and fills the last block as stated
        a = OracleAllocator(16, block)
        a.seq_add(0)
        slots = a.seq_append(0, length)
        assert len(a.seqs[0]["blocks"]) == int(blocks)
        last = a.seqs[0]["blocks"][-1]
        assert sum(1 for s in slots if s // block == last) == int(used_last)
        assert a.num_free() == 16 - int(blocks)


def test_allocation_example_matches_pages():
    rows = {r[0]: r[1:] for r in read_golden("allocation_example.txt")}
    block = int(rows["block"][0])
    lengths = [int(x) for x in rows["lengths"]]
    assert kv_math.allocated_tokens(lengths, block) == [int(x) for x in rows["allocated"]]
    assert kv_math.slack_tokens(lengths, block) == int(rows["slack"][0])
    a = OracleAllocator(64, block)
    for i, n in enumerate(lengths):
        a.seq_add(i)
        a.seq_append(i, n)
    assert [len(a.seqs[i]["blocks"]) * block for i in range(3)] == [int(x) for x in rows["allocated"]]


def test_kv_bytes_match_pages():
    rows = {r[0]: int(r[1]) for r in read_golden("kv_bytes.txt")}
    per_tok = kv_math.kv_bytes_per_token(rows["layers"], rows["kv_heads"], rows["head_dim"], rows["bytes_per_elem"])
    assert per_tok == rows["bytes_per_token"] == 128 * 1024
    assert per_tok * rows["tokens"] == rows["bytes_per_sequence"] == 1 << 30
    # one layer of the same cache, as the decode kernel reads it
    assert kv_math.kv_bytes_read([rows["tokens"]], rows["kv_heads"], rows["head_dim"]) * rows["layers"] == 1 << 30


def test_page_block_table_example_equals_contiguous():
    """Request A's blocks at physical slots [3, 6, 5, 1] of a 7-slot pool give the contiguous result."""
    rows = {r[0]: r[1:] for r in read_golden("block_table_example.txt")}
    pool = int(rows["pool"][0])
    table_a = [int(x) for x in rows["A"]]
    assert sorted(table_a + [int(rows["B1"][0]), int(rows["C2"][0]), int(rows["free"][0])]) == list(range(pool))
    bs, d, Hq, Hkv = 4, 16, 2, 1  # d a power of 4: 1/sqrt(d) is exact in fp32
    L = 14  # four logical blocks, the last one partly filled
    K = randn_bf16((Hkv, L, d), 1)
    V = randn_bf16((Hkv, L, d), 2)
    q = randn_bf16((1, 1, Hq, d), 3)
    kc, vc = paged_from_contiguous([K], [V], [table_a], pool, bs)
    tables = np.array([table_a], dtype=np.int32)
    out = OA.paged_attention(q, kc, vc, tables, [L], num_q_heads=Hq, num_kv_heads=Hkv,
                             head_dim=d, block_size=bs, scale=1 / math.sqrt(d))
    ref = sdpa_ref(q[0].permute(1, 0, 2), K, V)  # [Hq, 1, d]
    np.testing.assert_allclose(out[0, 0], ref[:, 0].numpy(), rtol=1e-12, atol=1e-12)


# ------------------------------------------------------ library special cases
# head dims are powers of 4 so that the fp32 scale 1/sqrt(d) equals SDPA's default exactly
@pytest.mark.parametrize("d,bs,Hq,Hkv,lens", [
    (64, 16, 4, 2, [17, 33, 64]),     # the tiny workload's shape
    (4, 4, 6, 3, [1, 5, 9, 40]),
    (16, 32, 8, 1, [31, 32, 33]),
])
def test_oracle_matches_sdpa_on_contiguous(d, bs, Hq, Hkv, lens):
    rng = np.random.default_rng(d + bs + Hq)
    nblk = [-(-n // bs) for n in lens]
    NB = sum(nblk) + 5
    perm = rng.permutation(NB)
    placement, pos = [], 0
    for c in nblk:
        placement.append([int(x) for x in perm[pos:pos + c]])
        pos += c
    K = [randn_bf16((Hkv, n, d), 100 + i) for i, n in enumerate(lens)]
    V = [randn_bf16((Hkv, n, d), 200 + i) for i, n in enumerate(lens)]
    q = randn_bf16((len(lens), 1, Hq, d), 300)
    kc, vc = paged_from_contiguous(K, V, placement, NB, bs)
    tables = np.full((len(lens), max(nblk) + 2), -1, dtype=np.int32)
    for i, p in enumerate(placement):
        tables[i, :len(p)] = p
    out = OA.paged_attention(q, kc, vc, tables, lens, num_q_heads=Hq, num_kv_heads=Hkv,
                             head_dim=d, block_size=bs, scale=1 / math.sqrt(d))
    for i in range(len(lens)):
        ref = sdpa_ref(q[i].permute(1, 0, 2), K[i], V[i])  # default scale 1/sqrt(d)
        np.testing.assert_allclose(out[i, 0], ref[:, 0].numpy(), rtol=1e-12, atol=1e-12)


def test_chunked_query_matches_masked_sdpa():
    d, bs, Hq, Hkv, R = 16, 8, 4, 2, 5
    lens = [5, 12, 29]
    nblk = [-(-n // bs) for n in lens]
    placement, pos = [], 0
    for c in nblk:
        placement.append(list(range(pos + c - 1, pos - 1, -1)))  # reversed placement
        pos += c
    K = [randn_bf16((Hkv, n, d), 10 + i) for i, n in enumerate(lens)]
    V = [randn_bf16((Hkv, n, d), 20 + i) for i, n in enumerate(lens)]
    q = randn_bf16((len(lens), R, Hq, d), 30)
    kc, vc = paged_from_contiguous(K, V, placement, pos, bs)
    tables = np.full((len(lens), max(nblk)), -1, dtype=np.int32)
    for i, p in enumerate(placement):
        tables[i, :len(p)] = p
    out = OA.paged_attention(q, kc, vc, tables, lens, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d,
                             block_size=bs, scale=0.3, q_len=R)
    for i, L in enumerate(lens):
        # row r sees keys t <= L - R + r; SDPA boolean mask: True = attend
        t = torch.arange(L)
        r = torch.arange(R)
        mask = t[None, :] <= (L - R + r[:, None])
        ref = sdpa_ref(q[i].permute(1, 0, 2), K[i], V[i], scale=float(np.float32(0.3)), mask=mask)
        np.testing.assert_allclose(out[i], ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)


def test_chunk_row_equals_single_token_decode_at_shorter_length():
    d, bs, Hq, Hkv, R, L = 8, 4, 2, 1, 16, 37
    nb = -(-L // bs)
    kc = randn_bf16((nb + 3, Hkv, bs, d), 5)
    vc = randn_bf16((nb + 3, Hkv, bs, d), 6)
    table = np.array([list(np.random.default_rng(1).permutation(nb + 3)[:nb])], dtype=np.int32)
    q = randn_bf16((1, R, Hq, d), 7)
    chunk = OA.paged_attention(q, kc, vc, table, [L], num_q_heads=Hq, num_kv_heads=Hkv,
                               head_dim=d, block_size=bs, scale=0.25, q_len=R)
    for r in range(R):
        single = OA.paged_attention(q[:, r:r + 1], kc, vc, table, [L - R + 1 + r], num_q_heads=Hq,
                                    num_kv_heads=Hkv, head_dim=d, block_size=bs, scale=0.25)
        assert np.array_equal(chunk[0, r], single[0, 0])


# ------------------------------------------------------------- closed forms
def _one_seq(L, d=8, bs=4, Hq=2, Hkv=1, seed=0):
    nb = -(-L // bs)
    kc = randn_bf16((nb + 2, Hkv, bs, d), seed)
    vc = randn_bf16((nb + 2, Hkv, bs, d), seed + 1)
    table = np.array([list(range(nb + 1, 1, -1))], dtype=np.int32)  # blocks nb+1 .. 2
    q = randn_bf16((1, 1, Hq, d), seed + 2)
    return q, kc, vc, table


def _run(q, kc, vc, table, L, Hq=2, Hkv=1, d=8, bs=4, scale=0.5):
    return OA.paged_attention(q, kc, vc, table, [L], num_q_heads=Hq, num_kv_heads=Hkv,
                              head_dim=d, block_size=bs, scale=scale)


def test_one_token_returns_its_value():
    q, kc, vc, table = _one_seq(1)
    out = _run(q, kc, vc, table, 1)
    v0 = OA.bf16_bits_to_f64(OA.as_bf16_bits(vc[table[0, 0], 0, 0]))
    for g in range(2):
        assert np.array_equal(out[0, 0, g], v0)


def test_uniform_values_return_that_value():
    L = 23
    q, kc, vc, table = _one_seq(L, seed=3)
    row = randn_bf16((8,), 99)
    vc[:] = row
    out = _run(q, kc, vc, table, L)
    np.testing.assert_allclose(out[0, 0], np.tile(row.double().numpy(), (2, 1)), rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("zero", ["k", "q"])
def test_zero_scores_average_the_values(zero):
    L, bs = 19, 4
    q, kc, vc, table = _one_seq(L, seed=4)
    if zero == "k":
        kc.zero_()
    else:
        q.zero_()
    out = _run(q, kc, vc, table, L)
    rows = []
    for t in range(L):
        rows.append(vc[table[0, t // bs], 0, t % bs].double().numpy())
    np.testing.assert_allclose(out[0, 0, 0], np.mean(rows, axis=0), rtol=1e-13, atol=1e-13)


def test_dominant_key_selects_its_value():
    L, bs, d = 30, 4, 8
    q, kc, vc, table = _one_seq(L, seed=5)
    kc.zero_()
    q.zero_()
    q[0, 0, :, 0] = 1.0
    t_star = 17
    kc[table[0, t_star // bs], 0, t_star % bs, 0] = 1024.0  # score 512 vs 0 at scale 0.5
    out = _run(q, kc, vc, table, L)
    v_star = vc[table[0, t_star // bs], 0, t_star % bs].double().numpy()
    np.testing.assert_allclose(out[0, 0, 0], v_star, rtol=1e-14, atol=1e-14)


def test_identical_queries_in_a_group_give_identical_outputs():
    L = 33
    q, kc, vc, table = _one_seq(L, Hq=4, Hkv=2, seed=6)
    q[0, 0, 1] = q[0, 0, 0]
    q[0, 0, 3] = q[0, 0, 2]
    out = _run(q, kc, vc, table, L, Hq=4, Hkv=2)
    assert np.array_equal(out[0, 0, 0], out[0, 0, 1])
    assert np.array_equal(out[0, 0, 2], out[0, 0, 3])
    assert not np.array_equal(out[0, 0, 0], out[0, 0, 2])  # different KV heads differ


def test_zero_length_gives_zeros():
    q, kc, vc, table = _one_seq(4, seed=7)
    out = _run(q, kc, vc, table, 0)
    assert not out.any()


# ------------------------------------------------------------- invariants
def test_physical_placement_does_not_change_the_result():
    rng = np.random.default_rng(8)
    lens = [3, 17, 40, 64]
    d, bs, Hq, Hkv = 16, 8, 4, 2
    nblk = [-(-n // bs) for n in lens]
    NB = sum(nblk) + 4
    K = [randn_bf16((Hkv, n, d), 50 + i) for i, n in enumerate(lens)]
    V = [randn_bf16((Hkv, n, d), 60 + i) for i, n in enumerate(lens)]
    q = randn_bf16((len(lens), 1, Hq, d), 70)
    outs = []
    for trial in range(3):
        perm = rng.permutation(NB)
        placement, pos = [], 0
        for c in nblk:
            placement.append([int(x) for x in perm[pos:pos + c]])
            pos += c
        kc, vc = paged_from_contiguous(K, V, placement, NB, bs, seed=trial)
        tables = np.full((len(lens), max(nblk)), -1, dtype=np.int32)
        for i, p in enumerate(placement):
            tables[i, :len(p)] = p
        outs.append(OA.paged_attention(q, kc, vc, tables, lens, num_q_heads=Hq, num_kv_heads=Hkv,
                                       head_dim=d, block_size=bs, scale=0.25))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_bad_block_id_is_an_error():
    q, kc, vc, table = _one_seq(9, seed=9)
    table[0, 1] = kc.shape[0]
    with pytest.raises(ValueError):
        _run(q, kc, vc, table, 9)


# ------------------------------------------------- write / copy restatements
def test_write_then_table_gather_reproduces_the_sequence():
    bs, Hkv, d, NB = 4, 2, 8, 12
    L = 10
    a = OracleAllocator(NB, bs)
    a.seq_add(0)
    slots = a.seq_append(0, L)
    k = randn_bf16((L, Hkv, d), 1).view(torch.int16).numpy().view(np.uint16)
    v = randn_bf16((L, Hkv, d), 2).view(torch.int16).numpy().view(np.uint16)
    canary = np.uint16(0x7FC1)
    kc = np.full((NB, Hkv, bs, d), canary, dtype=np.uint16)
    vc = kc.copy()
    cache_ops.write(k, v, np.array(slots, dtype=np.int64), kc, vc, bs)
    table = a.seqs[0]["blocks"]
    for t in range(L):
        assert np.array_equal(kc[table[t // bs], :, t % bs], k[t])
        assert np.array_equal(vc[table[t // bs], :, t % bs], v[t])
    touched = np.zeros((NB, bs), dtype=bool)
    for s in slots:
        touched[s // bs, s % bs] = True
    assert (kc.transpose(0, 2, 1, 3)[~touched] == canary).all()


def test_write_skips_negative_slots_and_rejects_overflow():
    bs, NB = 4, 3
    kc = np.zeros((NB, 1, bs, 2), dtype=np.uint16)
    vc = kc.copy()
    k = np.ones((2, 1, 2), dtype=np.uint16)
    cache_ops.write(k, k, np.array([-1, 5]), kc, vc, bs)
    assert kc.sum() == 2 and kc[1, 0, 1].tolist() == [1, 1]
    with pytest.raises(IndexError):
        cache_ops.write(k, k, np.array([NB * bs, 0]), kc, vc, bs)


def test_block_copy_restatement():
    kc = np.arange(5 * 2 * 3 * 4, dtype=np.uint16).reshape(5, 2, 3, 4)
    vc = kc[::-1].copy()
    k0, v0 = kc.copy(), vc.copy()
    cache_ops.block_copy(kc, vc, [[1, 3], [4, 0]])
    assert np.array_equal(kc[3], k0[1]) and np.array_equal(vc[3], v0[1])
    assert np.array_equal(kc[0], k0[4]) and np.array_equal(vc[0], v0[4])
    for b in (1, 2, 4):
        assert np.array_equal(kc[b], k0[b]) and np.array_equal(vc[b], v0[b])


# ---------------------------------------------------- sharing / copy-on-write
def test_shared_prefix_equals_private_copies():
    """Refcounted prefix blocks + copy-on-write give the same attention as private copies."""
    bs, Hkv, Hq, d, NB = 4, 1, 2, 8, 40
    prefix, samples = 10, 3  # prefix ends inside block 2 -> a real partial shared block
    suffix = [0, 3, 7]
    def fresh(n, seed):
        return randn_bf16((n, Hkv, d), seed).view(torch.int16).numpy().view(np.uint16)

    pk, pv = fresh(prefix, 1), fresh(prefix, 2)
    sk = [fresh(s, 10 + i) for i, s in enumerate(suffix)]
    sv = [fresh(s, 20 + i) for i, s in enumerate(suffix)]

    # shared layout
    a = OracleAllocator(NB, bs)
    kc = np.zeros((NB, Hkv, bs, d), dtype=np.uint16)
    vc = kc.copy()
    a.seq_add(100)
    cache_ops.write(pk, pv, np.array(a.seq_append(100, prefix)), kc, vc, bs)
    for i in range(samples):
        a.seq_fork(100, i)
    a.seq_free(100)
    pairs = []
    for i in range(samples):
        if suffix[i] == 0:
            continue
        last = a.seqs[i]["blocks"][-1]
        if a.refcount[last] > 1:
            with pytest.raises(AllocError) as err:
                a.seq_append(i, suffix[i])  # writing into a shared partial block is refused
            assert err.value.kind == "shared"
        pair = a.seq_cow(i)
        if pair is not None:
            pairs.append(pair)
            cache_ops.block_copy(kc, vc, [pair])
        cache_ops.write(sk[i], sv[i], np.array(a.seq_append(i, suffix[i])), kc, vc, bs)
    # samples 1 and 2 write into the shared partial block and each get a copy;
    # sample 0 keeps the original, now with refcount 1
    assert len(pairs) == 2
    tables, lens = a.block_table(range(samples), 8)
    # refcount conservation: sum of refcounts == number of table entries
    assert sum(a.refcount) == sum(1 for row in tables for b in row if b >= 0)

    # private layout: every sample written on its own
    b = OracleAllocator(NB, bs)
    kc2 = np.zeros_like(kc)
    vc2 = np.zeros_like(vc)
    for i in range(samples):
        b.seq_add(i)
        cache_ops.write(np.concatenate([pk, sk[i]]), np.concatenate([pv, sv[i]]),
                        np.array(b.seq_append(i, prefix + suffix[i])), kc2, vc2, bs)
    tables2, lens2 = b.block_table(range(samples), 8)
    assert lens == lens2
    q = randn_bf16((samples, 1, Hq, d), 77)
    kw = dict(num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_size=bs, scale=0.35)
    o1 = OA.paged_attention(q, kc, vc, np.array(tables, dtype=np.int32), lens, **kw)
    o2 = OA.paged_attention(q, kc2, vc2, np.array(tables2, dtype=np.int32), lens2, **kw)
    assert np.array_equal(o1, o2)
