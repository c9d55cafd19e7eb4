"""Pins of the chunked-prefill oracle (varying chunk length per sequence), no GPU.

The oracle composes one causal-chunk call per sequence; these tests check the
composition against things other than itself: torch SDPA with an explicit
causal mask on the contiguous K/V, the single-token decode of the same
oracle, and closed forms (one visible key, no visible key).
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as OA
from test_oracle_pins import paged_from_contiguous, randn_bf16, sdpa_ref


def _pool(lens, Hkv, d, bs, seed):
    nblk = [-(-n // bs) for n in lens]
    rng = np.random.default_rng(seed)
    perm = rng.permutation(sum(nblk) + 3)
    placement, pos = [], 0
    for c in nblk:
        placement.append([int(x) for x in perm[pos:pos + c]])
        pos += c
    K = [randn_bf16((Hkv, n, d), seed + 10 + i) for i, n in enumerate(lens)]
    V = [randn_bf16((Hkv, n, d), seed + 50 + i) for i, n in enumerate(lens)]
    kc, vc = paged_from_contiguous(K, V, placement, sum(nblk) + 3, bs, seed=seed)
    tables = np.full((len(lens), max(1, max(nblk))), -1, dtype=np.int32)
    for i, p in enumerate(placement):
        tables[i, :len(p)] = p
    return K, V, kc, vc, tables


@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (8, 1), (2, 2)])
def test_varlen_matches_masked_sdpa(Hq, Hkv):
    d, bs = 16, 8
    lens = [9, 30, 1, 17, 40]
    chunks = [9, 5, 1, 0, 33]  # a whole prompt, a chunk, a decode, nothing, a long chunk
    K, V, kc, vc, tables = _pool(lens, Hkv, d, bs, 3)
    q_start = np.concatenate([[0], np.cumsum(chunks)])
    q = randn_bf16((int(q_start[-1]), Hq, d), 77)
    out = OA.paged_attention_varlen(q, kc, vc, tables, lens, q_start, num_q_heads=Hq, num_kv_heads=Hkv,
                                    head_dim=d, block_size=bs, scale=0.35)
    assert out.shape == (int(q_start[-1]), Hq, d)
    for i, (L, c) in enumerate(zip(lens, chunks)):
        if c == 0:
            continue
        t, r = torch.arange(L), torch.arange(c)
        mask = t[None, :] <= (L - c + r[:, None])
        rows = q[q_start[i]:q_start[i + 1]]
        ref = sdpa_ref(rows.permute(1, 0, 2), K[i], V[i], scale=float(np.float32(0.35)), mask=mask)
        np.testing.assert_allclose(out[q_start[i]:q_start[i + 1]], ref.permute(1, 0, 2).numpy(),
                                   rtol=1e-12, atol=1e-12)


def test_single_token_chunks_equal_decode():
    d, bs, Hq, Hkv = 8, 4, 4, 2
    lens = [3, 11, 20]
    _, _, kc, vc, tables = _pool(lens, Hkv, d, bs, 9)
    q = randn_bf16((3, Hq, d), 5)
    vl = OA.paged_attention_varlen(q, kc, vc, tables, lens, [0, 1, 2, 3], num_q_heads=Hq, num_kv_heads=Hkv,
                                   head_dim=d, block_size=bs, scale=0.5)
    dec = OA.paged_attention(q[:, None], kc, vc, tables, lens, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d,
                             block_size=bs, scale=0.5)
    assert np.array_equal(vl, dec[:, 0])


def test_first_row_of_a_whole_prompt_returns_the_first_value():
    # a prompt prefilled from an empty cache: row 0 sees key 0 only, so its
    # output is V[0] exactly, whatever the scores
    d, bs, Hq, Hkv, L = 8, 4, 2, 1, 13
    K, V, kc, vc, tables = _pool([L], Hkv, d, bs, 21)
    q = randn_bf16((L, Hq, d), 4) * 5
    out = OA.paged_attention_varlen(q, kc, vc, tables, [L], [0, L], num_q_heads=Hq, num_kv_heads=Hkv,
                                    head_dim=d, block_size=bs, scale=1 / math.sqrt(d))
    for g in range(Hq):
        np.testing.assert_array_equal(out[0, g], V[0][0, 0].double().numpy())


def test_chunk_longer_than_the_sequence_gives_zero_rows():
    d, bs, Hq, Hkv = 8, 4, 2, 1
    _, _, kc, vc, tables = _pool([5], Hkv, d, bs, 2)
    q = randn_bf16((8, Hq, d), 1)
    out = OA.paged_attention_varlen(q, kc, vc, tables, [5], [0, 8], num_q_heads=Hq, num_kv_heads=Hkv,
                                    head_dim=d, block_size=bs, scale=0.5)
    assert not np.any(out[:3])   # rows 0..2 see L - 8 + 1 + r <= 0 keys
    assert np.all(np.any(out[3:] != 0, axis=-1))


def test_bad_q_start_is_rejected():
    d, bs, Hq, Hkv = 8, 4, 2, 1
    _, _, kc, vc, tables = _pool([5, 5], Hkv, d, bs, 2)
    q = randn_bf16((4, Hq, d), 1)
    for qs in ([0, 3, 2], [1, 2, 4], [0, 2]):
        with pytest.raises(ValueError):
            OA.paged_attention_varlen(q, kc, vc, tables, [5, 5], qs, num_q_heads=Hq, num_kv_heads=Hkv,
                                      head_dim=d, block_size=bs, scale=0.5)
