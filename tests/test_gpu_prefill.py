"""Parity of chunked prefill (paged_attention_prefill, through the C ABI) with the CPU oracle.

Bar: |out - ref| <= 1e-2 + 1e-2 * |ref| elementwise against the fp64 oracle on
the same bf16 inputs; rows that no sequence owns are left untouched (checked
bit for bit against a NaN canary).
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as OA
from paged_kv_cache_276_gb300 import inputs, native
from test_gpu_parity import assert_attention_close, bits, random_case, run_decode, status_tensor

pytestmark = pytest.mark.gpu

CANARY = 0x7FC1  # a NaN bit pattern


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_276_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def prefill_case(lens, chunks, bs, Hq, Hkv, seed, d=128, spare=3):
    rng = np.random.default_rng(seed)
    NB = sum(inputs.entries_to_fill(n, bs) for n in lens) + spare
    maxb = max(1, max(inputs.entries_to_fill(n, bs) for n in lens)) + 2
    tables, _ = inputs.permuted_tables(lens, bs, NB, rng, max_blocks=maxb)
    kc = inputs.randn_bf16((NB, Hkv, bs, d), seed * 10 + 1, "cuda")
    vc = inputs.randn_bf16((NB, Hkv, bs, d), seed * 10 + 2, "cuda")
    q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    q = inputs.randn_bf16((int(q_start[-1]), Hq, d), seed * 10 + 3, "cuda")
    return q, kc, vc, tables, q_start


def run_prefill(q, kc, vc, tables, lens, q_start, scale, status=None, out=None):
    dev = kc.device
    if out is None:
        out = torch.empty_like(q)
        out.view(torch.int16).fill_(CANARY)
    native.paged_attention_prefill(q, kc, vc, torch.as_tensor(np.asarray(tables, dtype=np.int32), device=dev),
                                   torch.as_tensor(np.asarray(lens, dtype=np.int32), device=dev),
                                   torch.as_tensor(np.asarray(q_start, dtype=np.int32), device=dev),
                                   scale, out, status)
    torch.cuda.synchronize()
    return out


def oracle_prefill(q, kc, vc, tables, lens, q_start, Hq, Hkv, bs, scale, d=128):
    return OA.paged_attention_varlen(bits(q), bits(kc), bits(vc), np.asarray(tables, dtype=np.int32),
                                     np.asarray(lens, dtype=np.int32), q_start, num_q_heads=Hq,
                                     num_kv_heads=Hkv, head_dim=d, block_size=bs, scale=scale)


@pytest.mark.parametrize("d,bs,Hq,Hkv,lens,chunks", [
    (64, 16, 32, 4, [700, 129, 40], [300, 129, 1]),      # head dim 64: one 128-byte half per row
    (64, 128, 16, 16, [1000, 64], [256, 64]),            # head dim 64, G = 1, blocks of 128
])
def test_prefill_head_dim_64_matches_oracle(d, bs, Hq, Hkv, lens, chunks):
    q, kc, vc, tables, q_start = prefill_case(lens, chunks, bs, Hq, Hkv, seed=d + bs, d=d)
    scale = float(np.float32(1 / math.sqrt(d)))
    st = status_tensor()
    out = run_prefill(q, kc, vc, tables, lens, q_start, scale, status=st)
    assert st.item() == 0
    ref = oracle_prefill(q, kc, vc, tables, lens, q_start, Hq, Hkv, bs, scale, d=d)
    assert_attention_close(out, ref, "prefill, head dim 64")


@pytest.mark.parametrize("bs,Hq,Hkv,lens,chunks", [
    # a whole prompt, a ragged chunk behind cached context, a decode row, an empty chunk
    (16, 64, 8, [300, 1000, 64, 77, 5], [300, 200, 1, 0, 5]),
    (32, 32, 4, [129, 2048, 16, 700], [129, 100, 16, 33]),
    (64, 16, 16, [513, 70, 1], [513, 70, 1]),            # G = 1: 128 tokens per tile
    (128, 16, 8, [1000, 250, 128], [17, 250, 128]),      # G = 2, blocks of 128 in 64-key tiles
    (16, 32, 8, [400, 9], [400, 9]),                     # G = 4
    (16, 32, 2, [333, 40, 2000], [333, 8, 65]),          # G = 16: 8 tokens per tile
])
def test_prefill_matches_oracle(bs, Hq, Hkv, lens, chunks):
    q, kc, vc, tables, q_start = prefill_case(lens, chunks, bs, Hq, Hkv, seed=bs + Hq + len(lens))
    scale = float(np.float32(1 / math.sqrt(128)))
    st = status_tensor()
    out = run_prefill(q, kc, vc, tables, lens, q_start, scale, status=st)
    assert st.item() == 0
    ref = oracle_prefill(q, kc, vc, tables, lens, q_start, Hq, Hkv, bs, scale)
    assert_attention_close(out, ref, "prefill")


def test_prefill_many_items_per_cta():
    """More query tiles than CTAs: every CTA walks several items, the query
    tile double buffer turns over, and the sequences of the same KV head are
    served in the interleaved order."""
    rng = np.random.default_rng(12)
    lens = [int(x) for x in rng.integers(300, 1600, size=6)]
    chunks = [min(L, 256) for L in lens]
    Hq, Hkv, bs = 32, 4, 16
    q, kc, vc, tables, q_start = prefill_case(lens, chunks, bs, Hq, Hkv, seed=12)
    scale = float(np.float32(1 / math.sqrt(128)))
    out = run_prefill(q, kc, vc, tables, lens, q_start, scale)
    ref = oracle_prefill(q, kc, vc, tables, lens, q_start, Hq, Hkv, bs, scale)
    assert_attention_close(out, ref, "prefill, many items")
    # the schedule is static and the arithmetic order fixed: repeated calls are
    # bit-identical (a read that races its copy would show up here first)
    for _ in range(3):
        again = run_prefill(q, kc, vc, tables, lens, q_start, scale)
        assert torch.equal(again.view(torch.int16), out.view(torch.int16))


def test_prefill_of_uniform_16_token_chunks_matches_the_decode_chunk():
    """The same 16-token causal chunks through both tensor-core schedules (the
    decode chunk on 64-key tiles with one partition per sequence, prefill on
    128-key tiles) agree within the attention tolerance, and with the oracle."""
    lens = [900, 40, 2500, 16]
    Hq, Hkv, bs, d = 64, 8, 16, 128
    q, kc, vc, tables = random_case(lens, d, bs, Hq, Hkv, seed=31, q_len=16)
    scale = float(np.float32(1 / math.sqrt(d)))
    part = 128 * math.ceil(max(lens) / 128)
    dec = run_decode(q, kc, vc, tables, lens, scale, part)
    q_start = np.arange(len(lens) + 1, dtype=np.int32) * 16
    pre = run_prefill(q.reshape(-1, Hq, d), kc, vc, tables, lens, q_start, scale)
    ref = oracle_prefill(q.reshape(-1, Hq, d), kc, vc, tables, lens, q_start, Hq, Hkv, bs, scale)
    assert_attention_close(pre, ref, "prefill")
    assert_attention_close(dec.reshape(-1, Hq, d), ref, "decode chunk")
    assert torch.allclose(dec.reshape(-1, Hq, d).float(), pre.float(), atol=1e-2, rtol=1e-2)


def test_prefill_rescales_running_max():
    """Keys grow in magnitude block by block, so the running max keeps moving."""
    lens, chunks = [1500, 700], [300, 700]
    Hq, Hkv, bs = 16, 2, 16
    q, kc, vc, tables, q_start = prefill_case(lens, chunks, bs, Hq, Hkv, seed=3)
    growth = torch.linspace(0.5, 6.0, kc.shape[0], device="cuda").view(-1, 1, 1, 1)
    kc = (kc.float() * growth).to(torch.bfloat16)
    scale = float(np.float32(1 / math.sqrt(128)))
    out = run_prefill(q, kc, vc, tables, lens, q_start, scale)
    ref = oracle_prefill(q, kc, vc, tables, lens, q_start, Hq, Hkv, bs, scale)
    assert_attention_close(out, ref, "prefill rescale")


@pytest.mark.parametrize("scale", [-0.07, 0.0])
def test_prefill_and_decode_chunk_with_negative_or_zero_scale(scale):
    lens, chunks = [300, 45], [300, 20]
    Hq, Hkv, bs = 64, 8, 16
    q, kc, vc, tables, q_start = prefill_case(lens, chunks, bs, Hq, Hkv, seed=8)
    out = run_prefill(q, kc, vc, tables, lens, q_start, scale)
    ref = oracle_prefill(q, kc, vc, tables, lens, q_start, Hq, Hkv, bs, scale)
    assert_attention_close(out, ref, f"prefill scale {scale}")
    # the 16-token decode chunk runs on the same tensor-core pipeline
    q16, kc16, vc16, t16 = random_case(lens, 128, bs, Hq, Hkv, seed=9, q_len=16)
    dec = run_decode(q16, kc16, vc16, t16, lens, scale, 128)
    ref16 = OA.paged_attention(bits(q16), bits(kc16), bits(vc16), t16, np.asarray(lens, dtype=np.int32),
                               num_q_heads=Hq, num_kv_heads=Hkv, head_dim=128, block_size=bs, scale=scale,
                               q_len=16)
    assert_attention_close(dec, ref16, f"decode chunk scale {scale}")


def test_prefill_edge_rows():
    """A chunk longer than its sequence (leading rows see no key: zeros), an
    empty sequence with an empty chunk, and rows no sequence owns (untouched)."""
    lens, chunks = [5, 0, 40], [8, 0, 40]
    Hq, Hkv, bs = 64, 8, 16
    q, kc, vc, tables, q_start = prefill_case(lens, chunks, bs, Hq, Hkv, seed=4)
    spare = 7  # rows past q_start[-1]
    qx = torch.cat([q, inputs.randn_bf16((spare,) + tuple(q.shape[1:]), 99, "cuda")])
    scale = 0.08
    st = status_tensor()
    out = run_prefill(qx, kc, vc, tables, lens, q_start, scale, status=st)
    assert st.item() == 0
    ref = oracle_prefill(q, kc, vc, tables, lens, q_start, Hq, Hkv, bs, scale)
    assert_attention_close(out[:len(q)], ref, "prefill edges")
    assert not out[:3].float().abs().sum()
    assert torch.all(out[len(q):].view(torch.int16) == CANARY)


def test_prefill_unwritten_tail_slots_never_leak_nan():
    lens, chunks = [17, 70], [17, 6]
    Hq, Hkv, bs = 32, 4, 32
    q, kc, vc, tables, q_start = prefill_case(lens, chunks, bs, Hq, Hkv, seed=6)
    for i, L in enumerate(lens):
        last = tables[i, (L - 1) // bs]
        off = L - ((L - 1) // bs) * bs
        kc[last, :, off:].view(torch.int16).fill_(CANARY)
        vc[last, :, off:].view(torch.int16).fill_(CANARY)
    out = run_prefill(q, kc, vc, tables, lens, q_start, 0.09)
    ref = oracle_prefill(q, kc, vc, tables, lens, q_start, Hq, Hkv, bs, 0.09)
    assert_attention_close(out, ref, "prefill nan tail")


def test_prefill_bad_inputs_set_status_without_fault():
    lens, chunks = [60, 90, 30], [20, 30, 10]
    Hq, Hkv, bs = 64, 8, 16
    q, kc, vc, tables, q_start = prefill_case(lens, chunks, bs, Hq, Hkv, seed=2)
    scale = 0.1
    ref = oracle_prefill(q, kc, vc, tables, lens, q_start, Hq, Hkv, bs, scale)
    # a last entry past the query rows: sequence 2 gets no rows (left untouched), the others are exact
    bad_qs = q_start.copy()
    bad_qs[3] = len(q) + 5
    st = status_tensor()
    out = run_prefill(q, kc, vc, tables, lens, bad_qs, scale, status=st)
    assert st.item() & native.PKV_STATUS_BAD_QSTART
    assert_attention_close(out[:q_start[2]], ref[:q_start[2]], "rows before the bad entry")
    assert torch.all(out[q_start[2]:].view(torch.int16) == CANARY)
    # a decreasing entry is reported too
    bad_qs = q_start.copy()
    bad_qs[2] = bad_qs[1] - 1
    st.zero_()
    run_prefill(q, kc, vc, tables, lens, bad_qs, scale, status=st)
    assert st.item() & native.PKV_STATUS_BAD_QSTART
    # a block id outside the pool reads as zeros and is reported
    bad_tbl = tables.copy()
    bad_tbl[1, 1] = kc.shape[0] + 3
    st.zero_()
    out = run_prefill(q, kc, vc, bad_tbl, lens, q_start, scale, status=st)
    assert st.item() & native.PKV_STATUS_BAD_BLOCK
    assert torch.isfinite(out.float()).all()
    assert_attention_close(out[:q_start[1]], ref[:q_start[1]], "sequence 0 beside a bad block")
    # a length past the table's capacity is clamped and reported
    st.zero_()
    run_prefill(q, kc, vc, tables, [60, tables.shape[1] * bs + 1, 30], q_start, scale, status=st)
    assert st.item() & native.PKV_STATUS_BAD_LEN


def test_mixed_step_of_decodes_and_a_prefill_chunk():
    """One call serves a batch the way a chunked-prefill scheduler builds it:
    many single-token decodes beside one long prompt chunk."""
    rng = np.random.default_rng(21)
    n_dec = 40
    lens = [int(x) for x in rng.integers(1, 3000, size=n_dec)] + [2600]
    chunks = [1] * n_dec + [512]
    Hq, Hkv, bs = 64, 8, 16
    q, kc, vc, tables, q_start = prefill_case(lens, chunks, bs, Hq, Hkv, seed=21)
    scale = float(np.float32(1 / math.sqrt(128)))
    out = run_prefill(q, kc, vc, tables, lens, q_start, scale)
    ref = oracle_prefill(q, kc, vc, tables, lens, q_start, Hq, Hkv, bs, scale)
    assert_attention_close(out, ref, "mixed step")
    # the decode rows also agree with the decode kernel itself
    dec = run_decode(q[:n_dec].unsqueeze(1), kc, vc, tables[:n_dec], lens[:n_dec], scale)
    assert torch.allclose(dec[:, 0].float(), out[:n_dec].float(), atol=1e-2, rtol=1e-2)


@pytest.mark.parametrize("tag,mode", [("prefill_long_context", "plain"), ("prefill_prompts", "plain"),
                                      ("prefill_mixed", "plain"), ("prefill_mixed", "mixed"),
                                      ("prefill_short_chunk", "plain"), ("prefill_short_chunk", "split")])
def test_prefill_workloads_every_sequence(tag, mode):
    """The benchmark's prefill workloads at full size, in the benchmark's launch
    configuration.  Every sequence is compared with the oracle on whole query
    tiles (128 / G tokens x the G heads of each KV head, the unit the kernel
    computes): its first and last tile and one tile in between, and the single
    row of every decode."""
    from paged_kv_cache_276_gb300.workloads import PrefillCase
    case = PrefillCase(inputs.PREFILL_WORKLOADS[tag], "cuda")
    st = status_tensor()
    if mode == "mixed":  # the benchmark's launch: decodes over their work list beside the chunks
        case.prepare_mixed()
        assert case.mixed_nd == 256 and 76 <= case.mixed_ctas <= 152
        case.attend_mixed(st)
    elif mode == "split":  # the benchmark's launch: the keys split into partitions
        case.prepare_split(inputs.PREFILL_WORKLOADS[tag].extra["split"])
        case.attend_split(st)
    else:
        case.attend(st)
    torch.cuda.synchronize()
    assert st.item() == 0
    kb, vb = bits(case.k_cache), bits(case.v_cache)
    qb = bits(case.q)
    out = case.out.float().cpu().double().numpy()
    tile = 128 // (case.Hq // case.Hkv)
    rng = np.random.default_rng(5)
    # (first row, row count, sequence, keys the last row sees) of every checked tile;
    # a decode is a one-row tile.  Rows lo..hi-1 of a chunk of c tokens in a sequence
    # of L see L - c + 1 + r keys: the causal rule of an (hi - lo)-row chunk whose
    # last row sees L - c + hi keys.
    groups = {}
    for i in range(case.B):
        L, c = int(case.lens[i]), int(case.chunks[i])
        if c == 0:
            continue
        ntiles = -(-c // tile)
        for t in sorted({0, ntiles - 1, int(rng.integers(0, ntiles))}):
            lo, hi = t * tile, min(c, (t + 1) * tile)
            groups.setdefault(hi - lo, []).append((int(case.q_start[i]) + lo, i, L - c + hi))
    checked = set()
    for n, tiles in groups.items():  # one oracle call per tile height
        first = np.array([t[0] for t in tiles])
        seqs = [t[1] for t in tiles]
        q = np.stack([qb[r:r + n] for r in first])
        ref = OA.paged_attention(q, kb, vb, case.tables[seqs], np.array([t[2] for t in tiles], dtype=np.int32),
                                 num_q_heads=case.Hq, num_kv_heads=case.Hkv, head_dim=case.d, block_size=case.bs,
                                 scale=case.scale, q_len=n)
        got = np.stack([out[r:r + n] for r in first])
        assert_attention_close(torch.as_tensor(got), ref, f"{tag}: {len(tiles)} tiles of {n} rows")
        checked.update(seqs)
    assert checked == {i for i in range(case.B) if case.chunks[i] > 0}


def test_prefill_at_the_sequence_limit():
    """1024 sequences (the most one prefill call takes): the per-sequence
    tables fill the kernel's shared memory and every lane of the setup warp
    scans 32 sequences."""
    rng = np.random.default_rng(44)
    B = 1024
    lens = [int(x) for x in rng.integers(1, 90, size=B)]
    chunks = [int(min(L, c)) for L, c in zip(lens, rng.integers(0, 40, size=B))]
    Hq, Hkv, bs = 16, 2, 16
    q, kc, vc, tables, q_start = prefill_case(lens, chunks, bs, Hq, Hkv, seed=44)
    scale = float(np.float32(1 / math.sqrt(128)))
    st = status_tensor()
    out = run_prefill(q, kc, vc, tables, lens, q_start, scale, status=st)
    assert st.item() == 0
    ref = oracle_prefill(q, kc, vc, tables, lens, q_start, Hq, Hkv, bs, scale)
    assert_attention_close(out, ref, "prefill, 1024 sequences")


def test_tensor_core_decode_chunk_at_the_sequence_limit():
    """2048 sequences (the most the tensor-core decode chunk takes) of short
    16-token chunks, 8 query heads per KV head."""
    rng = np.random.default_rng(45)
    lens = [int(x) for x in rng.integers(0, 200, size=2048)]
    Hq, Hkv, bs, d = 8, 1, 16, 128
    q, kc, vc, tables = random_case(lens, d, bs, Hq, Hkv, seed=45, q_len=16)
    scale = float(np.float32(1 / math.sqrt(d)))
    st = status_tensor()
    out = run_decode(q, kc, vc, tables, lens, scale, 128, status=st)
    assert st.item() == 0
    ref = OA.paged_attention(bits(q), bits(kc), bits(vc), tables, np.asarray(lens, dtype=np.int32), num_q_heads=Hq,
                             num_kv_heads=Hkv, head_dim=d, block_size=bs, scale=scale, q_len=16)
    assert_attention_close(out, ref, "decode chunk, 2048 sequences")


@pytest.mark.parametrize("d,bs,Hq,Hkv", [(128, 16, 64, 8), (64, 32, 32, 4), (128, 32, 16, 4)])
def test_both_prefill_schedules_match_the_oracle(d, bs, Hq, Hkv):
    """A batch of long chunks runs over pairs of query tiles; padding the
    batch with empty sequences (chunk 0: no rows) lowers the mean chunk below
    two query tiles, and the call then splits each query tile's keys between
    the two softmax sets instead.  Every real row matches the oracle both ways."""
    lens = [700, 129, 40, 1000, 3]
    chunks = [300, 129, 1, 257, 3]
    G = Hq // Hkv
    tile_tok = 128 // G
    n_pad = int(sum(chunks) // (2 * tile_tok)) + 1 - len(lens)  # mean chunk < 2 query tiles
    assert sum(chunks) >= 2 * tile_tok * len(lens)
    pad_lens, pad_chunks = lens + [17] * n_pad, chunks + [0] * n_pad
    assert sum(pad_chunks) < 2 * tile_tok * len(pad_lens)
    scale = float(np.float32(1 / math.sqrt(d)))
    for L_, C_ in ((lens, chunks), (pad_lens, pad_chunks)):
        q, kc, vc, tables, q_start = prefill_case(L_, C_, bs, Hq, Hkv, seed=40 + d, d=d)
        st = status_tensor()
        out = run_prefill(q, kc, vc, tables, L_, q_start, scale, status=st)
        assert st.item() == 0
        ref = oracle_prefill(q, kc, vc, tables, L_, q_start, Hq, Hkv, bs, scale, d=d)
        assert_attention_close(out, ref, f"prefill schedule for {len(L_)} sequences")


@pytest.mark.parametrize("d,bs,Hq,Hkv", [(128, 16, 24, 8), (128, 32, 48, 8), (64, 16, 12, 1), (128, 64, 40, 8),
                                         (128, 16, 6, 2)])
def test_prefill_groups_that_do_not_divide_the_tile(d, bs, Hq, Hkv):
    """G = 3, 6, 12, 5: query tiles of floor(128 / G) tokens x G heads with
    128 mod G spare rows.  Both schedules (pairs of query tiles for long
    chunks; the even / odd key split when most chunks are short) match the
    oracle, chunk ends fall inside tiles, and no row outside the chunks is
    written (the NaN canary survives)."""
    G = Hq // Hkv
    tile_tok = 128 // G
    lens = [700, 129, 40, 1000, 3, 2 * tile_tok + 1]
    chunks = [300, 129, 1, 257, 3, 2 * tile_tok + 1]
    n_pad = int(sum(chunks) // (2 * tile_tok)) + 1 - len(lens)
    pad_lens, pad_chunks = lens + [17] * max(n_pad, 0), chunks + [0] * max(n_pad, 0)
    assert sum(chunks) >= 2 * tile_tok * len(lens) and sum(pad_chunks) < 2 * tile_tok * len(pad_lens)
    scale = float(np.float32(1 / math.sqrt(d)))
    for L_, C_ in ((lens, chunks), (pad_lens, pad_chunks)):
        q, kc, vc, tables, q_start = prefill_case(L_, C_, bs, Hq, Hkv, seed=60 + G, d=d)
        out = torch.empty((int(q_start[-1]) + 5,) + tuple(q.shape[1:]), dtype=q.dtype, device=q.device)
        out.view(torch.int16).fill_(CANARY)
        st = status_tensor()
        run_prefill(q, kc, vc, tables, L_, q_start, scale, status=st, out=out[:q.shape[0]])
        assert st.item() == 0
        ref = oracle_prefill(q, kc, vc, tables, L_, q_start, Hq, Hkv, bs, scale, d=d)
        assert_attention_close(out[:q.shape[0]], ref, f"prefill, group {G}, {len(L_)} sequences")
        assert (bits(out[q.shape[0]:]) == CANARY).all()  # rows past the batch untouched


def run_prefill_split(q, kc, vc, tables, lens, q_start, scale, max_len, part, status=None):
    dev = kc.device
    out = torch.empty_like(q)
    out.view(torch.int16).fill_(CANARY)
    n = native.paged_attention_prefill_workspace_size(q.shape[0], q.shape[1], q.shape[2], max_len, part)
    ws = torch.randint(0, 256, (max(n, 16),), dtype=torch.uint8, device=dev)  # stale bytes: nothing needs clearing
    native.paged_attention_prefill_ex(q, kc, vc, torch.as_tensor(np.asarray(tables, dtype=np.int32), device=dev),
                                      torch.as_tensor(np.asarray(lens, dtype=np.int32), device=dev),
                                      torch.as_tensor(np.asarray(q_start, dtype=np.int32), device=dev), scale, out,
                                      max_len, part, ws, status)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("d,bs,Hq,Hkv,part", [(128, 16, 64, 8, 1024), (128, 32, 32, 8, 256), (64, 16, 24, 8, 128),
                                              (128, 128, 16, 16, 512)])
def test_prefill_split_over_keys_matches_the_oracle(d, bs, Hq, Hkv, part):
    """Split-K prefill: chunks behind long contexts, a decode row, a chunk whose
    early tiles fit one partition while its last ones need several, an empty
    chunk and a chunk shorter than a partition; the merged rows match the oracle
    and the unsplit call."""
    lens = [5000, 3000, 77, 2000, 300, 40]
    chunks = [128, 1, 77, 0, 300, 33]
    q, kc, vc, tables, q_start = prefill_case(lens, chunks, bs, Hq, Hkv, seed=90 + Hq + part, d=d)
    scale = float(np.float32(1 / math.sqrt(d)))
    st = status_tensor()
    out = run_prefill_split(q, kc, vc, tables, lens, q_start, scale, max(lens), part, status=st)
    assert st.item() == 0
    ref = oracle_prefill(q, kc, vc, tables, lens, q_start, Hq, Hkv, bs, scale, d=d)
    assert_attention_close(out, ref, f"split prefill, partitions of {part}")
    whole = run_prefill(q, kc, vc, tables, lens, q_start, scale)
    assert torch.allclose(out.float(), whole.float(), atol=1e-2, rtol=1e-2)


def test_prefill_split_of_a_short_chunk_behind_a_long_context():
    """One 128-token chunk behind 32k cached tokens (64 query / 8 KV heads):
    8 query tiles x 8 KV heads = 64 units of work unsplit; split over keys it
    runs as pairs of query tiles, 4 pairs x 8 KV heads x 16, 8 or 4 partitions
    of 2048, 4096 or 8192 (the benchmark's) keys.  Sampled tiles match the oracle."""
    L, c = 32768, 128
    Hq, Hkv, bs, d = 64, 8, 16, 128
    q, kc, vc, tables, q_start = prefill_case([L], [c], bs, Hq, Hkv, seed=97, d=d)
    scale = float(np.float32(1 / math.sqrt(d)))
    st = status_tensor()
    for part in (2048, 4096, 8192):
        out = run_prefill_split(q, kc, vc, tables, [L], q_start, scale, L, part, status=st)
        assert st.item() == 0
        for lo in (0, 64, 112):  # whole query tiles of 16 tokens
            ref = OA.paged_attention(bits(q[lo:lo + 16])[None], bits(kc), bits(vc), tables,
                                     np.array([L - c + lo + 16], dtype=np.int32), num_q_heads=Hq, num_kv_heads=Hkv,
                                     head_dim=d, block_size=bs, scale=scale, q_len=16)
            assert_attention_close(out[lo:lo + 16], ref[0], f"tile at row {lo}, partitions of {part}")


@pytest.mark.parametrize("ctas", [0, 24, 100])
def test_mixed_step_entry_matches_the_oracle(ctas):
    """paged_attention_mixed: 40 single-token decodes (rows 0..39, over their
    work list) beside two prompt chunks whose grid is capped at `ctas` CTAs
    (0: every SM).  The result is that of paged_attention_prefill over the
    whole batch, and matches the oracle."""
    rng = np.random.default_rng(23)
    n_dec = 40
    lens = [int(x) for x in rng.integers(1, 3000, size=n_dec)] + [2600, 900]
    chunks = [1] * n_dec + [512, 300]
    Hq, Hkv, bs, d = 32, 8, 16, 128
    q, kc, vc, tables, q_start = prefill_case(lens, chunks, bs, Hq, Hkv, seed=23)
    scale = float(np.float32(1 / math.sqrt(d)))
    dev = kc.device
    items = torch.as_tensor(native.pkv_decode_items(np.asarray(lens[:n_dec], dtype=np.int32), tables[:n_dec], Hkv, bs,
                                                    512, d), device=dev)
    n = native.paged_attention_workspace_size(n_dec, 1, Hq, d, max(lens[:n_dec]), 512)
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    out.view(torch.int16).fill_(CANARY)
    st = status_tensor()
    native.paged_attention_mixed(q, kc, vc, torch.as_tensor(np.asarray(tables, dtype=np.int32), device=dev),
                                 torch.as_tensor(np.asarray(lens, dtype=np.int32), device=dev),
                                 torch.as_tensor(q_start, device=dev), scale, out, n_dec, items, max(lens[:n_dec]),
                                 512, ws, ctas, d_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    ref = oracle_prefill(q, kc, vc, tables, lens, q_start, Hq, Hkv, bs, scale)
    assert_attention_close(out, ref, f"mixed step, chunks on {ctas or 'all'} CTAs")
    whole = run_prefill(q, kc, vc, tables, lens, q_start, scale)
    assert torch.allclose(out.float(), whole.float(), atol=1e-2, rtol=1e-2)


def test_prefill_output_on_a_16_byte_boundary_matches_the_aligned_one():
    """The epilogues write 32 bytes per store when the output is 32-byte
    aligned and 16 bytes otherwise: an output 16 bytes past an aligned base
    gets the same bits as the aligned one, for both schedules (pairs of query
    tiles, and single tiles once empty sequences lower the mean chunk)."""
    Hq, Hkv, bs, d = 64, 8, 16, 128
    scale = float(np.float32(1 / math.sqrt(d)))
    for lens, chunks in (([700, 300], [300, 256]), ([700, 300] + [9] * 40, [300, 256] + [0] * 40)):
        q, kc, vc, tables, q_start = prefill_case(lens, chunks, bs, Hq, Hkv, seed=77)
        aligned = run_prefill(q, kc, vc, tables, lens, q_start, scale)
        base = torch.empty(q.numel() + 8, dtype=q.dtype, device=q.device)
        shifted = base[8:].view(q.shape)
        assert shifted.data_ptr() % 32 == 16
        shifted.view(torch.int16).fill_(CANARY)
        run_prefill(q, kc, vc, tables, lens, q_start, scale, out=shifted)
        assert torch.equal(aligned.view(torch.int16), shifted.view(torch.int16))
        ref = oracle_prefill(q, kc, vc, tables, lens, q_start, Hq, Hkv, bs, scale)
        assert_attention_close(shifted, ref, "prefill into a 16-byte-aligned output")


def test_mixed_step_with_a_host_built_chunk_list():
    """paged_attention_mixed with the chunks' pkv_prefill_items list: the same
    bits as without it (each item is computed alike whichever CTA takes it),
    also with the list and no decodes; a list built for another grid size is
    reported (PKV_STATUS_BAD_ITEM) and leaves the chunk rows unwritten,
    without a fault."""
    rng = np.random.default_rng(31)
    n_dec = 24
    lens = [int(x) for x in rng.integers(1, 3000, size=n_dec)] + [2600, 900, 5000]
    chunks = [1] * n_dec + [512, 300, 1024]
    Hq, Hkv, bs, d = 32, 8, 16, 128
    q, kc, vc, tables, q_start = prefill_case(lens, chunks, bs, Hq, Hkv, seed=31)
    scale = float(np.float32(1 / math.sqrt(d)))
    dev = kc.device
    d_tables = torch.as_tensor(np.asarray(tables, dtype=np.int32), device=dev)
    d_lens = torch.as_tensor(np.asarray(lens, dtype=np.int32), device=dev)
    d_qs = torch.as_tensor(q_start, device=dev)
    items = torch.as_tensor(native.pkv_decode_items(np.asarray(lens[:n_dec], dtype=np.int32), tables[:n_dec], Hkv, bs,
                                                    512, d), device=dev)
    ws = torch.empty(native.paged_attention_workspace_size(n_dec, 1, Hq, d, max(lens[:n_dec]), 512),
                     dtype=torch.uint8, device=dev)
    total_q = int(q_start[-1])

    def mixed(ctas, grid_of_list, nd=n_dec):
        chunk_list = None
        if grid_of_list:
            w = native.pkv_prefill_items(np.asarray(lens[nd:]), q_start[nd:], total_q, Hq, Hkv, grid_of_list)
            chunk_list = torch.as_tensor(w, device=dev)
        out = torch.empty_like(q)
        out.view(torch.int16).fill_(CANARY)
        st = status_tensor()
        native.paged_attention_mixed(q, kc, vc, d_tables, d_lens, d_qs, scale, out, nd, items, max(lens[:n_dec]),
                                     512, ws, ctas, d_status=st, prefill_items=chunk_list)
        torch.cuda.synchronize()
        return out, st.item()

    plain, st0 = mixed(37, 0)
    listed, st1 = mixed(37, 37)
    assert st0 == 0 and st1 == 0
    assert torch.equal(plain.view(torch.int16), listed.view(torch.int16))
    whole = run_prefill(q, kc, vc, tables, lens, q_start, scale)
    only_chunks, st2 = mixed(23, 23, nd=0)  # no decodes: the list's grid still caps the chunks
    assert st2 == 0 and torch.equal(only_chunks.view(torch.int16), whole.view(torch.int16))
    ref = oracle_prefill(q, kc, vc, tables, lens, q_start, Hq, Hkv, bs, scale)
    assert_attention_close(listed, ref, "mixed step over the chunk list")
    wrong, st3 = mixed(37, 36)
    assert st3 & native.PKV_STATUS_BAD_ITEM
    assert torch.equal(wrong[:n_dec].view(torch.int16), plain[:n_dec].view(torch.int16))  # the decodes still run
    assert (wrong[n_dec:].view(torch.int16) == CANARY).all()
