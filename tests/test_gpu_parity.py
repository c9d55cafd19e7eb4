"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bars: bit-exact for pkv_write, pkv_block_copy and the bookkeeping; for the
bf16-in / fp32-accumulate attention output against the fp64 oracle on the same
bf16 inputs, |out - ref| <= 1e-2 + 1e-2 * |ref| elementwise.

Oracle inputs never come from the CUDA path: tables and slots come from the
oracle allocator or the seeded generators, caches are copied to the host
before any kernel writes them, and the oracle applies its own write and copy
to those host copies.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import cache_ops
from oracle.allocator import OracleAllocator
from paged_kv_cache_276_gb300 import inputs, native
from paged_kv_cache_276_gb300.workloads import DecodeSession

pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_276_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def bits(t):
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def assert_attention_close(got_bf16, ref, what=""):
    got = got_bf16.detach().float().cpu().double().numpy()
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance; "
                           f"max err {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")


def status_tensor():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def run_decode(q, kc, vc, tables, lens, scale, partition=0, max_len=None, status=None):
    dev = kc.device
    tables_d = torch.as_tensor(np.asarray(tables, dtype=np.int32), device=dev)
    lens_d = torch.as_tensor(np.asarray(lens, dtype=np.int32), device=dev)
    B, q_len, Hq, d = q.shape
    max_len = int(np.max(lens)) if max_len is None else max_len
    n = native.paged_attention_workspace_size(B, q_len, Hq, d, max_len, partition)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device=dev) if n else None
    out = torch.full_like(q, float("nan"))
    native.paged_attention_decode(q, kc, vc, tables_d, lens_d, max_len, scale, out, ws, partition, status)
    torch.cuda.synchronize()
    return out


def oracle_decode(q, kc, vc, tables, lens, w_or_dims, scale, q_len=1):
    Hq, Hkv, d, bs = w_or_dims
    return OA.paged_attention(bits(q), bits(kc), bits(vc), np.asarray(tables, dtype=np.int32),
                              np.asarray(lens, dtype=np.int32), num_q_heads=Hq, num_kv_heads=Hkv,
                              head_dim=d, block_size=bs, scale=scale, q_len=q_len)


def random_case(lens, d, bs, Hq, Hkv, seed, q_len=1, spare=3):
    rng = np.random.default_rng(seed)
    NB = sum(inputs.entries_to_fill(n, bs) for n in lens) + spare
    tables, _ = inputs.permuted_tables(lens, bs, NB, rng, max_blocks=max(1, max(inputs.entries_to_fill(n, bs) for n in lens)) + 2)
    kc = inputs.randn_bf16((NB, Hkv, bs, d), seed * 10 + 1, "cuda")
    vc = inputs.randn_bf16((NB, Hkv, bs, d), seed * 10 + 2, "cuda")
    q = inputs.randn_bf16((len(lens), q_len, Hq, d), seed * 10 + 3, "cuda")
    return q, kc, vc, tables


# ------------------------------------------------------------------ write / copy
@pytest.mark.parametrize("d,bs,Hkv", [(128, 16, 8), (64, 32, 2)])
def test_pkv_write_bit_exact(d, bs, Hkv):
    rng = np.random.default_rng(d + bs)
    NB, T = 41, 300
    slots = inputs.distinct_slots(T, NB * bs, rng, skip_fraction=0.1)
    k = inputs.randn_bf16((T, Hkv, d), 5, "cuda")
    v = inputs.randn_bf16((T, Hkv, d), 6, "cuda")
    canary = torch.full((NB, Hkv, bs, d), 0.0, dtype=torch.bfloat16, device="cuda")
    canary.view(torch.int16).fill_(0x7FC1)  # a NaN pattern: untouched slots must keep it bit for bit
    kc, vc = canary.clone(), canary.clone()
    kc_h, vc_h = bits(kc), bits(vc)
    cache_ops.write(bits(k), bits(v), slots, kc_h, vc_h, bs)
    st = status_tensor()
    native.pkv_write(k, v, torch.as_tensor(slots, device="cuda"), kc, vc, st)
    torch.cuda.synchronize()
    assert np.array_equal(bits(kc), kc_h) and np.array_equal(bits(vc), vc_h)
    assert st.item() == 0


def test_pkv_write_out_of_range_slot_sets_status_and_is_skipped():
    NB, bs, Hkv, d = 4, 16, 2, 64
    k = inputs.randn_bf16((3, Hkv, d), 1, "cuda")
    kc = torch.zeros((NB, Hkv, bs, d), dtype=torch.bfloat16, device="cuda")
    vc = kc.clone()
    st = status_tensor()
    native.pkv_write(k, k, torch.tensor([5, NB * bs, -3], device="cuda"), kc, vc, st)
    torch.cuda.synchronize()
    assert st.item() & native.PKV_STATUS_BAD_SLOT
    expect = np.zeros((NB, Hkv, bs, d), dtype=np.uint16)
    cache_ops.write(bits(k)[:1], bits(k)[:1], np.array([5]), expect, expect.copy(), bs)
    assert np.array_equal(bits(kc), expect)


@pytest.mark.parametrize("d,bs,Hkv", [(128, 16, 8), (64, 32, 2)])
def test_pkv_block_copy_bit_exact(d, bs, Hkv):
    rng = np.random.default_rng(7)
    NB = 60
    perm = rng.permutation(NB)
    pairs = np.stack([perm[:20], perm[20:40]], axis=1).astype(np.int32)
    kc = inputs.randn_bf16((NB, Hkv, bs, d), 11, "cuda")
    vc = inputs.randn_bf16((NB, Hkv, bs, d), 12, "cuda")
    kc_h, vc_h = bits(kc), bits(vc)
    cache_ops.block_copy(kc_h, vc_h, pairs)
    st = status_tensor()
    native.pkv_block_copy(kc, vc, torch.as_tensor(pairs, device="cuda"), st)
    torch.cuda.synchronize()
    assert np.array_equal(bits(kc), kc_h) and np.array_equal(bits(vc), vc_h)
    assert st.item() == 0
    bad = torch.tensor([[0, NB], [-1, 3]], dtype=torch.int32, device="cuda")
    native.pkv_block_copy(kc, vc, bad, st)
    torch.cuda.synchronize()
    assert st.item() & native.PKV_STATUS_BAD_BLOCK
    assert np.array_equal(bits(kc), kc_h)


# ------------------------------------------------------------------ swap out / in
@pytest.mark.parametrize("d,bs,Hkv", [(128, 16, 8), (64, 32, 2)])
def test_swap_out_and_in_bit_exact(d, bs, Hkv):
    NB = 40
    kc = inputs.randn_bf16((NB, Hkv, bs, d), 71, "cuda")
    vc = inputs.randn_bf16((NB, Hkv, bs, d), 72, "cuda")
    k_h, v_h = bits(kc), bits(vc)
    ids = np.array([5, 0, 39, 17, 18, 2], dtype=np.int32)
    ids_d = torch.as_tensor(ids, device="cuda")
    hk = torch.empty((len(ids), Hkv, bs, d), dtype=torch.bfloat16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    st = status_tensor()
    native.pkv_swap_out(kc, vc, ids_d, hk, hv, st)
    torch.cuda.synchronize()
    ek, ev = cache_ops.swap_out(k_h, v_h, ids)
    assert np.array_equal(hk.view(torch.int16).numpy().view(np.uint16), ek)
    assert np.array_equal(hv.view(torch.int16).numpy().view(np.uint16), ev)
    # back into other blocks
    dst = np.array([30, 31, 1, 3, 4, 6], dtype=np.int32)
    native.pkv_swap_in(hk, hv, torch.as_tensor(dst, device="cuda"), kc, vc, st)
    torch.cuda.synchronize()
    cache_ops.swap_in(ek, ev, dst, k_h, v_h)
    assert np.array_equal(bits(kc), k_h) and np.array_equal(bits(vc), v_h)
    assert st.item() == 0
    bad = torch.as_tensor(np.array([2, NB + 3], dtype=np.int32), device="cuda")
    hk2 = torch.zeros((2, Hkv, bs, d), dtype=torch.bfloat16).pin_memory()
    hv2 = torch.zeros_like(hk2).pin_memory()
    native.pkv_swap_out(kc, vc, bad, hk2, hv2, st)
    torch.cuda.synchronize()
    assert st.item() & native.PKV_STATUS_BAD_BLOCK
    assert np.array_equal(hk2[0].view(torch.int16).numpy().view(np.uint16), k_h[2])
    assert not hk2[1].view(torch.int16).any()  # skipped


def test_decode_after_a_swap_round_trip_is_bit_identical():
    """Swap one sequence out, let other writes reuse its blocks, swap it back
    into fresh blocks: the decode gives the same bits as before."""
    d, bs, Hq, Hkv = 128, 16, 32, 8
    NB = 100
    alloc = native.BlockAllocator(NB, bs)
    kc = inputs.randn_bf16((NB, Hkv, bs, d), 81, "cuda")
    vc = inputs.randn_bf16((NB, Hkv, bs, d), 82, "cuda")
    lens = [300, 700, 45]
    for i, n in enumerate(lens):
        alloc.seq_add(i)
        alloc.seq_append(i, n)
    q = inputs.randn_bf16((3, 1, Hq, d), 83, "cuda")

    def decode():
        table, ln = alloc.block_table(range(3), 48)
        return run_decode(q, kc, vc, table, ln, 0.09, 512)

    before = decode()
    out_ids = alloc.seq_swap_out(1)
    hk = torch.empty((len(out_ids), Hkv, bs, d), dtype=torch.bfloat16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    native.pkv_swap_out(kc, vc, torch.as_tensor(out_ids, device="cuda"), hk, hv)
    # another sequence takes the freed blocks and overwrites them
    alloc.seq_add(9)
    slots = alloc.seq_append(9, 700)
    junk = inputs.randn_bf16((700, Hkv, d), 84, "cuda")
    native.pkv_write(junk, junk, torch.as_tensor(slots, device="cuda"), kc, vc)
    alloc.seq_free(9)
    alloc.seq_add(10)
    alloc.seq_append(10, 5 * bs)  # holds the top of the free stack, so sequence 1 lands elsewhere
    in_ids = alloc.seq_swap_in(1)
    assert set(in_ids.tolist()) != set(out_ids.tolist())
    native.pkv_swap_in(hk, hv, torch.as_tensor(in_ids, device="cuda"), kc, vc)
    after = decode()
    assert torch.equal(after.view(torch.int16), before.view(torch.int16))
    alloc.close()


def test_decode_over_prefix_cached_blocks_equals_private_storage():
    """Sequence B shares its first blocks with A through the prefix cache (their
    slots come back -1 and pkv_write skips them); its decode is bit for bit the
    decode of the same tokens stored privately."""
    d, bs, Hq, Hkv = 128, 16, 32, 8
    NB, P = 64, 96
    kv_k = inputs.randn_bf16((3, P, Hkv, d), 91, "cuda")  # K / V of token id t at position p
    kv_v = inputs.randn_bf16((3, P, Hkv, d), 92, "cuda")

    def store(alloc, kc, vc, sid, toks, cached_ok):
        slots, cached = alloc.seq_append_tokens(sid, toks)
        if not cached_ok:
            assert cached == 0
        start = alloc.seq_len(sid) - len(toks)
        pos = torch.arange(start, start + len(toks), device="cuda")
        tid = torch.as_tensor(np.asarray(toks, dtype=np.int64), device="cuda")
        native.pkv_write(kv_k[tid, pos].contiguous(), kv_v[tid, pos].contiguous(),
                         torch.as_tensor(slots, device="cuda"), kc, vc)
        return cached

    rng = np.random.default_rng(17)
    prompt = rng.integers(0, 3, size=40).tolist()
    tail_a, tail_b = rng.integers(0, 3, size=9).tolist(), rng.integers(0, 3, size=21).tolist()
    q = inputs.randn_bf16((1, 1, Hq, d), 93, "cuda")
    # shared: A stores the prompt, B finds its two full blocks
    a = native.BlockAllocator(NB, bs)
    kc = torch.zeros((NB, Hkv, bs, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    a.seq_add(0)
    store(a, kc, vc, 0, prompt + tail_a, False)
    a.seq_add(1)
    assert store(a, kc, vc, 1, prompt + tail_b, True) == 32
    t1, l1 = a.block_table([1], 8)
    t0, _ = a.block_table([0], 8)
    assert t1[0, :2].tolist() == t0[0, :2].tolist()
    shared = run_decode(q, kc, vc, t1, l1, 0.09, 512)
    # private: B alone in a fresh pool
    b = native.BlockAllocator(NB, bs)
    kc2 = torch.zeros_like(kc)
    vc2 = torch.zeros_like(kc)
    b.seq_add(1)
    store(b, kc2, vc2, 1, prompt + tail_b, False)
    t2, l2 = b.block_table([1], 8)
    private = run_decode(q, kc2, vc2, t2, l2, 0.09, 512)
    assert torch.equal(shared.view(torch.int16), private.view(torch.int16))
    a.close()
    b.close()


# ------------------------------------------------------------------ attention
@pytest.mark.parametrize("d,bs,Hq,Hkv,lens,partition", [
    (64, 16, 4, 2, [17, 33, 64], 0),                      # the tiny workload's shapes
    (128, 16, 32, 8, [1, 15, 16, 17, 511, 512, 513, 1500], 512),
    (128, 32, 64, 8, [1, 31, 32, 33, 700, 2049], 512),
    (128, 16, 8, 8, [5, 100, 300], 32),                   # MHA, tiny partitions
    (128, 16, 16, 1, [77, 1024], 64),                     # group 16 (two n-tiles)
    (64, 32, 12, 4, [3, 64, 65, 1000], 96),
    (128, 32, 8, 2, [40, 2000], 0),
    (64, 16, 2, 1, [0, 1, 2, 1999], 128),                 # empty sequence gives zeros
    (128, 64, 32, 8, [1, 63, 64, 65, 700, 2049], 512),    # block 64: staged as 16-row units
    (64, 128, 8, 2, [5, 127, 128, 129, 1500], 256),       # block 128
    (128, 128, 16, 1, [77, 1024, 0], 0),                  # block 128, group 16, default partition
    # block 16 is staged two blocks per 32-row unit: partitions of an odd number
    # of blocks end inside a unit, whose second block is then past the partition
    (128, 16, 32, 8, [1, 15, 16, 17, 47, 48, 49, 1500], 48),
    (64, 16, 8, 2, [33, 700], 16),
])
def test_decode_matches_oracle(d, bs, Hq, Hkv, lens, partition):
    q, kc, vc, tables = random_case(lens, d, bs, Hq, Hkv, seed=d + bs + Hq + len(lens))
    scale = float(np.float32(1 / math.sqrt(d)))
    st = status_tensor()
    out = run_decode(q, kc, vc, tables, lens, scale, partition, status=st)
    ref = oracle_decode(q, kc, vc, tables, lens, (Hq, Hkv, d, bs), scale)
    assert_attention_close(out, ref, f"d{d} bs{bs} {Hq}/{Hkv} part{partition}")
    assert st.item() == 0


@pytest.mark.parametrize("d,bs,Hq,Hkv,lens,partition", [
    (128, 16, 64, 8, [16, 17, 40, 600], 512),     # 16 x 8 = 128 rows per KV head
    (128, 32, 64, 8, [1000, 31], 128),
    (64, 16, 8, 2, [3, 16, 100], 32),             # rows < 16: causal rows with nothing to see
    (128, 16, 16, 8, [530], 64),
    (128, 64, 64, 8, [100, 700, 16], 512),        # block 64: warp-MMA chunk kernel
    (64, 128, 8, 2, [1000, 3], 256),              # block 128
    (128, 16, 48, 8, [100, 530], 48),             # group 6, block 16: 3-block partitions end inside a unit
])
def test_chunked_causal_query_matches_oracle(d, bs, Hq, Hkv, lens, partition):
    q, kc, vc, tables = random_case(lens, d, bs, Hq, Hkv, seed=3 + d + bs + Hq, q_len=16)
    scale = float(np.float32(1 / math.sqrt(d)))
    out = run_decode(q, kc, vc, tables, lens, scale, partition)
    ref = oracle_decode(q, kc, vc, tables, lens, (Hq, Hkv, d, bs), scale, q_len=16)
    assert_attention_close(out, ref, "chunk")


@pytest.mark.parametrize("bs,lens,partition", [
    (16, [16, 17, 40, 600, 64, 65, 1000], 512),
    (32, [1000, 31, 2048, 3], 128),
    (16, [0, 5, 15, 16, 200, 0, 130], 128),        # empty and shorter-than-chunk sequences
    (16, [int(x) for x in np.random.default_rng(4).integers(1, 3000, size=40)], 256),  # many runs per CTA
    (32, [4096, 4096, 100, 7], 128),
    (64, [3000, 129, 1], 384),
    (128, [2500, 700, 128, 127], 256),
])
def test_chunk_tensor_core_path_matches_oracle(bs, lens, partition):
    """16-token causal chunk with 8 query heads per KV head and head dim 128: the tcgen05 kernel."""
    d, Hq, Hkv = 128, 64, 8
    q, kc, vc, tables = random_case(lens, d, bs, Hq, Hkv, seed=17 + bs + len(lens), q_len=16)
    scale = float(np.float32(1 / math.sqrt(d)))
    st = status_tensor()
    out = run_decode(q, kc, vc, tables, lens, scale, partition, status=st)
    assert st.item() == 0
    ref = oracle_decode(q, kc, vc, tables, lens, (Hq, Hkv, d, bs), scale, q_len=16)
    assert_attention_close(out, ref, "tcgen05 chunk")


@pytest.mark.parametrize("bs,Hq,Hkv,lens,partition", [
    (16, 32, 8, [3000, 1, 0, 700, 64, 65, 2049], 512),     # G = 4, empty and one-token sequences
    (32, 64, 8, [5000, 17, 1300], 0),                      # G = 8, the default partition
    (64, 16, 16, [900, 4100, 63], 256),                    # G = 1
    (128, 32, 2, [2500, 129, 40], 384),                    # G = 16, blocks of 128
])
def test_single_token_decode_on_tensor_cores(bs, Hq, Hkv, lens, partition):
    """A bound of 16384 on the lengths sends single-token decodes (head dim 128)
    to the tcgen05 kernel, G valid rows of a 128-row tile; the warp-MMA kernel
    (a smaller bound) must agree with it and both with the oracle."""
    d = 128
    q, kc, vc, tables = random_case(lens, d, bs, Hq, Hkv, seed=41 + bs + Hq)
    scale = float(np.float32(1 / math.sqrt(d)))
    st = status_tensor()
    tc = run_decode(q, kc, vc, tables, lens, scale, partition, max_len=16384, status=st)
    assert st.item() == 0
    ref = oracle_decode(q, kc, vc, tables, lens, (Hq, Hkv, d, bs), scale)
    assert_attention_close(tc, ref, "tcgen05 single-token decode")
    mma = run_decode(q, kc, vc, tables, lens, scale, partition)
    assert torch.allclose(tc.float(), mma.float(), atol=1e-2, rtol=1e-2)


@pytest.mark.parametrize("q_len,G,lens,max_len", [
    (16, 8, [900, 17, 2500], None),          # 16-token chunk, head dim 64, on the tcgen05 kernel
    (1, 4, [3000, 1, 700], 16384),           # a single-token decode routed to it by the length bound
])
def test_tensor_core_kernel_head_dim_64(q_len, G, lens, max_len):
    d, bs, Hkv = 64, 32, 2
    Hq = G * Hkv
    q, kc, vc, tables = random_case(lens, d, bs, Hq, Hkv, seed=51 + q_len, q_len=q_len)
    scale = float(np.float32(1 / math.sqrt(d)))
    st = status_tensor()
    out = run_decode(q, kc, vc, tables, lens, scale, 256, max_len=max_len, status=st)
    assert st.item() == 0
    ref = oracle_decode(q, kc, vc, tables, lens, (Hq, Hkv, d, bs), scale, q_len=q_len)
    assert_attention_close(out, ref, f"tcgen05, head dim 64, q_len {q_len}")


def test_chunk_tensor_core_rescales_running_max():
    """Keys grow in magnitude block by block, so the running max keeps moving (rescale path)."""
    d, bs, Hq, Hkv = 128, 16, 16, 2
    lens = [1500, 700]
    q, kc, vc, tables = random_case(lens, d, bs, Hq, Hkv, seed=3, q_len=16)
    growth = torch.linspace(0.5, 6.0, kc.shape[0], device="cuda").view(-1, 1, 1, 1)
    kc = (kc.float() * growth).to(torch.bfloat16)
    scale = float(np.float32(1 / math.sqrt(d)))
    out = run_decode(q, kc, vc, tables, lens, scale, 512)
    ref = oracle_decode(q, kc, vc, tables, lens, (Hq, Hkv, d, bs), scale, q_len=16)
    assert_attention_close(out, ref, "tcgen05 chunk rescale")


def test_chunk_tensor_core_and_warp_mma_paths_agree():
    d, bs, Hq, Hkv = 128, 16, 64, 8
    lens = [900, 2500, 17]
    q, kc, vc, tables = random_case(lens, d, bs, Hq, Hkv, seed=5, q_len=16)
    scale = float(np.float32(1 / math.sqrt(d)))
    a = run_decode(q, kc, vc, tables, lens, scale, 512).float()   # tcgen05
    b = run_decode(q, kc, vc, tables, lens, scale, 496).float()   # not a multiple of 128: warp MMA
    assert torch.allclose(a, b, atol=1e-2, rtol=1e-2)


def test_partition_size_changes_little_and_placement_changes_nothing():
    lens = [900, 2500, 4096, 37]
    d, bs, Hq, Hkv = 128, 16, 32, 8
    q, kc, vc, tables = random_case(lens, d, bs, Hq, Hkv, seed=99)
    scale = float(np.float32(1 / math.sqrt(d)))
    ref = oracle_decode(q, kc, vc, tables, lens, (Hq, Hkv, d, bs), scale)
    outs = {}
    for part in (16, 64, 512, 4096):
        outs[part] = run_decode(q, kc, vc, tables, lens, scale, part)
        assert_attention_close(outs[part], ref, f"partition {part}")
    # move every block to a new physical place: same logical content, same bits out
    NB = kc.shape[0]
    perm = torch.randperm(NB, generator=torch.Generator().manual_seed(5))
    kc2 = torch.empty_like(kc)
    vc2 = torch.empty_like(vc)
    kc2[perm.cuda()] = kc
    vc2[perm.cuda()] = vc
    tables2 = np.where(tables >= 0, perm.numpy()[np.maximum(tables, 0)], -1).astype(np.int32)
    moved = run_decode(q, kc2, vc2, tables2, lens, scale, 512)
    assert torch.equal(moved.view(torch.int16), outs[512].view(torch.int16))


# ------------------------------------------------ the library's default schedule
# partition_size 0: 768-token partitions, chosen by the library.
@pytest.mark.parametrize("d,bs,Hq,Hkv,lens", [
    (128, 16, 32, 8, [int(x) for x in np.random.default_rng(7).integers(0, 3000, size=37)]),  # mixed, empties
    (128, 32, 64, 8, [1, 31, 32, 33, 700, 2049, 0, 5000]),
    (64, 16, 8, 1, [40000]),                 # one sequence over 53 partitions
    (64, 32, 6, 2, [17, 33, 64]),            # one partition each: no merge
    (128, 16, 8, 8, [300, 1, 4095, 16, 17]),  # one query head per KV head
    (128, 16, 16, 2, [0, 0, 0]),             # nothing to read: zeros
])
def test_default_schedule_matches_oracle(d, bs, Hq, Hkv, lens):
    q, kc, vc, tables = random_case(lens, d, bs, Hq, Hkv, seed=41 + d + bs + Hq + len(lens))
    scale = float(np.float32(1 / math.sqrt(d)))
    st = status_tensor()
    out = run_decode(q, kc, vc, tables, lens, scale, 0, status=st)
    ref = oracle_decode(q, kc, vc, tables, lens, (Hq, Hkv, d, bs), scale)
    assert_attention_close(out, ref, f"default d{d} bs{bs} {Hq}/{Hkv}")
    assert st.item() == 0


def test_default_schedule_is_the_768_token_partition_and_placement_changes_nothing():
    lens = [900, 2500, 4096, 37, 1, 1500]
    d, bs, Hq, Hkv = 128, 16, 32, 8
    q, kc, vc, tables = random_case(lens, d, bs, Hq, Hkv, seed=77)
    scale = float(np.float32(1 / math.sqrt(d)))
    bal = run_decode(q, kc, vc, tables, lens, scale, 0)
    grid = run_decode(q, kc, vc, tables, lens, scale, 768)
    assert torch.equal(bal.view(torch.int16), grid.view(torch.int16))
    NB = kc.shape[0]
    perm = torch.randperm(NB, generator=torch.Generator().manual_seed(9))
    kc2 = torch.empty_like(kc)
    vc2 = torch.empty_like(vc)
    kc2[perm.cuda()] = kc
    vc2[perm.cuda()] = vc
    tables2 = np.where(tables >= 0, perm.numpy()[np.maximum(tables, 0)], -1).astype(np.int32)
    moved = run_decode(q, kc2, vc2, tables2, lens, scale, 0)
    assert torch.equal(moved.view(torch.int16), bal.view(torch.int16))


def test_default_schedule_reuses_a_dirty_workspace():
    """The workspace starts as random bytes and is reused by successive calls
    with different batches: nothing in it needs clearing."""
    d, bs, Hq, Hkv = 128, 16, 32, 8
    n = native.paged_attention_workspace_size(64, 1, Hq, d, 6000, 0)
    ws = torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda")
    rng = np.random.default_rng(31)
    for call in range(4):
        lens = [int(x) for x in rng.integers(1, 6000, size=int(rng.integers(3, 64)))]
        q, kc, vc, tables = random_case(lens, d, bs, Hq, Hkv, seed=200 + call)
        out = torch.full_like(q, float("nan"))
        native.paged_attention_decode(q, kc, vc, torch.as_tensor(tables, device="cuda"),
                                      torch.as_tensor(np.asarray(lens, dtype=np.int32), device="cuda"),
                                      max(lens), 0.09, out, ws, 0)
        torch.cuda.synchronize()
        ref = oracle_decode(q, kc, vc, tables, lens, (Hq, Hkv, d, bs), 0.09)
        assert_attention_close(out, ref, f"call {call}")


def test_default_schedule_at_the_edges():
    """4100 sequences, a group of 16, and no workspace for a batch that fits one
    partition per sequence."""
    rng = np.random.default_rng(12)
    lens = [int(x) for x in rng.integers(0, 40, size=4100)]
    d, bs, Hq, Hkv = 64, 16, 4, 2
    q, kc, vc, tables = random_case(lens, d, bs, Hq, Hkv, seed=13)
    out = run_decode(q, kc, vc, tables, lens, 0.125, 0)
    ref = oracle_decode(q, kc, vc, tables, lens, (Hq, Hkv, d, bs), 0.125)
    assert_attention_close(out, ref, "4100 sequences")
    lens = [77, 1024, 3000]
    q, kc, vc, tables = random_case(lens, 128, 16, 16, 1, seed=14)
    out = run_decode(q, kc, vc, tables, lens, 0.09, 0)
    ref = oracle_decode(q, kc, vc, tables, lens, (16, 1, 128, 16), 0.09)
    assert_attention_close(out, ref, "group 16")
    lens = [100, 700, 768]  # one 768-token partition each: no workspace needed
    q, kc, vc, tables = random_case(lens, 128, 16, 32, 8, seed=15)
    out = torch.full_like(q, float("nan"))
    native.paged_attention_decode(q, kc, vc, torch.as_tensor(tables, device="cuda"),
                                  torch.as_tensor(np.asarray(lens, dtype=np.int32), device="cuda"), 768, 0.09,
                                  out, None, 0)
    torch.cuda.synchronize()
    ref = oracle_decode(q, kc, vc, tables, lens, (32, 8, 128, 16), 0.09)
    assert_attention_close(out, ref, "no workspace")


def test_decode_ex_marks_the_main_kernel_and_changes_nothing():
    """paged_attention_decode_ex records its event between the main kernel and
    the merge; the output is bit for bit paged_attention_decode's."""
    lens = [900, 2500, 37, 1500]
    d, bs, Hq, Hkv = 128, 16, 32, 8
    q, kc, vc, tables = random_case(lens, d, bs, Hq, Hkv, seed=61)
    tables_d = torch.as_tensor(tables, device="cuda")
    lens_d = torch.as_tensor(np.asarray(lens, dtype=np.int32), device="cuda")
    n = native.paged_attention_workspace_size(len(lens), 1, Hq, d, max(lens), 512)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    a = torch.empty_like(q)
    b = torch.empty_like(q)
    native.paged_attention_decode(q, kc, vc, tables_d, lens_d, max(lens), 0.09, a, ws, 512)
    e0, em, e1 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    for e in (e0, em, e1):
        e.record()
    e0.record()
    native.paged_attention_decode(q, kc, vc, tables_d, lens_d, max(lens), 0.09, b, ws, 512, main_done_event=em)
    e1.record()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    t_main, t_all = e0.elapsed_time(em), e0.elapsed_time(e1)
    assert 0 < t_main <= t_all


def test_bad_block_and_length_set_status_without_fault():
    lens = [40, 70]
    d, bs, Hq, Hkv = 128, 16, 8, 2
    q, kc, vc, tables = random_case(lens, d, bs, Hq, Hkv, seed=5)
    scale = 0.1
    bad = tables.copy()
    bad[1, 2] = kc.shape[0] + 5
    st = status_tensor()
    out = run_decode(q, kc, vc, bad, lens, scale, status=st)
    assert st.item() & native.PKV_STATUS_BAD_BLOCK
    assert torch.isfinite(out.float()).all()
    # sequence 0 is untouched by the bad entry of sequence 1
    ref = oracle_decode(q, kc, vc, tables, lens, (Hq, Hkv, d, bs), scale)
    assert_attention_close(out[:1], ref[:1])
    st.zero_()
    too_long = [40, tables.shape[1] * bs + 1]
    run_decode(q, kc, vc, tables, too_long, scale, max_len=max(too_long), status=st)
    assert st.item() & native.PKV_STATUS_BAD_LEN


def test_unwritten_tail_slots_never_leak_nan():
    d, bs, Hq, Hkv = 128, 16, 8, 2
    lens = [17, 3]
    q, kc, vc, tables = random_case(lens, d, bs, Hq, Hkv, seed=8)
    # poison every slot past each sequence's end with NaN bit patterns
    for i, L in enumerate(lens):
        last = tables[i, (L - 1) // bs]
        off = L - ((L - 1) // bs) * bs
        kc[last, :, off:].view(torch.int16).fill_(0x7FC1)
        vc[last, :, off:].view(torch.int16).fill_(0x7FC1)
    out = run_decode(q, kc, vc, tables, lens, 0.09)
    ref = oracle_decode(q, kc, vc, tables, lens, (Hq, Hkv, d, bs), 0.09)
    assert_attention_close(out, ref, "nan tail")


# ------------------------------------------------------------------ workloads
class RecordingAllocator:
    """The native allocator, logging every call and its result so that the same
    calls can be replayed on the oracle allocator afterwards (the oracle never
    enters a product object)."""

    def __init__(self, num_blocks, block_size):
        self.inner = native.BlockAllocator(num_blocks, block_size)
        self.num_blocks, self.block_size = num_blocks, block_size
        self.log = []

    def __getattr__(self, name):
        fn = getattr(self.inner, name)

        def call(*args):
            res = fn(*args)
            self.log.append((name, tuple(list(a) if isinstance(a, range) else a for a in args), res))
            return res
        return call


def _plain(x):
    if x is None:
        return None
    if isinstance(x, tuple):
        return tuple(_plain(v) for v in x)
    return np.asarray(x).astype(np.int64).tolist()


def replay_on_oracle(rec):
    """Every call the native allocator served, again on the oracle allocator:
    each result (slots, copy-on-write pairs, tables, lengths) bit for bit, then
    every refcount and the free count."""
    oa = OracleAllocator(rec.num_blocks, rec.block_size)
    for name, args, res in rec.log:
        want = getattr(oa, name)(*args)
        assert _plain(res) == _plain(want), f"native {name}{args[:2]} differs from the oracle allocator"
    assert rec.inner.num_free() == oa.num_free()
    assert [rec.inner.refcount(b) for b in range(rec.num_blocks)] == oa.refcount
    return oa


def session_step_parity(w, block_size=None, q_len=None, layers=None, check_layers=(0,), prefix_len=None, seed=0,
                        fused=False, planned=False):
    """One full step of a workload on the GPU, on the native allocator and in the
    launch configuration the benchmark times (fused: the new tokens' store inside
    the decode grid; planned: over the host-built work list, as the benchmark's
    single-token step runs it).  The
    allocator's calls are replayed on the oracle allocator, the oracle's write
    and copy run on host copies of the checked layers' caches, and every
    sequence's output on those layers is compared with the fp64 oracle."""
    sess = DecodeSession(w, "cuda", allocator_factory=RecordingAllocator, block_size=block_size, q_len=q_len,
                         layers=layers, extra_steps=1, prefix_len=prefix_len)
    assert isinstance(sess.alloc.inner, native.BlockAllocator)
    pre = {l: (bits(sess.k_caches[l]), bits(sess.v_caches[l])) for l in check_layers}
    st = status_tensor()
    sess.apply_setup_copies(st)
    for l in check_layers:
        cache_ops.block_copy(pre[l][0], pre[l][1], sess.setup_cow_pairs)
    step = sess.plan_step()
    replay_on_oracle(sess.alloc)
    (q, ks, vs), = sess.new_token_tensors(1, seed=w.seed + seed)
    outs = [torch.empty_like(q) for _ in range(sess.layers)]
    ws = sess.workspace(step.max_len)
    sess.run_step(step, q, ks, vs, None, ws, st, per_layer_out=outs, fused=fused, planned=planned)
    torch.cuda.synchronize()
    assert st.item() == 0
    slots = step.slots.cpu().numpy()
    for l in check_layers:
        kh, vh = pre.pop(l)
        cache_ops.write(bits(ks[l]), bits(vs[l]), slots, kh, vh, sess.bs)
        assert np.array_equal(bits(sess.k_caches[l]), kh), "pkv_write / block copy not bit-exact"
        assert np.array_equal(bits(sess.v_caches[l]), vh)
        ref = OA.paged_attention(bits(q), kh, vh, step.host_tables, step.host_lens, num_q_heads=sess.Hq,
                                 num_kv_heads=sess.Hkv, head_dim=sess.d, block_size=sess.bs, scale=sess.scale,
                                 q_len=sess.q_len)
        assert_attention_close(outs[l], ref, f"workload {w.number} layer {l}")
        del kh, vh, ref
    return sess, step


def test_workload_tiny_full():
    session_step_parity(inputs.WORKLOADS[1])


@pytest.mark.parametrize("fused,planned", [(False, False), (True, False), (True, True)])
def test_workload_batched_gqa_whole_batch(fused, planned):
    session_step_parity(inputs.WORKLOADS[2], fused=fused, planned=planned)


@pytest.mark.parametrize("fused,planned", [(False, False), (True, True)])
def test_workload_continuous_batching_whole_batch(fused, planned):
    session_step_parity(inputs.WORKLOADS[3], check_layers=(0, 15, 31), fused=fused, planned=planned)


@pytest.mark.parametrize("fused,planned", [(False, False), (True, True)])
def test_workload_shared_prefix_whole_batch(fused, planned):
    sess, _ = session_step_parity(inputs.WORKLOADS[4], fused=fused, planned=planned)
    assert len(sess.setup_cow_pairs) == 64 * 7


def test_workload_shared_prefix_partial_block_cow():
    w = inputs.WORKLOADS[4]
    sess, _ = session_step_parity(w, prefix_len=2043, seed=1)
    assert len(sess.setup_cow_pairs) == 64 * 7


@pytest.mark.parametrize("bs,q_len", [(16, 1), (32, 1), (16, 16), (32, 16)])
def test_workload_long_context_whole_batch(bs, q_len):
    session_step_parity(inputs.WORKLOADS[5], block_size=bs, q_len=q_len, fused=q_len == 1, planned=q_len == 1)


def test_shared_prefix_layout_equals_private_copies_bit_exact():
    """Refcounted shared blocks and fully private copies give identical bits."""
    w = inputs.WORKLOADS[4]
    sess = DecodeSession(w, "cuda", extra_steps=1)
    sess.apply_setup_copies()
    step = sess.plan_step()
    (q, ks, vs), = sess.new_token_tensors(1, seed=3)
    sess.run_step(step, q, ks, vs, out := torch.empty_like(q), sess.workspace(step.max_len))
    torch.cuda.synchronize()
    # private layout: copy every sequence's blocks to fresh places, one owner each
    kc, vc = sess.k_caches[0], sess.v_caches[0]
    T = step.host_tables
    used = [(i, j) for i in range(sess.B) for j in range(inputs.entries_to_fill(step.host_lens[i], sess.bs))]
    kc2 = torch.empty((len(used) + 1,) + tuple(kc.shape[1:]), dtype=kc.dtype, device="cuda")
    vc2 = torch.empty_like(kc2)
    T2 = np.full_like(T, -1)
    src = torch.as_tensor([T[i, j] for i, j in used], device="cuda", dtype=torch.long)
    kc2[:len(used)] = kc[src]
    vc2[:len(used)] = vc[src]
    for n, (i, j) in enumerate(used):
        T2[i, j] = n
    out2 = run_decode(q, kc2, vc2, T2, step.host_lens, sess.scale, sess.partition_size, step.max_len)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


# ------------------------------------------------------------------ decode with the new token's store
def _newest_slots(tables, lens, bs):
    return np.array([int(tables[i][(n - 1) // bs]) * bs + (n - 1) % bs if n > 0 else -1
                     for i, n in enumerate(lens)], dtype=np.int64)


@pytest.mark.parametrize("d,bs,Hq,Hkv,part", [(128, 16, 32, 8, 256), (64, 32, 16, 4, 0), (128, 128, 32, 2, 512),
                                             (128, 64, 8, 8, 128), (64, 16, 64, 4, 0)])
def test_decode_write_equals_write_then_decode(d, bs, Hq, Hkv, part):
    """paged_attention_decode_write = pkv_write of the newest tokens + single-token
    decode: the same output and cache bits, and the oracle on the written cache."""
    lens = [1, 17, 300, 1025, 64, 2000, 33]
    q, kc, vc, tables = random_case(lens, d, bs, Hq, Hkv, seed=d + bs + Hq)
    B = len(lens)
    slots = _newest_slots(tables, lens, bs)
    slots[4] = -1  # no store for one sequence
    k_new = inputs.randn_bf16((B, Hkv, d), 901, "cuda")
    v_new = inputs.randn_bf16((B, Hkv, d), 902, "cuda")
    slots_d = torch.as_tensor(slots, device="cuda")
    tables_d = torch.as_tensor(np.asarray(tables, dtype=np.int32), device="cuda")
    lens_d = torch.as_tensor(np.asarray(lens, dtype=np.int32), device="cuda")
    max_len = max(lens)
    n = native.paged_attention_workspace_size(B, 1, Hq, d, max_len, part)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
    kc2, vc2 = kc.clone(), vc.clone()
    st = status_tensor()
    native.pkv_write(k_new, v_new, slots_d, kc, vc, st)
    ref_out = torch.empty_like(q)
    native.paged_attention_decode(q, kc, vc, tables_d, lens_d, max_len, 0.09, ref_out, ws, part, st)
    out = torch.empty_like(q)
    native.paged_attention_decode_write(q, k_new, v_new, slots_d, kc2, vc2, tables_d, lens_d, max_len, 0.09, out,
                                        ws, part, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(kc2.view(torch.int16), kc.view(torch.int16))
    assert torch.equal(vc2.view(torch.int16), vc.view(torch.int16))
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    ref = oracle_decode(q, kc2, vc2, tables, lens, (Hq, Hkv, d, bs), 0.09)
    assert_attention_close(out, ref, "decode with the new token's store")


def test_decode_write_reports_a_slot_other_than_the_newest_position():
    d, bs, Hq, Hkv = 128, 16, 32, 8
    lens = [40, 100, 7]
    q, kc, vc, tables = random_case(lens, d, bs, Hq, Hkv, seed=77, spare=8)
    slots = _newest_slots(tables, lens, bs)
    foreign = int(slots[1]) - 3  # a slot of sequence 1 that is not its newest token's
    slots[1] = foreign
    k_new = inputs.randn_bf16((3, Hkv, d), 903, "cuda")
    v_new = inputs.randn_bf16((3, Hkv, d), 904, "cuda")
    before_k = bits(kc)
    st = status_tensor()
    out = torch.empty_like(q)
    native.paged_attention_decode_write(q, k_new, v_new, torch.as_tensor(slots, device="cuda"), kc, vc,
                                        torch.as_tensor(np.asarray(tables, dtype=np.int32), device="cuda"),
                                        torch.as_tensor(np.asarray(lens, dtype=np.int32), device="cuda"), max(lens),
                                        0.09, out, None, 0, st)
    torch.cuda.synchronize()
    assert st.item() & native.PKV_STATUS_BAD_SLOT
    after_k = bits(kc)
    blk, off = divmod(foreign, bs)
    assert np.array_equal(after_k[blk, :, off], before_k[blk, :, off])  # not stored
    for i in (0, 2):  # the other sequences' tokens are stored
        b, o = divmod(int(slots[i]), bs)
        assert np.array_equal(after_k[b, :, o], bits(k_new)[i])


def test_decode_write_on_the_tensor_core_route_equals_write_then_decode():
    """max_seq_len >= 16384 routes single-token decodes to the tensor cores; the
    store then runs as its own launch first, with the same result."""
    d, bs, Hq, Hkv = 128, 32, 64, 8
    lens = [16400, 300, 17000]
    q, kc, vc, tables = random_case(lens, d, bs, Hq, Hkv, seed=88)
    B = len(lens)
    slots = _newest_slots(tables, lens, bs)
    k_new = inputs.randn_bf16((B, Hkv, d), 905, "cuda")
    v_new = inputs.randn_bf16((B, Hkv, d), 906, "cuda")
    slots_d = torch.as_tensor(slots, device="cuda")
    tables_d = torch.as_tensor(np.asarray(tables, dtype=np.int32), device="cuda")
    lens_d = torch.as_tensor(np.asarray(lens, dtype=np.int32), device="cuda")
    n = native.paged_attention_workspace_size(B, 1, Hq, d, max(lens), 512)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
    kc2, vc2 = kc.clone(), vc.clone()
    st = status_tensor()
    native.pkv_write(k_new, v_new, slots_d, kc, vc, st)
    ref_out = torch.empty_like(q)
    native.paged_attention_decode(q, kc, vc, tables_d, lens_d, max(lens), 0.09, ref_out, ws, 512, st)
    out = torch.empty_like(q)
    native.paged_attention_decode_write(q, k_new, v_new, slots_d, kc2, vc2, tables_d, lens_d, max(lens), 0.09, out,
                                        ws, 512, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(kc2.view(torch.int16), kc.view(torch.int16))
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))


# ------------------------------------------------------------------ host-built work list
@pytest.mark.parametrize("d,bs,Hq,Hkv,part", [(128, 16, 32, 8, 768), (64, 32, 16, 4, 256), (128, 128, 32, 2, 512),
                                             (128, 64, 8, 8, 128), (64, 16, 64, 4, 0),
                                             (128, 16, 32, 8, 48)])  # 3-block partitions of 32-row units
def test_decode_items_equals_the_grid_decode_bit_exact(d, bs, Hq, Hkv, part):
    """paged_attention_decode_items (the host-built, longest-first list) gives the
    same bits as paged_attention_decode_write / paged_attention_decode, with and
    without the new tokens' store, and with a grid larger than the list."""
    lens = [1, 17, 300, 1025, 64, 2000, 33, 0, 4000]
    q, kc, vc, tables = random_case(lens, d, bs, Hq, Hkv, seed=d + bs + Hq + 5)
    B = len(lens)
    slots = _newest_slots(tables, lens, bs)
    k_new = inputs.randn_bf16((B, Hkv, d), 911, "cuda")
    v_new = inputs.randn_bf16((B, Hkv, d), 912, "cuda")
    slots_d = torch.as_tensor(slots, device="cuda")
    tables_d = torch.as_tensor(np.asarray(tables, dtype=np.int32), device="cuda")
    lens_d = torch.as_tensor(np.asarray(lens, dtype=np.int32), device="cuda")
    max_len = max(lens)
    n = native.paged_attention_workspace_size(B, 1, Hq, d, max_len, part)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
    items = native.pkv_decode_items(np.asarray(lens, dtype=np.int32), tables, Hkv, bs, part, d)
    count, part = int(items[0, 0]), int(items[0, 1])  # part 0: the size the list chose
    padded = np.zeros((items.shape[0] + 37, 4), dtype=np.int32)  # room for a grid of 37 more CTAs
    padded[:items.shape[0]] = items
    items_d = torch.as_tensor(padded, device="cuda")
    st = status_tensor()
    kc2, vc2 = kc.clone(), vc.clone()
    ref = torch.empty_like(q)
    native.paged_attention_decode_write(q, k_new, v_new, slots_d, kc, vc, tables_d, lens_d, max_len, 0.09, ref, ws,
                                        part, st)
    got = torch.full_like(q, float("nan"))
    native.paged_attention_decode_items(q, k_new, v_new, slots_d, kc2, vc2, tables_d, lens_d, max_len, 0.09, got,
                                        items_d, grid_items=count, workspace=ws, partition_size=part, d_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(kc2.view(torch.int16), kc.view(torch.int16)) and torch.equal(vc2.view(torch.int16),
                                                                                    vc.view(torch.int16))
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    # no store, and a grid of more CTAs than items
    ref2 = torch.empty_like(q)
    native.paged_attention_decode(q, kc, vc, tables_d, lens_d, max_len, 0.09, ref2, ws, part, st)
    got2 = torch.full_like(q, float("nan"))
    native.paged_attention_decode_items(q, None, None, None, kc, vc, tables_d, lens_d, max_len, 0.09, got2, items_d,
                                        grid_items=padded.shape[0] - 1, workspace=ws, partition_size=part,
                                        d_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(got2.view(torch.int16), ref2.view(torch.int16))
    oracle = oracle_decode(q, kc, vc, tables, lens, (Hq, Hkv, d, bs), 0.09)
    assert_attention_close(got2, oracle, "decode over the work list")


def test_decode_items_built_for_other_lengths_is_reported():
    d, bs, Hq, Hkv = 128, 16, 32, 8
    lens = [900, 40, 2000]
    q, kc, vc, tables = random_case(lens, d, bs, Hq, Hkv, seed=97)
    items = native.pkv_decode_items(np.asarray([900, 40, 1990], dtype=np.int32), tables, Hkv, bs, 512, d)
    st = status_tensor()
    out = torch.empty_like(q)
    n = native.paged_attention_workspace_size(3, 1, Hq, d, 2000, 512)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    native.paged_attention_decode_items(q, None, None, None, kc, vc, torch.as_tensor(tables, device="cuda"),
                                        torch.as_tensor(np.asarray(lens, dtype=np.int32), device="cuda"), 2000, 0.09,
                                        out, torch.as_tensor(items, device="cuda"), workspace=ws, partition_size=512,
                                        d_status=st)
    torch.cuda.synchronize()
    assert st.item() & native.PKV_STATUS_BAD_ITEM
    # the sequences the list describes correctly are still right
    ref = oracle_decode(q, kc, vc, tables, lens, (Hq, Hkv, d, bs), 0.09)
    assert_attention_close(out[:2], ref[:2], "sequences the list matches")


def test_decode_items_overlap_across_layers_is_bit_exact():
    """PKV_DECODE_OVERLAP: eight "layers" (own caches, queries, new tokens and
    outputs; shared tables, work list and one workspace) launched back to
    back, each streaming while the one before finishes and writing only after
    it: every layer's output and stored token equal those of the same calls
    without the flag, and a layer matches the oracle."""
    d, bs, Hq, Hkv = 128, 16, 32, 8
    lens = [1, 700, 3000, 2047, 64, 4000, 129, 900] * 4
    B, layers = len(lens), 8
    q0, kc0, _, tables = random_case(lens, d, bs, Hq, Hkv, seed=300)
    NB = kc0.shape[0]
    caches = [(inputs.randn_bf16((NB, Hkv, bs, d), 600 + 2 * l, "cuda"),
               inputs.randn_bf16((NB, Hkv, bs, d), 601 + 2 * l, "cuda")) for l in range(layers)]
    qs = [inputs.randn_bf16(tuple(q0.shape), 700 + l, "cuda") for l in range(layers)]
    knew = [inputs.randn_bf16((B, Hkv, d), 400 + l, "cuda") for l in range(layers)]
    vnew = [inputs.randn_bf16((B, Hkv, d), 500 + l, "cuda") for l in range(layers)]
    slots_d = torch.as_tensor(_newest_slots(tables, lens, bs), device="cuda")
    tables_d = torch.as_tensor(np.asarray(tables, dtype=np.int32), device="cuda")
    lens_d = torch.as_tensor(np.asarray(lens, dtype=np.int32), device="cuda")
    items = native.pkv_decode_items(np.asarray(lens, dtype=np.int32), tables, Hkv, bs, 1024, d)
    items_d = torch.as_tensor(items, device="cuda")
    part = int(items[0, 1])
    max_len = max(lens)
    ws = torch.empty(native.paged_attention_workspace_size(B, 1, Hq, d, max_len, part), dtype=torch.uint8,
                     device="cuda")
    st = status_tensor()

    def run(overlap):
        kcs = [(kc.clone(), vc.clone()) for kc, vc in caches]
        outs = [torch.full_like(qs[0], float("nan")) for _ in range(layers)]
        for l in range(layers):
            native.paged_attention_decode_items(qs[l], knew[l], vnew[l], slots_d, kcs[l][0], kcs[l][1], tables_d,
                                                lens_d, max_len, 0.09, outs[l], items_d, workspace=ws,
                                                partition_size=part, d_status=st, overlap=overlap)
        torch.cuda.synchronize()
        return kcs, outs

    ref_c, ref_o = run(False)
    for _ in range(3):
        got_c, got_o = run(True)
        assert st.item() == 0
        for l in range(layers):
            assert torch.equal(got_o[l].view(torch.int16), ref_o[l].view(torch.int16)), f"layer {l}"
            assert torch.equal(got_c[l][0].view(torch.int16), ref_c[l][0].view(torch.int16))
            assert torch.equal(got_c[l][1].view(torch.int16), ref_c[l][1].view(torch.int16))
    ref = oracle_decode(qs[3], got_c[3][0], got_c[3][1], tables, lens, (Hq, Hkv, d, bs), 0.09)
    assert_attention_close(got_o[3], ref, "an overlapped layer against the oracle")
