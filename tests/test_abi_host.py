"""The C-ABI library builds, loads and exports every declared symbol; host-side
argument checks and the host allocator work without a GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

from conftest import ROOT, read_golden

HEADER = os.path.join(ROOT, "include", "pkv.h")


@pytest.fixture(scope="module")
def native():
    from paged_kv_cache_276_gb300 import build, native
    build.build()
    return native


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(p[a-z_]+)\s*\(", text)) - {"pkv_bf16"})


def test_every_declared_symbol_is_exported(native):
    names = declared_functions()
    assert "paged_attention_decode" in names and "pkv_write" in names and "pkv_block_copy" in names
    lib = native.lib()
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"
    assert set(names) == set(native.SIGNATURES), "binding signatures out of sync with the header"


def test_error_strings(native):
    assert native.error_string(0) == "ok"
    assert "shared" in native.error_string(native.PKV_ERR_SHARED)


def test_workspace_size_host_only(native):
    f = native.paged_attention_workspace_size
    assert f(32, 1, 32, 128, 512, 512) == 0          # one partition: no scratch
    n = f(32, 1, 32, 128, 4096, 512)
    assert n >= 32 * 32 * 8 * 128 * 4 + 32 * 32 * 8 * 8
    assert f(16, 16, 64, 128, 32768, 512) > f(16, 1, 64, 128, 32768, 512)
    assert f(-1, 1, 1, 64, 1, 0) == 0


def test_decode_rejects_bad_sizes_before_launch(native):
    lib = native.lib()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: every case fails validation first
    args = dict(q=fake, k=fake, v=fake, tbl=fake, maxb=4, lens=fake, B=2, maxlen=64, qlen=1, Hq=8, Hkv=2,
                d=128, bs=16, NB=8, scale=0.1, part=0, out=fake, ws=None, wsb=0, st=None, stream=None)

    def call(**kw):
        a = dict(args, **kw)
        return lib.paged_attention_decode(a["q"], a["k"], a["v"], a["tbl"], a["maxb"], a["lens"], a["B"],
                                          a["maxlen"], a["qlen"], a["Hq"], a["Hkv"], a["d"], a["bs"], a["NB"],
                                          a["scale"], a["part"], a["out"], a["ws"], a["wsb"], a["st"],
                                          a["stream"])
    assert call(d=96) == native.PKV_ERR_UNSUPPORTED
    assert call(bs=8) == native.PKV_ERR_UNSUPPORTED
    assert call(bs=256) == native.PKV_ERR_UNSUPPORTED
    assert call(qlen=3) == native.PKV_ERR_UNSUPPORTED
    assert call(Hq=7) == native.PKV_ERR_ARG
    assert call(Hq=40, Hkv=2) == native.PKV_ERR_UNSUPPORTED       # group 20 > 16
    assert call(qlen=16, Hq=32, Hkv=2) == native.PKV_ERR_UNSUPPORTED  # 16 x 16 rows > 128
    assert call(part=24) == native.PKV_ERR_ARG                   # not a multiple of the block
    assert call(maxlen=4096) == native.PKV_ERR_WORKSPACE          # 8 partitions, no scratch
    assert call(scale=float("nan")) == native.PKV_ERR_ARG
    assert call(q=ctypes.c_void_p((1 << 20) + 2)) == native.PKV_ERR_ARG  # misaligned
    assert call(B=0) == native.PKV_OK                            # nothing to do, nothing launched


def test_static_scratch_decode_gives_the_regular_error_codes(native):
    """The allocation-free decode checks its arguments the way paged_attention_decode
    does before it compares the scratch need with its fixed array."""
    lib = native.lib()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: every case fails validation first
    args = dict(q=fake, k=fake, v=fake, tbl=fake, maxb=4, lens=fake, B=2, maxlen=64, qlen=1, Hq=8, Hkv=2,
                d=128, bs=16, NB=8, scale=0.1, part=0, out=fake)

    def regular(**kw):
        a = dict(args, **kw)
        return lib.paged_attention_decode(a["q"], a["k"], a["v"], a["tbl"], a["maxb"], a["lens"], a["B"],
                                          a["maxlen"], a["qlen"], a["Hq"], a["Hkv"], a["d"], a["bs"], a["NB"],
                                          a["scale"], a["part"], a["out"], None, 0, None, None)

    def static(**kw):
        a = dict(args, **kw)
        return lib.paged_attention_decode_static_scratch(a["q"], a["k"], a["v"], a["tbl"], a["maxb"], a["lens"],
                                                         a["B"], a["maxlen"], a["qlen"], a["Hq"], a["Hkv"], a["d"],
                                                         a["bs"], a["NB"], a["scale"], a["part"], a["out"], None,
                                                         None)
    # each of these also asks for far more scratch than the array holds
    big = dict(maxlen=1 << 19, part=16)
    cases = [dict(d=96), dict(bs=8), dict(qlen=3), dict(qlen=0), dict(Hq=7), dict(Hq=40, Hkv=2),
             dict(qlen=16, Hq=32, Hkv=2), dict(part=24), dict(scale=float("nan")), dict(NB=0),
             dict(q=ctypes.c_void_p((1 << 20) + 2)), dict(tbl=None)]
    for kw in cases:
        want = regular(**kw)
        assert want not in (native.PKV_OK, native.PKV_ERR_WORKSPACE), kw
        assert static(**kw) == want, kw
        assert static(**{**big, **kw}) == want, kw
    assert static(**big) == native.PKV_ERR_WORKSPACE
    assert static(B=0, **big) == native.PKV_OK  # nothing to do, nothing launched


def test_prefill_rejects_bad_sizes_before_launch(native):
    lib = native.lib()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: every case fails validation first
    args = dict(q=fake, k=fake, v=fake, tbl=fake, maxb=4, lens=fake, qs=fake, B=2, T=40, Hq=64, Hkv=8,
                d=128, bs=16, NB=8, scale=0.1, out=fake, st=None, stream=None)

    def call(**kw):
        a = dict(args, **kw)
        return lib.paged_attention_prefill(a["q"], a["k"], a["v"], a["tbl"], a["maxb"], a["lens"], a["qs"],
                                           a["B"], a["T"], a["Hq"], a["Hkv"], a["d"], a["bs"], a["NB"],
                                           a["scale"], a["out"], a["st"], a["stream"])
    assert call(d=96) == native.PKV_ERR_UNSUPPORTED               # tensor-core tiles: head dim 64 or 128
    assert call(bs=8) == native.PKV_ERR_UNSUPPORTED
    assert call(bs=256) == native.PKV_ERR_UNSUPPORTED
    assert call(Hq=24, NB=0) == native.PKV_ERR_ARG                # group 3 passes the shape checks
    assert call(Hq=64, Hkv=2) == native.PKV_ERR_UNSUPPORTED       # group 32 > 16
    assert call(Hq=7, Hkv=2) == native.PKV_ERR_ARG
    assert call(B=1025) == native.PKV_ERR_UNSUPPORTED
    assert call(T=-1) == native.PKV_ERR_ARG
    assert call(scale=float("inf")) == native.PKV_ERR_ARG
    assert call(qs=None) == native.PKV_ERR_ARG
    assert call(out=ctypes.c_void_p((1 << 20) + 8)) == native.PKV_ERR_ARG  # misaligned
    assert call(qs=ctypes.c_void_p((1 << 20) + 2)) == native.PKV_ERR_ARG
    assert call(NB=0) == native.PKV_ERR_ARG
    assert call(B=0) == native.PKV_OK                             # nothing to do, nothing launched
    assert call(T=0) == native.PKV_OK


def test_write_and_copy_reject_bad_sizes_before_launch(native):
    lib = native.lib()
    fake = ctypes.c_void_p(1 << 20)
    assert lib.pkv_write(fake, fake, fake, 4, fake, fake, 8, 16, 2, 12, None, None) == native.PKV_ERR_ARG
    assert lib.pkv_write(fake, fake, fake, 0, fake, fake, 8, 16, 2, 64, None, None) == native.PKV_OK
    assert lib.pkv_write(None, fake, fake, 4, fake, fake, 8, 16, 2, 64, None, None) == native.PKV_ERR_ARG
    assert lib.pkv_block_copy(fake, fake, fake, -1, 8, 16, 2, 64, None, None) == native.PKV_ERR_ARG
    assert lib.pkv_block_copy(fake, fake, fake, 0, 8, 16, 2, 64, None, None) == native.PKV_OK


# ------------------------------------------------------------- allocator
def test_native_allocator_page_examples(native):
    for length, block, blocks, _cap, unused, used_last, _o in read_golden("block_counts.txt"):
        a = native.BlockAllocator(16, int(block))
        a.seq_add(7)
        slots = a.seq_append(7, int(length))
        table, lens = a.block_table([7], 8)
        nb = int((table[0] >= 0).sum())
        assert nb == int(blocks) and lens[0] == int(length)
        assert nb * int(block) - int(length) == int(unused)
        assert int((slots // int(block) == table[0, nb - 1]).sum()) == int(used_last)
        assert table[0, 0] == 0  # LIFO stack starts with block 0 on top


def _kind(code):
    from paged_kv_cache_276_gb300 import native
    return {native.PKV_ERR_ARG: "arg", native.PKV_ERR_OOM: "oom", native.PKV_ERR_RANGE: "range",
            native.PKV_ERR_SHARED: "shared"}[code]


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_native_allocator_matches_oracle_bit_exact(native, seed):
    """Same random sequence of add / append / fork / cow / free on both; every table, length,
    refcount, free count, slot list and error kind must agree."""
    from oracle.allocator import AllocError, OracleAllocator
    rng = np.random.default_rng(seed)
    NB, bs = 48, [4, 16, 8, 32][seed]
    na = native.BlockAllocator(NB, bs)
    oa = OracleAllocator(NB, bs)
    live = []
    next_id = 0
    for step in range(600):
        op = rng.choice(["add", "append", "append", "fork", "cow", "free", "bad", "swap_out", "swap_in"])
        ids = list(oa.seqs)
        res_o = res_n = None
        err_o = err_n = None
        if op == "add" or not ids:
            sid = next_id if rng.random() > 0.05 or not ids else ids[0]  # sometimes a duplicate
            next_id += 1
            try:
                oa.seq_add(sid)
            except AllocError as e:
                err_o = e.kind
            try:
                na.seq_add(sid)
            except native.PkvError as e:
                err_n = _kind(e.code)
        elif op == "append":
            sid = int(rng.choice(ids))
            n = int(rng.integers(0, 3 * bs))
            try:
                res_o = oa.seq_append(sid, n)
            except AllocError as e:
                err_o = e.kind
            try:
                res_n = list(na.seq_append(sid, n))
            except native.PkvError as e:
                err_n = _kind(e.code)
        elif op == "fork":
            sid = int(rng.choice(ids))
            child = next_id
            next_id += 1
            try:
                oa.seq_fork(sid, child)
            except AllocError as e:
                err_o = e.kind
            try:
                na.seq_fork(sid, child)
            except native.PkvError as e:
                err_n = _kind(e.code)
        elif op == "cow":
            sid = int(rng.choice(ids))
            nb = len(oa.seqs[sid]["blocks"])
            logical = -1 if rng.random() < 0.5 or nb == 0 else int(rng.integers(0, nb + 1))
            try:
                res_o = oa.seq_cow(sid, logical)
            except AllocError as e:
                err_o = e.kind
            try:
                res_n = na.seq_cow(sid, logical)
            except native.PkvError as e:
                err_n = _kind(e.code)
        elif op == "free":
            sid = int(rng.choice(ids))
            oa.seq_free(sid)
            na.seq_free(sid)
        elif op in ("swap_out", "swap_in"):
            sid = int(rng.choice(ids))
            f_o = oa.seq_swap_out if op == "swap_out" else oa.seq_swap_in
            f_n = na.seq_swap_out if op == "swap_out" else na.seq_swap_in
            try:
                res_o = f_o(sid, 64)
            except AllocError as e:
                err_o = e.kind
            try:
                res_n = list(f_n(sid, 64))
            except native.PkvError as e:
                err_n = _kind(e.code)
        else:  # unknown id
            with pytest.raises(AllocError):
                oa.seq_free(10 ** 9)
            with pytest.raises(native.PkvError):
                na.seq_free(10 ** 9)
        assert err_o == err_n, (step, op, err_o, err_n)
        if res_o is not None or res_n is not None:
            assert (list(res_o) if isinstance(res_o, list) else res_o) == \
                (list(res_n) if isinstance(res_n, list) else res_n), (step, op)
        # full state comparison (swapped-out sequences have no table)
        ids = sorted(i for i in oa.seqs if not oa.seqs[i]["swapped"])
        assert na.num_free() == oa.num_free()
        if ids:
            maxb = max(1, max(len(oa.seqs[i]["blocks"]) for i in ids))
            t_o, l_o = oa.block_table(ids, maxb)
            t_n, l_n = na.block_table(ids, maxb)
            assert t_n.tolist() == t_o and l_n.tolist() == l_o
        for b in range(NB):
            assert na.refcount(b) == oa.refcount[b]
        for i in oa.seqs:
            assert na.seq_len(i) == oa.seqs[i]["len"]
        # invariants
        assert sum(oa.refcount) == sum(len(oa.seqs[i]["blocks"]) for i in oa.seqs)
        assert oa.num_free() + sum(1 for r in oa.refcount if r > 0) == NB
    na.close()


def test_native_allocator_oom_leaves_state_unchanged(native):
    a = native.BlockAllocator(4, 16)
    a.seq_add(1)
    a.seq_append(1, 40)  # 3 blocks
    before = (a.block_table([1], 8), a.num_free())
    with pytest.raises(native.PkvError) as e:
        a.seq_append(1, 40)  # needs 3 more, 1 free
    assert e.value.code == native.PKV_ERR_OOM
    after = (a.block_table([1], 8), a.num_free())
    assert np.array_equal(before[0][0], after[0][0]) and before[1] == after[1] and a.seq_len(1) == 40
    with pytest.raises(native.PkvError) as e:
        a.block_table([1], 2)
    assert e.value.code == native.PKV_ERR_RANGE


def test_swapped_sequence_is_refused_until_swapped_back(native):
    a = native.BlockAllocator(8, 16)
    a.seq_add(1)
    a.seq_append(1, 40)  # blocks 0, 1, 2
    a.seq_fork(1, 2)      # shared with sequence 2
    out = a.seq_swap_out(1)
    assert out.tolist() == [0, 1, 2] and a.seq_len(1) == 40 and a.num_free() == 5  # still held by 2
    for call in (lambda: a.seq_append(1, 1), lambda: a.seq_fork(1, 3), lambda: a.seq_cow(1),
                 lambda: a.block_table([1], 8), lambda: a.seq_swap_out(1)):
        with pytest.raises(native.PkvError) as e:
            call()
        assert e.value.code == native.PKV_ERR_ARG
    a.seq_free(2)  # the shared blocks return to the pool
    assert a.num_free() == 8
    back = a.seq_swap_in(1)
    assert len(back) == 3 and a.num_free() == 5
    table, lens = a.block_table([1], 4)
    assert table[0, :3].tolist() == back.tolist() and lens[0] == 40
    with pytest.raises(native.PkvError):
        a.seq_swap_in(1)  # resident again
    a.close()
    b = native.BlockAllocator(2, 16)
    b.seq_add(7)
    b.seq_append(7, 20)
    b.seq_swap_out(7)
    b.seq_add(8)
    b.seq_append(8, 17)
    with pytest.raises(native.PkvError) as e:
        b.seq_swap_in(7)  # needs 2 blocks, none free
    assert e.value.code == native.PKV_ERR_OOM
    b.seq_free(8)
    assert len(b.seq_swap_in(7)) == 2
    b.close()


def test_swap_copies_reject_bad_arguments_before_launch(native):
    lib = native.lib()
    fake = ctypes.c_void_p(1 << 20)
    assert lib.pkv_swap_out(fake, fake, fake, 0, fake, fake, 8, 16, 2, 64, None, None) == native.PKV_OK
    assert lib.pkv_swap_out(fake, fake, fake, -1, fake, fake, 8, 16, 2, 64, None, None) == native.PKV_ERR_ARG
    assert lib.pkv_swap_in(fake, fake, None, 3, fake, fake, 8, 16, 2, 64, None, None) == native.PKV_ERR_ARG
    assert lib.pkv_swap_in(fake, fake, fake, 3, fake, fake, 8, 16, 2, 60, None, None) == native.PKV_ERR_ARG


def test_batched_append_equals_single_appends_and_is_all_or_nothing(native):
    rng = np.random.default_rng(3)
    a = native.BlockAllocator(64, 16)
    b = native.BlockAllocator(64, 16)
    for x in (a, b):
        for i in range(6):
            x.seq_add(i)
            x.seq_append(i, int(rng.integers(0, 40)) if x is a else 0)
    # give b the same lengths as a
    b.close()
    b = native.BlockAllocator(64, 16)
    for i in range(6):
        b.seq_add(i)
        b.seq_append(i, a.seq_len(i))
    ids = [4, 0, 5, 2]
    got = a.seq_append_batch(ids, 3)
    want = np.concatenate([b.seq_append(i, 3) for i in ids])
    assert got.tolist() == want.tolist()
    assert a.block_table(range(6), 8)[0].tolist() == b.block_table(range(6), 8)[0].tolist()
    before = (a.block_table(range(6), 8)[0].copy(), a.num_free())
    for bad in ([1, 1], [1, 99]):
        with pytest.raises(native.PkvError) as e:
            a.seq_append_batch(bad, 2)
        assert e.value.code == native.PKV_ERR_ARG
    with pytest.raises(native.PkvError) as e:
        a.seq_append_batch([0, 1, 2, 3, 4, 5], 200)  # more blocks than free in total
    assert e.value.code == native.PKV_ERR_OOM
    assert np.array_equal(a.block_table(range(6), 8)[0], before[0]) and a.num_free() == before[1]
    a.close()
    b.close()


def test_large_batched_append_rejects_duplicates(native):
    a = native.BlockAllocator(400, 16)
    for i in range(40):
        a.seq_add(i)
    ids = list(range(40))
    with pytest.raises(native.PkvError) as e:
        a.seq_append_batch(ids + [17], 1)  # 41 ids: the sorted check of large batches
    assert e.value.code == native.PKV_ERR_ARG
    assert all(a.seq_len(i) == 0 for i in ids)
    slots = a.seq_append_batch(ids[::-1], 3)
    assert len(set(slots.tolist())) == 120 and all(a.seq_len(i) == 3 for i in ids)
    a.close()


def test_step_layout_host_only(native):
    import ctypes
    B, ql, Hq, Hkv, d, L, mb = 32, 1, 32, 8, 128, 3, 260
    cfg = native.StepConfig(L, B, ql, Hq, Hkv, d, 16, 9000, mb, 768, 0.088, 1)
    lay = native.StepLayout()
    assert native.lib().pkv_step_layout_of(ctypes.byref(cfg), ctypes.byref(lay)) == native.PKV_OK
    up = lambda x: -(-x // 256) * 256  # noqa: E731
    assert lay.q_layer_bytes == up(B * ql * Hq * d * 2) and lay.kv_layer_bytes == up(B * ql * Hkv * d * 2)
    # the segments every layer reads, then each layer's queries, keys and values
    segs = [(lay.slots_offset, B * ql * 8), (lay.tables_offset, B * mb * 4), (lay.lens_offset, B * 4),
            (lay.items_offset, (1 + lay.max_items) * 16)]
    for l in range(L):
        segs += [(lay.q_offset + l * lay.layer_stride, lay.q_layer_bytes),
                 (lay.k_offset + l * lay.layer_stride, lay.kv_layer_bytes),
                 (lay.v_offset + l * lay.layer_stride, lay.kv_layer_bytes)]
    end = 0
    for off, size in segs:  # in order, 256-byte aligned, not overlapping
        assert off % 256 == 0 and off >= end
        end = off + size
    assert lay.stage_bytes >= end and lay.stage_bytes % 256 == 0
    assert lay.layer_stride == lay.q_layer_bytes + 2 * lay.kv_layer_bytes
    # the work list holds every sequence's partitions x KV heads and the merge list
    assert lay.max_items == B * Hkv * -(-(mb * 16) // 768) + -(-B // 4)
    assert lay.out_layer_bytes == lay.q_layer_bytes and lay.out_bytes == L * lay.q_layer_bytes
    assert lay.workspace_bytes == native.paged_attention_workspace_size(B, ql, Hq, d, mb * 16, 768)
    for field, bad in (("num_layers", 0), ("max_seqs", 0), ("q_len", 0), ("block_size", 0),
                       ("max_blocks_per_seq", 0), ("partition_size", -1), ("max_blocks_per_seq", 1 << 28)):
        c = native.StepConfig(L, B, ql, Hq, Hkv, d, 16, 9000, mb, 768, 0.088, 1)
        setattr(c, field, bad)
        assert native.lib().pkv_step_layout_of(ctypes.byref(c), ctypes.byref(lay)) == native.PKV_ERR_ARG
    assert native.lib().pkv_step_layout_of(None, ctypes.byref(lay)) == native.PKV_ERR_ARG


def test_step_create_and_run_reject_bad_arguments_before_any_launch(native):
    import ctypes
    cfg = native.StepConfig(1, 2, 1, 8, 2, 64, 16, 64, 8, 0, 0.1, 1)
    h = ctypes.c_void_p()
    a = native.BlockAllocator(64, 16)
    lib = native.lib()
    arr = (ctypes.c_void_p * 1)(16)
    # null buffers, then a missing workspace (the layout needs one: 128-token tables, 768-token partitions -> 0)
    assert lib.pkv_step_create(ctypes.byref(cfg), a._h, arr, arr, None, None, None, None, None, 0, None,
                               ctypes.byref(h)) == native.PKV_ERR_ARG
    assert lib.pkv_step_create(ctypes.byref(cfg), None, arr, arr, 16, 16, 16, 16, None, 0, None,
                               ctypes.byref(h)) == native.PKV_ERR_ARG
    assert lib.pkv_step_create(ctypes.byref(cfg), a._h, arr, arr, 24, 16, 16, 16, None, 0, None,
                               ctypes.byref(h)) == native.PKV_ERR_ARG   # misaligned
    cfg.partition_size = 16  # 8 partitions: a workspace is needed
    assert lib.pkv_step_create(ctypes.byref(cfg), a._h, arr, arr, 16, 16, 16, 16, None, 0, None,
                               ctypes.byref(h)) == native.PKV_ERR_WORKSPACE
    assert not h.value
    assert lib.pkv_step_run(None, None, 0, None) == native.PKV_ERR_ARG
    assert lib.pkv_step_wait(None) == native.PKV_ERR_ARG
    lib.pkv_step_destroy(None)
    a.close()


def test_decode_write_rejects_bad_arguments_before_launch(native):
    lib = native.lib()
    args = dict(q=16, kn=16, vn=16, slots=16, kc=16, vc=16, tb=16, lens=16)

    def call(**over):
        a = {**args, **over}
        return lib.paged_attention_decode_write(a["q"], a["kn"], a["vn"], a["slots"], a["kc"], a["vc"], a["tb"], 4,
                                                a["lens"], 2, 64, 32, 8, 128, 16, 10, 0.1, 0, 16, None, 0, None, None,
                                                None)
    assert call(kn=None) == native.PKV_ERR_ARG       # no new keys
    assert call(slots=None) == native.PKV_ERR_ARG
    assert call(vn=24) == native.PKV_ERR_ARG         # misaligned
    assert call(slots=12) == native.PKV_ERR_ARG      # int64 slots must be 8-byte aligned
    assert call(q=24) == native.PKV_ERR_ARG


def test_decode_work_list_is_longest_first_and_complete(native):
    """pkv_decode_items: one item per (partition, KV head), longest partition
    first, ties in sequence / partition / head order, with each item's length
    and first physical block; a length-0 sequence gets empty items."""
    lens = np.array([0, 5, 1000, 768], dtype=np.int32)
    tables = np.full((4, 70), -1, dtype=np.int32)
    tables[1, 0] = 7
    tables[2, :63] = np.arange(100, 163)
    tables[3, :48] = np.arange(200, 248)
    items = native.pkv_decode_items(lens, tables, num_kv_heads=2, block_size=16, partition_size=768)
    # header: 10 items, partition 768, one sequence to merge, its list at row 11
    assert items[0].tolist() == [10, 768, 1, 11] and items.shape == (12, 4)

    def it(seq, part, h, L, b0):
        return [seq, h | (part << 16), L, b0]
    want = [it(2, 0, 0, 1000, 100), it(2, 0, 1, 1000, 100),   # 768 tokens
            it(3, 0, 0, 768, 200), it(3, 0, 1, 768, 200),     # 768 tokens
            it(2, 1, 0, 1000, 148), it(2, 1, 1, 1000, 148),   # 232 tokens, from logical block 48
            it(1, 0, 0, 5, 7), it(1, 0, 1, 5, 7),             # 5 tokens
            it(0, 0, 0, 0, -1), it(0, 0, 1, 0, -1)]           # empty: zeros
    assert items[1:11].tolist() == want
    assert items[11].tolist() == [2, -1, -1, -1]  # sequence 2 spans two partitions
    # without tables the first block is unknown (-1)
    assert native.pkv_decode_items(lens, None, 2, 16, 768)[1:11, 3].tolist() == [-1] * 10
    # a length past the table, a partition that is not a multiple of the block, no room
    lib = native.lib()
    n = ctypes.c_int(0)
    buf = np.zeros((11, 4), dtype=np.int32)
    bad = np.array([16 * 70 + 1], dtype=np.int32)
    assert lib.pkv_decode_items(bad.ctypes.data, None, 70, 1, 2, 128, 16, 0, buf.ctypes.data, 10,
                                ctypes.byref(n)) == native.PKV_ERR_RANGE
    assert lib.pkv_decode_items(lens.ctypes.data, None, 70, 4, 2, 128, 16, 24, buf.ctypes.data, 10,
                                ctypes.byref(n)) == native.PKV_ERR_ARG
    assert lib.pkv_decode_items(lens.ctypes.data, None, 70, 4, 2, 128, 16, 768, buf.ctypes.data, 10,
                                ctypes.byref(n)) == native.PKV_ERR_RANGE and n.value == 11  # items + merge row


def test_decode_work_list_chooses_its_partition():
    """partition_size 0: the list is built for one of 768 / 1024 / 1536 / 2048
    tokens, or 3072 / 4096 when the tables share no block (a multiple of the
    block), reported in row 0, and is the list an explicit request for that
    size gives."""
    from paged_kv_cache_276_gb300 import build, native as nat
    build.build()
    rng = np.random.default_rng(4)
    for B, hi, bs in ((32, 4096, 16), (256, 8192, 16), (3, 300, 128), (64, 20000, 32)):
        lens = rng.integers(0, hi, size=B).astype(np.int32)
        mb = -(-hi // bs)
        private = np.arange(B * mb, dtype=np.int32).reshape(B, mb)
        shared = private.copy()
        shared[:, 0] = 7  # every sequence's first block is the same
        for tables, allowed in ((None, (768, 1024, 1536, 2048)), (shared, (768, 1024, 1536, 2048)),
                                (private, (768, 1024, 1536, 2048, 3072, 4096))):
            auto = nat.pkv_decode_items(lens, tables, 8, bs, 0)
            part = int(auto[0, 1])
            assert part in allowed and part % bs == 0
            assert np.array_equal(auto, nat.pkv_decode_items(lens, tables, 8, bs, part))
            assert auto[0, 0] == sum(max(1, -(-int(L) // part)) for L in lens) * 8


def test_decode_items_rejects_bad_arguments_before_launch(native):
    lib = native.lib()
    fake = ctypes.c_void_p(1 << 20)
    base = [fake, None, None, None, fake, fake, fake, 4, fake, 2, 64, 8, 2, 128, 16, 8, 0.1, 0]

    def call(items=fake, grid=3, flags=0, **kw):
        a = list(base)
        for k, v in kw.items():
            a[{"k_new": 1, "slots": 3, "Hq": 11, "d": 13}[k]] = v
        return lib.paged_attention_decode_items(*a, items, grid, fake, None, 0, None, None, None, flags)
    assert call(items=None) == native.PKV_ERR_ARG
    assert call(flags=2) == native.PKV_ERR_ARG                                 # an unknown flag
    assert call(grid=0) == native.PKV_ERR_ARG
    assert call(items=ctypes.c_void_p((1 << 20) + 4)) == native.PKV_ERR_ARG   # items must be 16-byte aligned
    assert call(k_new=fake) == native.PKV_ERR_ARG                             # a store needs k, v and slots
    assert call(d=96) == native.PKV_ERR_UNSUPPORTED
    assert call(Hq=7) == native.PKV_ERR_ARG


def test_split_prefill_sizes_and_argument_checks(native):
    f = native.paged_attention_prefill_workspace_size
    assert f(128, 64, 128, 32768, 0) == 0                     # no split: no workspace
    n = f(128, 64, 128, 32768, 4096)                          # 8 partitions per row
    assert n >= 128 * 64 * 8 * (128 * 4 + 8)
    assert f(128, 64, 128, 32768, 100) == 0                   # not whole 128-key tiles: invalid
    lib = native.lib()
    fake = ctypes.c_void_p(1 << 20)

    def call(part=4096, ws=None, wsb=0, maxlen=32768):
        return lib.paged_attention_prefill_ex(fake, fake, fake, fake, 4, fake, fake, 1, 128, 64, 8, 128, 16, 8, 0.1,
                                              maxlen, part, fake, ws, wsb, None, None)
    assert call(part=100) == native.PKV_ERR_ARG
    assert call(part=-128) == native.PKV_ERR_ARG
    assert call() == native.PKV_ERR_WORKSPACE                  # the split needs its workspace
    assert call(ws=fake, wsb=n - 1) == native.PKV_ERR_WORKSPACE
    assert call(ws=ctypes.c_void_p((1 << 20) + 8), wsb=n) == native.PKV_ERR_WORKSPACE  # misaligned


def _prefill_item_costs(lens, q_start, total_q, Hq, Hkv):
    """Items in the kernel's numbering (per sequence, KV head, pair of query
    tiles or single tile, longest first) and their key tiles."""
    G = Hq // Hkv
    tile_tok = 128 // G
    B = len(lens)
    pairs = total_q >= 2 * tile_tok * B
    span = 2 * tile_tok if pairs else tile_tok
    tiles = []
    for s in range(B):
        c, L = int(q_start[s + 1] - q_start[s]), max(0, int(lens[s]))
        npairs = -(-c // span)
        for _ in range(Hkv):
            for part in range(npairs):
                qt = npairs - 1 - part
                k_hi = min(L, max(0, L - c + min(c, span * (qt + 1))))
                tiles.append(-(-k_hi // 128))
    return np.array(tiles), pairs


@pytest.mark.parametrize("grid", [1, 7, 89, 152])
def test_prefill_items_hand_out_every_item_once(native, grid):
    """pkv_prefill_items: every item of the batch exactly once, each CTA's
    range in order, and the longest-first hand-out keeps every CTA within one
    item of the mean load."""
    rng = np.random.default_rng(grid)
    for Hq, Hkv in ((32, 8), (64, 8), (24, 8)):
        B = 6
        chunks = rng.integers(0, 1500, B)
        lens = chunks + rng.integers(0, 9000, B)
        q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
        total_q = int(q_start[-1])
        w = native.pkv_prefill_items(lens, q_start, total_q, Hq, Hkv, grid)
        tiles, _ = _prefill_item_costs(lens, q_start, total_q, Hq, Hkv)
        n = len(tiles)
        assert w[0] == grid and w[1] == n and len(w) == 3 + grid + n
        off = w[2:3 + grid]
        assert off[0] == 0 and off[-1] == n and np.all(np.diff(off) >= 0)
        items = w[3 + grid:]
        assert sorted(items.tolist()) == list(range(n))
        if n:
            cost = tiles + 2.0  # any positive per-item cost bounds the spread the same way
            loads = [cost[items[off[g]:off[g + 1]]].sum() for g in range(grid)]
            assert max(loads) <= cost.sum() / grid + cost.max() + 1e-9


@pytest.mark.parametrize("grid", [7, 89, 152])
def test_mixed_step_cost_model_prices_the_items_as_the_list_does(native, grid):
    """workloads.prefill_item_costs (the mixed-step grid policy's cost model)
    prices every item as pkv_prefill_items balances it: with those costs each
    CTA's last item went to a least-loaded CTA (the longest-first hand-out's
    invariant), and its key tiles are the kernel's numbering's."""
    from paged_kv_cache_276_gb300 import workloads
    rng = np.random.default_rng(100 + grid)
    for Hq, Hkv in ((32, 8), (64, 8), (24, 8)):
        B = 6
        chunks = rng.integers(0, 1500, B)
        lens = chunks + rng.integers(0, 9000, B)
        q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
        total_q = int(q_start[-1])
        cost = workloads.prefill_item_costs(lens, q_start, total_q, Hq, Hkv)
        tiles, pairs = _prefill_item_costs(lens, q_start, total_q, Hq, Hkv)
        assert len(cost) == len(tiles) and np.all(cost >= tiles * 0.55 + 2.0) and np.all(cost <= tiles + 2.0)
        w = native.pkv_prefill_items(lens, q_start, total_q, Hq, Hkv, grid)
        off, items = w[2:3 + grid], w[3 + grid:]
        loads = np.array([cost[items[off[g]:off[g + 1]]].sum() for g in range(grid)])
        for g in range(grid):
            if off[g + 1] > off[g]:
                assert loads[g] - cost[items[off[g + 1] - 1]] <= loads.min() + 1e-6


def test_mixed_step_grid_is_the_estimates_minimum(native):
    """mixed_prefill_ctas on the mixed workload (256 decodes beside two
    1024-token chunks): at least half the SMs, no estimate below its own."""
    import types
    from paged_kv_cache_276_gb300 import inputs, workloads
    pw = inputs.PREFILL_WORKLOADS["prefill_mixed"]
    lens, chunks = inputs.prefill_shape(pw)
    q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    case = types.SimpleNamespace(lens=lens, chunks=chunks, q_start=q_start, total_q=int(q_start[-1]),
                                 Hq=pw.num_q_heads, Hkv=pw.num_kv_heads, d=pw.head_dim, B=len(lens),
                                 num_decodes=int((chunks == 1).sum()), bs=pw.block_size)
    g = workloads.mixed_prefill_ctas(case)
    assert 76 <= g <= 152
    t = workloads.mixed_step_time(case, g)
    assert all(t <= workloads.mixed_step_time(case, x) for x in range(76, 153, 4))
    # the decodes (up to 4096 tokens) run unsplit beside the chunks
    assert workloads.mixed_decode_partition(case, g) == 4096


def test_prefill_items_rejects_bad_arguments(native):
    lens = np.array([100, 200], dtype=np.int32)
    qs = np.array([0, 50, 150], dtype=np.int32)
    f = native.lib().pkv_prefill_items
    out = np.zeros(64, dtype=np.int32)
    n = ctypes.c_int(0)
    args = lambda **kw: [kw.get("lens", lens.ctypes.data), kw.get("qs", qs.ctypes.data), kw.get("B", 2),
                         kw.get("total_q", 150), kw.get("Hq", 32), kw.get("Hkv", 8), kw.get("grid", 4),
                         out.ctypes.data, kw.get("max_ints", 64), ctypes.byref(n)]
    assert f(*args()) == native.PKV_OK
    assert f(*args(grid=0)) == native.PKV_ERR_ARG
    assert f(*args(Hq=30)) == native.PKV_ERR_ARG
    assert f(*args(Hq=136, Hkv=8)) == native.PKV_ERR_UNSUPPORTED
    assert f(*args(total_q=100)) == native.PKV_ERR_ARG  # q_start past total_q
    bad = np.array([0, 80, 60], dtype=np.int32)
    assert f(*args(qs=bad.ctypes.data)) == native.PKV_ERR_ARG
    assert f(*args(max_ints=5)) == native.PKV_ERR_RANGE and n.value == 3 + 4 + (1 + 2) * 8  # pairs: 1 + 2 per head
