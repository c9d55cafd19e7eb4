"""The decode step runner (pkv_step_*) against the oracle.

Per step the oracle side repeats what the runner does, with its own pieces:
the oracle allocator (same LIFO policy, same initial calls) takes the same
appends, the oracle write stores the step's new keys and values into host
copies of the caches taken before any kernel ran, and the fp64 oracle decodes
over those copies.  The runner's slots, tables and lengths must equal the
oracle allocator's bit for bit; its outputs must be within the attention
tolerance |out - ref| <= 1e-2 + 1e-2 |ref|.  With and without CUDA graphs the
runner enqueues the same kernels on the same data, so their outputs must agree
bit for bit.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import cache_ops
from oracle.allocator import OracleAllocator
from paged_kv_cache_276_gb300 import inputs, native

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


def assert_close(got, ref, what):
    got = got.float().double().numpy()
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside tolerance, max err {err.max():.3e}"


class Case:
    """Native allocator + device caches for the runner, oracle allocator + host
    cache copies for the oracle, built by the same calls."""

    def __init__(self, ids, lens, Hq, Hkv, d, bs, layers, seed, spare=40, max_blocks=None):
        self.ids, self.Hq, self.Hkv, self.d, self.bs, self.layers = list(ids), Hq, Hkv, d, bs, layers
        NB = sum(inputs.entries_to_fill(n, bs) for n in lens) + spare
        self.NB = NB
        self.alloc = native.BlockAllocator(NB, bs)
        self.oalloc = OracleAllocator(NB, bs)
        for sid, n in zip(ids, lens):
            for a in (self.alloc, self.oalloc):
                a.seq_add(sid)
                if n:
                    a.seq_append(sid, int(n))
        self.max_blocks = max_blocks or max(inputs.entries_to_fill(n, bs) for n in lens) + 8
        self.kc = [inputs.randn_bf16((NB, Hkv, bs, d), seed * 10 + 2 * l, "cuda") for l in range(layers)]
        self.vc = [inputs.randn_bf16((NB, Hkv, bs, d), seed * 10 + 2 * l + 1, "cuda") for l in range(layers)]
        self.kc_h = [bits(t) for t in self.kc]
        self.vc_h = [bits(t) for t in self.vc]
        self.seed = seed

    def runner(self, q_len, partition, use_graph, max_seqs=None, scale=0.088):
        self.q_len, self.scale = q_len, scale
        return native.DecodeStep(self.alloc, self.kc, self.vc, max_seqs or len(self.ids), q_len, self.Hq,
                                 self.max_blocks, scale, partition, use_graph=use_graph)

    def step(self, run, ids, s, check=True):
        """Fill the step's inputs, run it, check it against the oracle; returns the outputs."""
        n, ql = len(ids), self.q_len
        base = self.seed * 1000 + 31 * s
        qs = [inputs.randn_bf16((n, ql, self.Hq, self.d), base + 3 * l, "cpu") for l in range(self.layers)]
        ks = [inputs.randn_bf16((n * ql, self.Hkv, self.d), base + 3 * l + 1, "cpu") for l in range(self.layers)]
        vs = [inputs.randn_bf16((n * ql, self.Hkv, self.d), base + 3 * l + 2, "cpu") for l in range(self.layers)]
        for l in range(self.layers):
            run.q(l)[:n].copy_(qs[l])
            run.k(l)[:n * ql].copy_(ks[l])
            run.v(l)[:n * ql].copy_(vs[l])
        run.run(np.asarray(ids, dtype=np.int64))
        run.wait()
        slots_o = np.concatenate([np.asarray(self.oalloc.seq_append(i, ql), dtype=np.int64) for i in ids])
        table_o, lens_o = self.oalloc.block_table(ids, self.max_blocks)
        assert np.array_equal(run.slots[:n * ql].numpy(), slots_o)
        assert np.array_equal(run.tables[:n].numpy(), np.asarray(table_o, dtype=np.int32))
        assert np.array_equal(run.lens[:n].numpy(), np.asarray(lens_o, dtype=np.int32))
        outs = [run.out(l)[:n].clone() for l in range(self.layers)]
        for l in range(self.layers):  # the oracle's caches follow every step
            cache_ops.write(bits(ks[l]), bits(vs[l]), slots_o, self.kc_h[l], self.vc_h[l], self.bs)
        if check:
            for l in range(self.layers):
                ref = OA.paged_attention(bits(qs[l]), self.kc_h[l], self.vc_h[l], table_o, lens_o,
                                         num_q_heads=self.Hq, num_kv_heads=self.Hkv, head_dim=self.d,
                                         block_size=self.bs, scale=self.scale, q_len=ql)
                assert_close(outs[l], ref, f"step {s} layer {l}")
        return outs


@pytest.mark.parametrize("use_graph", [True, False])
def test_runner_matches_oracle_over_steps(use_graph):
    # lengths 255 and 511 cross a 256-token partition boundary on the second
    # step, so the graph path captures a second graph mid-run
    ids = [10, 3, 7, 42, 5, 8]
    case = Case(ids, [1, 17, 255, 511, 1500, 2047], 32, 8, 128, 16, 2, seed=5)
    run = case.runner(1, 256, use_graph)
    try:
        for s in range(4):
            case.step(run, ids, s)
    finally:
        run.close()


def test_graph_and_eager_runners_agree_bit_for_bit():
    ids = list(range(9))
    lens = [1, 40, 700, 768, 769, 1536, 3000, 4095, 12]
    outs = {}
    for use_graph in (True, False):
        case = Case(ids, lens, 32, 8, 128, 16, 1, seed=9)
        run = case.runner(1, 0, use_graph)
        try:
            outs[use_graph] = [case.step(run, ids, s, check=(s == 2))[0] for s in range(3)]
        finally:
            run.close()
    for a, b in zip(outs[True], outs[False]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_subsets_of_the_batch():
    ids = [0, 1, 2, 3, 4, 5, 6, 7]
    case = Case(ids, [100, 200, 300, 400, 500, 600, 700, 800], 16, 4, 64, 32, 1, seed=13)
    run = case.runner(1, 256, True, max_seqs=8)
    try:
        case.step(run, [6, 1, 3], 0)
        case.step(run, ids, 1)
        case.step(run, [6, 1, 3], 2)  # the first graph again
        case.step(run, [2], 3)
    finally:
        run.close()


def test_chunk_of_16_tokens_through_the_runner():
    ids = [0, 1, 2]
    case = Case(ids, [16, 900, 2000], 64, 8, 128, 16, 1, seed=17)
    run = case.runner(16, 128, True)
    try:
        for s in range(2):
            case.step(run, ids, s)
    finally:
        run.close()


def test_runner_errors_change_nothing():
    ids = [0, 1]
    case = Case(ids, [30, 60], 8, 2, 64, 16, 1, seed=21, max_blocks=5)
    run = case.runner(1, 0, True)
    try:
        before = [case.alloc.seq_len(i) for i in ids]
        for bad, code in (([0, 99], native.PKV_ERR_ARG), ([1, 1], native.PKV_ERR_ARG),
                          ([0, 1, 0], native.PKV_ERR_ARG)):
            with pytest.raises(native.PkvError) as e:
                run.run(np.asarray(bad, dtype=np.int64))
            assert e.value.code == code
        assert [case.alloc.seq_len(i) for i in ids] == before
        case.step(run, ids, 0)
        # 5 blocks of 16 hold 80 tokens: sequence 1 (61 tokens now) fills them after 19 more steps
        for s in range(1, 20):
            case.step(run, ids, s, check=(s == 19))
        with pytest.raises(native.PkvError) as e:
            run.run(np.asarray(ids, dtype=np.int64))
        assert e.value.code == native.PKV_ERR_RANGE
        assert case.alloc.seq_len(1) == 80 and case.alloc.seq_len(0) == 50
    finally:
        run.close()


def test_runner_refuses_pageable_host_buffers():
    case = Case([0], [10], 8, 2, 64, 16, 1, seed=23)
    cfg = native.StepConfig(1, 1, 1, 8, 2, 64, 16, case.NB, case.max_blocks, 0, 0.1, 1)
    lay = native.StepLayout()
    assert native.lib().pkv_step_layout_of(ctypes.byref(cfg), ctypes.byref(lay)) == 0
    pageable = torch.empty(lay.stage_bytes + 64, dtype=torch.uint8)
    pinned_out = torch.empty(lay.out_bytes, dtype=torch.uint8).pin_memory()
    dev = torch.empty(lay.stage_bytes + lay.out_bytes + 64, dtype=torch.uint8, device="cuda")
    ws = torch.empty(max(lay.workspace_bytes, 16), dtype=torch.uint8, device="cuda")
    kp = (ctypes.c_void_p * 1)(case.kc[0].data_ptr())
    vp = (ctypes.c_void_p * 1)(case.vc[0].data_ptr())
    h = ctypes.c_void_p()
    off = (-pageable.data_ptr()) % 16
    rc = native.lib().pkv_step_create(ctypes.byref(cfg), case.alloc._h, kp, vp, pageable.data_ptr() + off,
                                      dev.data_ptr(), dev.data_ptr() + lay.stage_bytes, pinned_out.data_ptr(),
                                      ws.data_ptr(), lay.workspace_bytes, None, ctypes.byref(h))
    assert rc == native.PKV_ERR_ARG and not h.value
