"""The allocation-free decode entry point gives the same results as the regular one.

paged_attention_decode_static_scratch serves callers that cannot allocate
device memory (an engine whose device memory is all handed to its own arena at
start-up, or a plugin whose host framework owns every allocation).  It keeps
its split-K scratch in a fixed array inside the library instead of a
caller-provided workspace.  This test calls it through the C ABI twice in a row,
on two different batches that both need the cross-partition scratch, and
compares each output with the regular entry point's on the same inputs, within
the attention tolerance used by the other tests.  Both kernel families write
their partials into the array: the CUDA-core split-K decode (length bound
below 16384) and the tensor-core kernel (single-token decodes with a bound of
16384 or more, and the 16-token causal chunk), each followed by the merge.  It
also checks that a call needing more scratch than the array holds is refused
before launching.

Kept in a file of its own that pytest collects last.
"""
import ctypes

import numpy as np
import pytest
import torch

from paged_kv_cache_276_gb300 import inputs, native

pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 1e-2


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_276_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    return native.lib()


def make_case(lens, seed, Hq=32, Hkv=8, d=128, bs=16, q_len=1):
    rng = np.random.default_rng(seed)
    NB = sum(inputs.entries_to_fill(n, bs) for n in lens) + 4
    tables, _ = inputs.permuted_tables(lens, bs, NB, rng)
    dev = torch.device("cuda:0")
    return dict(
        q=inputs.randn_bf16((len(lens), q_len, Hq, d), seed + 1, dev),
        kc=inputs.randn_bf16((NB, Hkv, bs, d), seed + 2, dev),
        vc=inputs.randn_bf16((NB, Hkv, bs, d), seed + 3, dev),
        tables=torch.as_tensor(tables, device=dev),
        lens=torch.as_tensor(np.asarray(lens, dtype=np.int32), device=dev),
        max_len=int(max(lens)), Hq=Hq, Hkv=Hkv, d=d, bs=bs, NB=NB, q_len=q_len,
        scale=float(np.float32(d ** -0.5)))


def p(t):
    return ctypes.c_void_p(t.data_ptr())


def call_regular(lib, c, partition, out):
    n = lib.paged_attention_workspace_size(len(c["lens"]), c["q_len"], c["Hq"], c["d"], c["max_len"], partition)
    assert 0 < n <= native.STATIC_SCRATCH_BYTES, "the case must need cross-partition scratch that fits the array"
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    rc = lib.paged_attention_decode(p(c["q"]), p(c["kc"]), p(c["vc"]), p(c["tables"]), c["tables"].shape[1],
                                    p(c["lens"]), len(c["lens"]), c["max_len"], c["q_len"], c["Hq"], c["Hkv"], c["d"],
                                    c["bs"], c["NB"], c["scale"], partition, p(out), p(ws), n, None,
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, native.error_string(rc)
    torch.cuda.synchronize()


def call_static(lib, c, partition, out, status=None):
    return lib.paged_attention_decode_static_scratch(
        p(c["q"]), p(c["kc"]), p(c["vc"]), p(c["tables"]), c["tables"].shape[1], p(c["lens"]), len(c["lens"]),
        c["max_len"], c["q_len"], c["Hq"], c["Hkv"], c["d"], c["bs"], c["NB"], c["scale"], partition, p(out),
        None if status is None else p(status), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def check_twice(lib, cases):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for c, partition in cases:  # two calls in a row; the second reuses the array the first filled
        ref = torch.empty_like(c["q"])
        call_regular(lib, c, partition, ref)
        got = torch.full_like(c["q"], float("nan"))
        rc = call_static(lib, c, partition, got, status)
        assert rc == 0, native.error_string(rc)
        torch.cuda.synchronize()
        g = got.float().cpu().double().numpy()
        r = ref.float().cpu().double().numpy()
        assert np.isfinite(g).all()
        assert (np.abs(g - r) <= ATOL + RTOL * np.abs(r)).all()
    assert status.item() == 0


def test_static_scratch_matches_regular_entry_point_twice(lib):
    check_twice(lib, [(make_case([3000, 17, 1200, 4096, 513, 1, 2048, 700], seed=11), 512),
                      (make_case([900, 2500, 40, 1600], seed=23, Hq=64, Hkv=8), 128)])


def test_static_scratch_matches_regular_entry_point_on_the_tensor_core_route(lib):
    """Length bounds of 16384 and more (and 16-token chunks) run the tcgen05
    kernel, whose per-run partials also go to the array."""
    check_twice(lib, [(make_case([20000, 17000], seed=31, Hq=64, Hkv=8), 512),
                      (make_case([16500, 300, 16384], seed=37, Hq=32, Hkv=8, bs=32), 1024),
                      (make_case([5000, 1800], seed=41, Hq=32, Hkv=8, q_len=16), 512)])


def test_static_scratch_refuses_oversized_requests(lib):
    c = make_case([64, 64], seed=5)
    # announce a length bound whose split-K scratch exceeds the array
    B, Hq, d = 2, c["Hq"], c["d"]
    bound = 8192  # 512 partitions of 16 tokens x 64 query rows
    need = lib.paged_attention_workspace_size(B, 1, Hq, d, bound, 16)
    assert need > native.STATIC_SCRATCH_BYTES
    c = dict(c, max_len=bound)
    out = torch.zeros_like(c["q"])
    assert call_static(lib, c, 16, out) == native.PKV_ERR_WORKSPACE
    assert not out.any()  # nothing was launched
