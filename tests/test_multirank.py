"""The benchmark's multi-rank host path on CPU: two ranks over gloo (no GPU).

Every rank runs its own replica batch (weak scaling, no data-path
collective); only the step time is reduced (max over ranks) and the ranks meet
at barriers around the timed region.  The reference arm runs on rank 0 only.
"""
import json
import os
import socket
import sys

import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    from paged_kv_cache_276_gb300 import inputs
    r, w, local = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    try:
        bench.barrier(w)
        step_ms = bench.max_over_ranks(1.0 + 2.0 * r, w)   # the slowest rank's time wins
        bench.barrier(w)
        ref_line = bench.run_reference(type("A", (), {"steps": 1, "warmup": 0})(), r, w) if r != 0 else "rank0"
        # each rank's replica batch, as the benchmark's runner builds it (the
        # rank salts every tensor seed): a checksum of its first cache
        from paged_kv_cache_276_gb300.workloads import DecodeSession
        sess = DecodeSession(inputs.WORKLOADS[1], "cpu", seed_salt=r, extra_steps=2)
        cache_sum = float(sess.k_caches[0].float().abs().sum())
        with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
            json.dump({"rank": r, "world": w, "local": local, "step_ms": step_ms,
                       "ref_line_is_none": ref_line is None, "cache_sum": cache_sum}, f)
    finally:
        dist.destroy_process_group()


def test_two_ranks_over_gloo(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    assert [x["rank"] for x in res] == [0, 1]
    assert all(x["world"] == 2 and x["local"] == x["rank"] for x in res)
    assert all(x["step_ms"] == 3.0 for x in res)         # max over ranks, on every rank
    assert res[1]["ref_line_is_none"]                     # the reference arm prints on rank 0 only
    assert res[0]["cache_sum"] != res[1]["cache_sum"]    # independent replica batches


def test_single_rank_defaults(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.max_over_ranks(4.5, 1) == 4.5
