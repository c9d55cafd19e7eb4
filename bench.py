#!/usr/bin/env python3
"""Benchmark of the paged KV-cache decode hot path on one GB300 (or N replicas).

A step is one pass of the whole hot path over one batch: host allocator work
(block tables, slots, copy-on-write decisions), the store of the new tokens'
keys and values, any ``pkv_block_copy``, and the paged decode (with its
cross-partition combine), for every layer of the workload.

Headline: the continuous-batching mix (256 sequences, log-normal lengths with
median 512, block 16, 32 query / 8 KV heads, head dim 128, bf16, 32 layers with
a block pool each: 128 KiB of cache per token), timed as whole 32-layer steps.
Metric: KV-cache GB/s read (valid K and V rows) per step; query tokens/s
alongside.  The other decode workloads and the chunked-prefill workloads are
reported compactly under "workloads" and "prefill".

``--impl reference`` times the fp64 CPU oracle on a bounded sample of the same
workload instead.  Multi-GPU (torchrun): every rank runs its own independent
replica (weak scaling, no data-path collective); the step time is the max over
ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = 3
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
DEFAULT_PARTITION = 768  # the library's split-K partition when the caller passes 0


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ------------------------------------------------------------------ helpers
def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak():
    """Dense bf16 TFLOP/s: the measured burst figure (a kernel timed on its own)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured burst bf16_tflops"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def _source_sha(parts):
    """sha256 over (file, cut marker or None) parts of csrc: each file up to its
    marker (its host section), whole if the marker is None."""
    csrc = os.path.join(ROOT, "paged_kv_cache_276_gb300", "csrc")
    h = hashlib.sha256()
    for name, marker in parts:
        text = open(os.path.join(csrc, name), "rb").read()
        cut = text.find(marker) if marker else -1
        h.update(text[:cut] if cut >= 0 else text)
    return h.hexdigest()


HOST_MARK = b"// ------------------------------------------------------------------ host"
COMBINE_MARK = b"// ---------------------------------------------- cross-partition combine"
# the device code each traffic record covers (the decode record: decode.cu up to
# its split-K merge kernel, whose code does not change the main kernel's traffic)
TRAFFIC_SOURCES = {
    "decode_kernel_traffic.txt": [("decode.cu", COMBINE_MARK), ("attend.cuh", None), ("ptx.cuh", None)],
    "chunk_tc_kernel_traffic.txt": [("chunk_tc.cu", HOST_MARK), ("tc.cuh", None), ("ptx.cuh", None)],
}


def kernel_traffic(record, workload_tag):
    """DRAM bytes per launch of a kernel from its committed ncu summary under
    profiles/, only while the kernel's device code still hashes to the value the
    capture was taken at (else None)."""
    path = os.path.join(ROOT, "profiles", record)
    try:
        rec = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    rec[k.strip()] = v.strip()
        if rec.get("source_sha256") != _source_sha(TRAFFIC_SOURCES[record]):
            return None
        key = f"dram_bytes_per_launch[{workload_tag}]"
        return float(rec[key]) if key in rec else None
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def gpu_id():
    """nvidia-smi identifier of the current CUDA device (UUID when torch exposes it)."""
    import torch
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    uuid = getattr(props, "uuid", None)
    if uuid:
        u = str(uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [v for v in vis.split(",") if v.strip()]
    return ids[torch.cuda.current_device()] if ids else str(torch.cuda.current_device())


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------- our arm
class Runner:
    """Plans steps, times them on the device and end to end."""

    def __init__(self, wnum, device, rank, block_size=None, q_len=None, steps_needed=8, layers=None):
        import torch
        from paged_kv_cache_276_gb300 import inputs
        from paged_kv_cache_276_gb300.workloads import DecodeSession
        self.torch = torch
        w = inputs.WORKLOADS[wnum]
        self.w = w
        # weak scaling: every rank owns an independent batch of the same shape
        self.sess = DecodeSession(w, device, block_size=block_size, q_len=q_len, extra_steps=steps_needed + 2,
                                  seed_salt=rank, layers=layers)
        self.sess.apply_setup_copies()
        self.device = device
        self.rank = rank

    def plan(self, n):
        steps = self.sess.plan_steps(n)
        toks = self.sess.new_token_tensors(n, seed=self.w.seed + 17 * self.rank)
        return steps, toks

    def layer_call(self, p, q, ks, vs, l, out, ws, status, stream, d0=None, dm=None):
        """One layer of a planned step, as the step runner runs it: the block
        copies of copy-on-write, then (single tokens) the decode with the new
        token's store over the host-built work list, overlapping the layer
        before (independent inputs; not behind this layer's block copies,
        which it reads), or pkv_write and the decode.  d0 is
        recorded right before the decode call; dm is recorded by the library
        right after its main kernel."""
        from paged_kv_cache_276_gb300 import native
        sess = self.sess
        if p.cow_pairs is not None:
            native.pkv_block_copy(sess.k_caches[l], sess.v_caches[l], p.cow_pairs, status, stream)
        if sess.q_len == 1:
            if d0 is not None:
                d0.record(stream)
            native.paged_attention_decode_items(q, ks[l], vs[l], p.slots, sess.k_caches[l], sess.v_caches[l],
                                                p.tables, p.lens, p.max_len, sess.scale, out, p.items, workspace=ws,
                                                partition_size=p.partition, d_status=status, stream=stream,
                                                main_done_event=dm, overlap=p.cow_pairs is None)
        else:
            native.pkv_write(ks[l], vs[l], p.slots, sess.k_caches[l], sess.v_caches[l], status, stream)
            if d0 is not None:
                d0.record(stream)
            native.paged_attention_decode(q, sess.k_caches[l], sess.v_caches[l], p.tables, p.lens, p.max_len,
                                          sess.scale, out, ws, sess.partition_size, status, stream,
                                          main_done_event=dm)

    def time_device(self, warmup, steps, world):
        """Per-step CUDA-event times with an L2 flush before every step (outside
        the events); decode launches timed separately for the roofline."""
        torch = self.torch
        from paged_kv_cache_276_gb300 import native
        sess = self.sess
        plans, toks = self.plan(warmup + steps)
        max_len = max(p.max_len for p in plans)
        ws = sess.workspace(max_len)
        out = torch.empty_like(toks[0][0])
        l2 = torch.cuda.get_device_properties(0).L2_cache_size
        flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=self.device)
        stream = torch.cuda.current_stream()
        status = torch.zeros(1, dtype=torch.int32, device=self.device)
        # every event is created (recorded once) before the timed loop; the
        # library records `dm` itself right after the main decode kernel
        pool = []
        for _ in range((warmup + 2 * steps) * (3 * sess.layers + 2)):
            e = torch.cuda.Event(enable_timing=True)
            e.record(stream)
            pool.append(e)
        ev = pool.pop
        step_ms, dec_ms, main_ms = [], [], []
        launches = 0
        fused = sess.q_len == 1  # single-token decode: the new token's store folded into the decode
        barrier(world)
        torch.cuda.synchronize()
        with ClockSampler(gpu_id()) as clocks:
            for i in range(warmup + steps):
                p = plans[i]
                q, ks, vs = toks[i]
                flush.fill_(float(i))
                s0, s1 = ev(), ev()
                s0.record(stream)
                # no event between the layers: one would make each layer's
                # kernels wait for the previous layer's to finish
                for l in range(sess.layers):
                    self.layer_call(p, q, ks, vs, l, out, ws, status, stream)
                    nparts = math.ceil(p.max_len / (p.partition or DEFAULT_PARTITION)) if p.max_len else 1
                    # (copy,) (write,) decode, cross-partition combine
                    launches += (i >= warmup) * ((1 if fused else 2) + (nparts > 1) + (p.cow_pairs is not None))
                s1.record(stream)
                if i >= warmup:
                    step_ms.append((s0, s1))
            torch.cuda.synchronize()
            # Call pass: the timed steps again (same slots, same values, so the
            # writes change nothing), an event on each side of every layer's
            # decode call (the call's time, with its split-K merge)
            for i in range(warmup, warmup + steps):
                p = plans[i]
                q, ks, vs = toks[i]
                flush.fill_(float(i))
                for l in range(sess.layers):
                    d0, d1 = ev(), ev()
                    self.layer_call(p, q, ks, vs, l, out, ws, status, stream, d0=d0)
                    d1.record(stream)
                    dec_ms.append((d0, d1))
            torch.cuda.synchronize()
            # Main-kernel pass: the timed steps again (same slots, same values,
            # so the writes change nothing), each decode call handed an event
            # that the library records right after its main kernel.  Kept out
            # of the steps above: the event stops the merge kernel from
            # launching early behind the main kernel.
            for i in range(warmup, warmup + steps):
                p = plans[i]
                q, ks, vs = toks[i]
                flush.fill_(float(i))
                for l in range(sess.layers):
                    d0, dm = ev(), ev()
                    self.layer_call(p, q, ks, vs, l, out, ws, status, stream, d0=d0, dm=dm)
                    main_ms.append((d0, dm))
            torch.cuda.synchronize()
        barrier(world)
        if status.item() != 0:
            raise RuntimeError(f"device status {status.item()} during the benchmark")
        step_t = [a.elapsed_time(b) for a, b in step_ms]
        dec_t = [a.elapsed_time(b) for a, b in dec_ms]
        main_t = [a.elapsed_time(b) for a, b in main_ms]
        timed = plans[warmup:]
        kv_bytes = [sess.kv_bytes(p) for p in timed]
        return {
            "ms_per_step": sum(step_t) / len(step_t),
            "step_ms_p10": float(np.percentile(step_t, 10)), "step_ms_p90": float(np.percentile(step_t, 90)),
            "decode_ms_avg": sum(dec_t) / len(dec_t),
            "main_ms_avg": sum(main_t) / len(main_t),
            "kv_bytes_per_step": sum(kv_bytes) / len(kv_bytes),
            "kv_bytes_per_decode": sum(kv_bytes) / len(kv_bytes) / sess.layers,
            "query_tokens_per_step": sess.B * sess.q_len,
            "launches": launches,
            "clocks": clocks.summary(),
        }

    def time_e2e_step(self, steps, use_graph=True):
        """Same metric through the step runner (pkv_step_run: one C call per
        step, the device part one CUDA graph launch when ``use_graph``): the
        allocator append and table fill, the host -> device copy of the step's
        inputs from page-locked memory, the layers' writes and decodes, and the
        device -> host copy of the outputs, all inside the timed region."""
        torch = self.torch
        from paged_kv_cache_276_gb300 import native
        sess = self.sess
        toks = sess.new_token_tensors(1, seed=self.w.seed + 5)
        step = native.DecodeStep(sess.alloc, sess.k_caches, sess.v_caches, sess.B, sess.q_len, sess.Hq,
                                 sess.max_blocks, sess.scale, sess.partition_size, use_graph=use_graph)
        try:
            for l in range(sess.layers):  # one query set for every layer, as the device-timed step
                step.q(l).copy_(toks[0][0].cpu())
                step.k(l).copy_(toks[0][1][l].cpu())
                step.v(l).copy_(toks[0][2][l].cpu())
            seq_ids = np.arange(sess.B, dtype=np.int64)
            stream = torch.cuda.current_stream().cuda_stream  # the raw handle, looked up once
            times, kv = [], []
            for i in range(steps + 1):
                torch.cuda.synchronize()
                t0 = time.perf_counter()
                step.run(seq_ids, stream)
                step.wait()
                t1 = time.perf_counter()
                if i:  # the first pass captures the graph and warms the copy paths
                    times.append((t1 - t0) * 1e3)
                    kv.append(int(step.lens.numpy().astype(np.int64).sum()) * 2 * sess.Hkv * sess.d * 2 * sess.layers)
            return {"ms_per_step": sum(times) / len(times), "kv_bytes_per_step": sum(kv) / len(kv),
                    "h2d": int(step.layout.stage_bytes), "d2h": int(step.layout.out_bytes)}
        finally:
            step.close()


def cpu_oracle_baseline(wnum, budget_s=12.0, reps=None, warmup=0, layers_per_rep=None):
    """The fp64 oracle as it stands, on this host's cores.  A rep decodes the
    whole batch of the workload (every sequence) over ``layers_per_rep`` layers
    (default: all of the workload's layers); the layers of a workload share the
    sequence lengths, so the host keeps one layer's pool and decodes it once per
    layer.  Repeated ``reps`` times, or until ~budget_s seconds have passed."""
    from oracle import attention as OA
    from paged_kv_cache_276_gb300 import inputs
    w = inputs.WORKLOADS[wnum]
    layers = layers_per_rep or w.layers
    rng = inputs.rng_for(w)
    lens = inputs.lengths(w, rng)
    NB = inputs.pool_size(lens, w.block_size, 0.10)
    tables, _ = inputs.permuted_tables(lens, w.block_size, NB, rng)
    shape = (NB, w.num_kv_heads, w.block_size, w.head_dim)
    kb = OA.as_bf16_bits(inputs.randn_bf16(shape, w.seed + 1))
    vb = OA.as_bf16_bits(inputs.randn_bf16(shape, w.seed + 2))
    qb = OA.as_bf16_bits(inputs.randn_bf16((len(lens), 1, w.num_q_heads, w.head_dim), w.seed + 3))
    cores = OA.set_threads(os.cpu_count() or 1)

    def one():
        for _ in range(layers):
            OA.paged_attention(qb, kb, vb, tables, lens, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                               head_dim=w.head_dim, block_size=w.block_size, scale=w.scale)

    for _ in range(warmup):
        one()
    n, t0 = 0, time.perf_counter()
    while True:
        one()
        n += 1
        el = time.perf_counter() - t0
        if (reps is not None and n >= reps) or (reps is None and el >= budget_s):
            break
    kv = int(lens.astype(np.int64).sum()) * 2 * w.num_kv_heads * w.head_dim * 2 * layers
    what = "whole decode steps" if layers == w.layers else f"samples of {layers} of the {w.layers} layer decodes"
    return {"value": kv * n / el / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} {what} of all {len(lens)} sequences ({int(lens.sum())} tokens) in {el:.1f} s, fp64",
            "seconds": el, "reps": n, "query_tok_s": len(lens) * n * layers / w.layers / el}


def workload_desc(wnum, bs=None, q_len=None, layers=None):
    from paged_kv_cache_276_gb300 import inputs
    w = inputs.WORKLOADS[wnum]
    bs = bs or w.block_size
    q_len = q_len or w.q_len
    layers = layers or w.layers
    lens = {1: "L=[17,33,64]", 2: "L~U{1..4096}", 3: "L=lognormal(median 512, sigma 1) clip [1,8192]",
            4: "2048 shared prefix + U{0..512} suffix", 5: "L=32768"}[wnum]
    return (f"{w.name}: {w.num_seqs} seqs, {lens}, block {bs}, {w.num_q_heads}q/{w.num_kv_heads}kv heads, "
            f"d {w.head_dim}, {layers} layer(s), q_len {q_len}, bf16")


NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal


def run_ours(args, rank, world, local):
    import torch
    from paged_kv_cache_276_gb300 import build
    build.build()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    peak, peak_kind = measured_hbm_peak()

    e2e_steps = max(3, min(args.steps, 10))
    r = Runner(HEADLINE, device, rank, steps_needed=args.warmup + args.steps + 2 * (e2e_steps + 1) + 8,
               layers=args.layers)
    dev_res = r.time_device(args.warmup, args.steps, world)
    ms = max_over_ranks(dev_res["ms_per_step"], world)
    total_bytes = dev_res["kv_bytes_per_step"] * world
    value = total_bytes / (ms * 1e-3) / 1e9

    def e2e_gbs(res):
        t = max_over_ranks(res["ms_per_step"], world)
        return res["kv_bytes_per_step"] * world / (t * 1e-3) / 1e9, t

    e2e = r.time_e2e_step(e2e_steps, use_graph=False)
    e2e_value, e2e_ms = e2e_gbs(e2e)
    e2e_graph, e2e_graph_ms = e2e_gbs(r.time_e2e_step(e2e_steps, use_graph=True))
    # the dominant kernel: the decode's main kernel, timed from an event before
    # the call to the event the library records right after it
    main_gbs = dev_res["kv_bytes_per_decode"] / (dev_res["main_ms_avg"] * 1e-3) / 1e9
    op_gbs = dev_res["kv_bytes_per_decode"] / (dev_res["decode_ms_avg"] * 1e-3) / 1e9
    layers = r.sess.layers
    del r
    torch.cuda.empty_cache()
    line = {
        "metric": "paged decode attention KV-cache read bandwidth (valid K+V bytes / step time)",
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16 K/V/Q, seeded lengths and block placement)",
        "config": {"workload": workload_desc(HEADLINE, layers=layers),
                   "parallelism": f"replicas x{world} (independent batches)",
                   "l2": "flushed before every step (write of 2x L2), outside the events",
                   "kv_bytes_per_step": int(dev_res["kv_bytes_per_step"]),
                   "query_tokens_per_step": dev_res["query_tokens_per_step"]},
        "query_tok_s": round(dev_res["query_tokens_per_step"] * world / (ms * 1e-3), 1),
        "roofline": {"bound": "hbm", "achieved": round(main_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(main_gbs / peak, 4), "peak_kind": f"{peak_kind} hbm_gbs",
                     "traffic": kernel_traffic("decode_kernel_traffic.txt", "continuous_batching"),
                     "kernel": "decode_kernel", "bytes_per_launch": int(dev_res["kv_bytes_per_decode"]),
                     "ms_per_launch": round(dev_res["main_ms_avg"], 5),
                     "frac_of_nominal": round(main_gbs / NOMINAL_HBM_GBS, 4),
                     "call_frac": round(op_gbs / peak, 4)},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": e2e["h2d"],
                "d2h_bytes_per_step": e2e["d2h"], "ms_per_step": round(e2e_ms, 4),
                "graph_value": round(e2e_graph, 2), "graph_ms_per_step": round(e2e_graph_ms, 4)},
        "gpu_launches": dev_res["launches"],
        "clocks": dev_res["clocks"],
    }
    if not args.no_workloads:
        line["workloads"] = other_workloads(args, device, rank, world, peak)
        line["prefill"] = prefill_bench(device, cpu=rank == 0 and world == 1 and not args.no_cpu_baseline,
                                        compact=True)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            cb = cpu_oracle_baseline(HEADLINE, budget_s=args.cpu_seconds, layers_per_rep=1)
            line["cpu_baseline"] = {k: (round(v, 4) if k == "value" else v) for k, v in cb.items()
                                    if k in ("value", "unit", "cores", "kind", "sample")}
        except Exception as e:  # reported, never fatal
            line["cpu_baseline"] = {"error": repr(e)}
    return line


WORKLOAD_CASES = [(1, None, None), (2, None, None), (4, None, None), (5, 16, None), (5, 32, None), (5, 16, 16),
                  (5, 32, 16), (3, None, None)]


def case_tag(wnum, bs, q_len):
    return f"w{wnum}" + (f"_bs{bs}" if bs else "") + (f"_q{q_len}" if q_len else "")


def other_workloads(args, device, rank, world, peak, only=None):
    """The other decode workloads, a few numbers each: step time and KV GB/s,
    the decode kernel's and the whole decode call's fraction of the HBM peak,
    and query tokens/s.  The headline workload is timed again only when named."""
    res = {}
    for wnum, bs, q_len in WORKLOAD_CASES:
        tag = case_tag(wnum, bs, q_len)
        if (only is None and wnum == HEADLINE) or (only is not None and tag != only):
            continue
        try:
            steps = 5 if wnum == 3 else 10
            layers = args.layers if wnum == 3 else None
            r = Runner(wnum, device, rank, block_size=bs, q_len=q_len, steps_needed=steps + 3, layers=layers)
            d = r.time_device(3, steps, world)
            ms = max_over_ranks(d["ms_per_step"], world)
            dec = d["kv_bytes_per_decode"] / (d["main_ms_avg"] * 1e-3) / 1e9
            op = d["kv_bytes_per_decode"] / (d["decode_ms_avg"] * 1e-3) / 1e9
            res[tag] = {"ms": round(ms, 5), "gbs": round(d["kv_bytes_per_step"] * world / (ms * 1e-3) / 1e9, 1),
                        "kernel_frac": round(dec / peak, 4), "call_frac": round(op / peak, 4),
                        "tok_s": round(d["query_tokens_per_step"] * world / (ms * 1e-3), 1)}
            if only is not None:  # a profiling run: the long form
                res[tag].update(workload=workload_desc(wnum, bs, q_len, layers), kernel_gbs=round(dec, 1),
                                kernel_ms=round(d["main_ms_avg"], 5), call_ms=round(d["decode_ms_avg"], 5),
                                clocks=d["clocks"])
            del r
            import torch
            torch.cuda.empty_cache()
        except Exception as e:
            res[tag] = {"error": repr(e)}
            log(f"workload {tag} failed: {e!r}")
    return res


def block_sweep(device, peak):
    """Block-size trade-off: decode bandwidth at block 16/32/64/128 on the
    batched and mixed length distributions (one layer each), and the memory
    simulation (paged at block 8..128 versus one contiguous reservation per
    request) on request streams drawn from the same distributions."""
    import torch
    from paged_kv_cache_276_gb300 import inputs, waste
    out = {"decode": {}, "memory": {}}
    for wnum in (2, 3):
        for bs in (16, 32, 64, 128):
            tag = f"w{wnum}_bs{bs}"
            try:
                r = Runner(wnum, device, 0, block_size=bs, steps_needed=16, layers=1)
                d = r.time_device(3, 10, 1)
                main = d["kv_bytes_per_decode"] / (d["main_ms_avg"] * 1e-3) / 1e9
                call = d["kv_bytes_per_decode"] / (d["decode_ms_avg"] * 1e-3) / 1e9
                out["decode"][tag] = {"decode_kernel_gbs": round(main, 1), "frac": round(main / peak, 4),
                                      "decode_call_gbs": round(call, 1), "call_frac": round(call / peak, 4)}
                del r
                torch.cuda.empty_cache()
            except Exception as e:
                out["decode"][tag] = {"error": repr(e)}
    for wnum, n, reserve in ((2, 256, 4096), (3, 512, 8192)):
        w = inputs.WORKLOADS[wnum]
        rng = np.random.default_rng(w.seed + 31)
        finals = np.concatenate([inputs.lengths(w, rng) for _ in range(-(-n // w.num_seqs))])[:n]
        prompts, finals = waste.request_stream(finals, rng)
        cap = 16 * reserve
        rows = {}
        c = waste.simulate(prompts, finals, cap, "contiguous", reserve=reserve)
        rows["contiguous"] = c
        for bs in (8, 16, 32, 64, 128):
            rows[f"paged_bs{bs}"] = waste.simulate(prompts, finals, cap, "paged", block_size=bs)
        out["memory"][f"w{wnum}"] = {
            "requests": n, "capacity_tokens": cap, "contiguous_reservation": reserve,
            **{k: {"token_state_fraction": round(v.token_state_fraction, 4), "utilisation": round(v.utilisation, 4),
                   "mean_running": round(v.mean_running, 2), "tokens_per_step": round(v.tokens_per_step, 2),
                   "steps": v.steps, "preemptions": v.preemptions} for k, v in rows.items()}}
    return out


def swap_bench(device):
    """Bandwidth of pkv_swap_out / pkv_swap_in: whole blocks (block 16, 8 KV
    heads, head dim 128: 64 KiB of K and V each) between a device pool and
    page-locked host buffers, CUDA events around each call, 2 x L2 of cache
    flushed before each."""
    import torch
    from paged_kv_cache_276_gb300 import inputs, native
    NB, Hkv, bs, d = 8192, 8, 16, 128
    kc = inputs.randn_bf16((NB, Hkv, bs, d), 5, device)
    vc = inputs.randn_bf16((NB, Hkv, bs, d), 6, device)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=device)
    res = {}
    for n in (256, 2048):
        ids = torch.as_tensor(np.random.default_rng(n).permutation(NB)[:n].astype(np.int32), device=device)
        hk = torch.empty((n, Hkv, bs, d), dtype=torch.bfloat16).pin_memory()
        hv = torch.empty_like(hk).pin_memory()
        nbytes = 2 * n * Hkv * bs * d * 2
        for name, call in (("out", lambda: native.pkv_swap_out(kc, vc, ids, hk, hv)),
                           ("in", lambda: native.pkv_swap_in(hk, hv, ids, kc, vc))):
            for _ in range(3):
                call()
            ts = []
            for _ in range(10):
                flush.fill_(1.0)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                call()
                e1.record()
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1))
            ms = float(np.median(ts))
            res[f"{name}_{n}_blocks"] = {"bytes": nbytes, "ms": round(ms, 4), "gbs": round(nbytes / ms / 1e6, 1)}
    return res


def prefill_cpu_baseline(case, rows=16, max_seqs=8):
    """The fp64 oracle as it stands on this host's cores, on a bounded sample of a
    prefill workload: the last ``rows`` query rows of the chunks of up to
    ``max_seqs`` sequences (those rows see the most keys), in TFLOP/s of the
    same algorithmic count as the kernel's."""
    from oracle import attention as OA
    seqs = [i for i in range(case.B) if int(case.chunks[i]) >= rows][:max_seqs]
    if not seqs:
        return {"error": "no chunk of that many rows"}
    kb, vb = OA.as_bf16_bits(case.k_cache), OA.as_bf16_bits(case.v_cache)
    qall = OA.as_bf16_bits(case.q)
    q = np.stack([qall[int(case.q_start[i]) + int(case.chunks[i]) - rows:int(case.q_start[i]) + int(case.chunks[i])]
                  for i in seqs])
    lens = case.lens[seqs]
    cores = OA.set_threads(os.cpu_count() or 1)
    t0 = time.perf_counter()
    OA.paged_attention(q, kb, vb, case.tables[seqs], lens, num_q_heads=case.Hq, num_kv_heads=case.Hkv,
                       head_dim=case.d, block_size=case.bs, scale=case.scale, q_len=rows)
    el = time.perf_counter() - t0
    keys = sum(rows * int(L) - rows * (rows - 1) // 2 for L in lens)
    fl = 4 * case.d * case.Hq * keys
    return {"value": fl / el / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"the last {rows} query rows of {len(seqs)} sequences' chunks ({fl / 1e9:.1f} GFLOP) in "
                      f"{el:.2f} s, fp64, OpenMP over (sequence, KV head)", "seconds": el}


def prefill_bench(device, steps=10, warmup=3, only=None, cpu=False, compact=False):
    """Chunked prefill (paged_attention_prefill) on the prefill workloads: a
    step is the chunk's pkv_write plus the attention call; the attention call
    is also timed alone (the tensor-core roofline).  2 x L2 is written before
    every step, outside the events."""
    import torch
    from paged_kv_cache_276_gb300 import inputs
    from paged_kv_cache_276_gb300.workloads import PrefillCase
    peak, peak_kind = measured_tensor_peak()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream()
    res = {}
    for tag, pw in inputs.PREFILL_WORKLOADS.items():
        if only is not None and tag != only:
            continue
        try:
            case = PrefillCase(pw, device)
            # a batch led by single-token decodes runs as one mixed step: the
            # decodes over their work list beside the chunks on the tensor cores
            mixed = 0 < case.num_decodes < case.B
            split = pw.extra.get("split", 0)
            if mixed:
                case.prepare_mixed()
            if split:
                case.prepare_split(split)
            attend = case.attend_mixed if mixed else case.attend_split if split else case.attend
            status = torch.zeros(1, dtype=torch.int32, device=device)
            pool = []
            for _ in range(4 * (warmup + steps)):  # created and recorded once, before the timed loop
                e = torch.cuda.Event(enable_timing=True)
                e.record(stream)
                pool.append(e)
            step_ev, att_ev = [], []
            torch.cuda.synchronize()
            with ClockSampler(gpu_id()) as clocks:
                for i in range(warmup + steps):
                    flush.fill_(float(i))
                    a0, a1 = pool.pop(), pool.pop()
                    a0.record(stream)
                    case.write(status, stream)  # the chunk's pkv_write, then the attention
                    attend(status, stream)
                    a1.record(stream)
                    flush.fill_(float(i) + 0.5)
                    b0, b1 = pool.pop(), pool.pop()
                    b0.record(stream)
                    attend(status, stream)  # the attention call alone
                    b1.record(stream)
                    if i >= warmup:
                        step_ev.append((a0, a1))
                        att_ev.append((b0, b1))
                torch.cuda.synchronize()
            if status.item() != 0:
                raise RuntimeError(f"device status {status.item()}")
            step_ms = [x.elapsed_time(y) for x, y in step_ev]
            att_ms = [x.elapsed_time(y) for x, y in att_ev]
            sm, am = sum(step_ms) / steps, sum(att_ms) / steps
            fl = case.flops()
            tf = fl / (am * 1e-3) / 1e12
            kv_gbs = case.kv_bytes() / (am * 1e-3) / 1e9
            hbm_peak, hbm_kind = measured_hbm_peak()
            traffic = kernel_traffic("chunk_tc_kernel_traffic.txt", tag)
            if mixed:  # the call's two kernels: the chunks' and the decodes' launches
                tc_part = kernel_traffic("chunk_tc_kernel_traffic.txt", tag + "_chunks")
                dec_part = kernel_traffic("decode_kernel_traffic.txt", tag + "_decodes")
                traffic = tc_part + dec_part if tc_part is not None and dec_part is not None else None
            if case.kv_bytes() / (hbm_peak * 1e9) > fl / (peak * 1e12):
                # more time in moving K/V than in the products at the peaks: bandwidth-bound
                roof = {"bound": "hbm", "achieved": round(kv_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                        "frac": round(kv_gbs / hbm_peak, 4), "peak_kind": f"{hbm_kind} hbm_gbs",
                        "traffic": traffic, "tflops": round(tf, 1)}
            else:
                roof = {"bound": "tensor", "achieved": round(tf, 1), "peak": peak, "unit": "TFLOP/s",
                        "frac": round(tf / peak, 4), "peak_kind": peak_kind, "traffic": traffic}
            res[tag] = {"ms": round(am, 5), "roofline": roof, "kv_gbs": round(kv_gbs, 1),
                        "rows_s": round(case.total_q / (sm * 1e-3), 1), "step_ms": round(sm, 5)}
            if mixed:
                res[tag]["call"] = (f"paged_attention_mixed ({case.mixed_nd} decodes in {case.mixed_part}-token partitions, "
                                    f"chunks on {case.mixed_ctas} CTAs over their list)")
            if split:  # the same call without the split, for comparison
                res[tag]["call"] = f"paged_attention_prefill_ex (keys split into {split}-token partitions)"
                us = []
                for i in range(steps):
                    flush.fill_(float(i) + 0.25)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    case.attend(status, stream)
                    e1.record(stream)
                    torch.cuda.synchronize()
                    us.append(e0.elapsed_time(e1))
                res[tag]["unsplit_ms"] = round(sum(us) / len(us), 5)
            if not compact:
                res[tag].update(
                    workload=f"{pw.name}: {case.B} seqs, (L, chunk) = "
                    + (f"({int(case.lens[0])}, {int(case.chunks[0])})" if "decodes" not in pw.extra else
                       "256 x (U{1..4096}, 1) + (8192, 1024) + (16384, 1024)")
                    + f", block {pw.block_size}, {pw.num_q_heads}q/{pw.num_kv_heads}kv, d {pw.head_dim}, bf16",
                    query_rows=case.total_q, flops_per_call=fl, kv_bytes_per_call=case.kv_bytes(),
                    step_tflops=round(fl / (sm * 1e-3) / 1e12, 1), clocks=clocks.summary())
            if cpu:
                try:
                    cb = prefill_cpu_baseline(case)
                    if compact:
                        res[tag]["cpu_tflops"] = round(cb["value"], 5) if "value" in cb else None
                    else:
                        cb["value"] = round(cb["value"], 6) if "value" in cb else None
                        res[tag]["cpu_baseline"] = cb
                except Exception as e:  # reported, never fatal
                    res[tag]["cpu_baseline"] = {"error": repr(e)}
            del case
            torch.cuda.empty_cache()
        except Exception as e:
            res[tag] = {"error": repr(e)}
            log(f"prefill {tag} failed: {e!r}")
    return res


def run_reference(args, rank, world):
    """The oracle as the reference arm, on this host's cores (rank 0 only): W
    untimed and K timed steps, each a bounded sample of the headline workload's
    step (every sequence, 4 of its 32 layer decodes)."""
    if rank != 0:
        return None
    cb = cpu_oracle_baseline(HEADLINE, reps=args.steps, warmup=args.warmup, layers_per_rep=4)
    ms = cb["seconds"] * 1e3 / cb["reps"]
    return {
        "impl": "reference", "metric": "paged decode attention KV-cache read bandwidth (valid K+V bytes / step time)",
        "value": round(cb["value"], 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": workload_desc(HEADLINE), "parallelism": "host cores (OpenMP)"},
        "query_tok_s": round(cb["query_tok_s"], 3),
        "cpu_baseline": {"kind": "oracle", "cores": cb["cores"], "sample": cb["sample"], "value": round(cb["value"], 4),
                         "unit": "GB/s"},
        "e2e": {"value": round(cb["value"], 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-workloads", action="store_true", help="headline only")
    ap.add_argument("--layers", type=int, default=None,
                    help="decode only this many layers of the multi-layer workload (profiling runs only)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--workload", default=None, choices=[case_tag(*c) for c in WORKLOAD_CASES],
                    help="time only this secondary workload (for profiling runs; no headline line)")
    ap.add_argument("--swap", action="store_true", help="bandwidth of the block swap-out / swap-in copies")
    ap.add_argument("--prefill", nargs="?", const="all", default=None,
                    choices=["all", "prefill_long_context", "prefill_prompts", "prefill_mixed", "prefill_short_chunk"],
                    help="chunked prefill only (all workloads, or the one named)")
    ap.add_argument("--block-sweep", action="store_true",
                    help="block-size trade-off: decode GB/s at block 16..128 and the memory simulation")
    args = ap.parse_args()
    if args.warmup < 3:
        log("warmup raised to 3")
        args.warmup = 3
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        if args.impl == "ours":
            import torch
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
        else:
            dist.init_process_group("gloo")
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    elif args.swap:
        import torch
        from paged_kv_cache_276_gb300 import build
        build.build()
        torch.cuda.set_device(local)
        line = {"swap": swap_bench(torch.device("cuda", local))}
    elif args.prefill:
        import torch
        from paged_kv_cache_276_gb300 import build
        build.build()
        torch.cuda.set_device(local)
        line = {"prefill": prefill_bench(torch.device("cuda", local), steps=args.steps, warmup=args.warmup,
                                         only=None if args.prefill == "all" else args.prefill,
                                         cpu=rank == 0 and world == 1 and not args.no_cpu_baseline)}
    elif args.block_sweep:
        import torch
        from paged_kv_cache_276_gb300 import build
        build.build()
        torch.cuda.set_device(local)
        line = {"block_sweep": block_sweep(torch.device("cuda", local), measured_hbm_peak()[0])}
    elif args.workload:
        import torch
        from paged_kv_cache_276_gb300 import build
        build.build()
        torch.cuda.set_device(local)
        line = {"workloads": other_workloads(args, torch.device("cuda", local), rank, world, measured_hbm_peak()[0],
                                             only=args.workload)}
    else:
        line = run_ours(args, rank, world, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
