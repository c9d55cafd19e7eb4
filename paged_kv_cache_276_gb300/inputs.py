"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle side.

This module only draws random numbers and lays them out: sequence lengths,
physical block placements, bf16 N(0,1) tensors.  It holds none of the
attention, write or copy arithmetic and imports neither the oracle nor the
CUDA binding, so both sides can be fed from it.

The one count it takes is how many block-table entries to fill for a sequence
of L tokens (enough entries to cover L); each side decides on its own how many
entries it reads.

Workloads (seed = 1000 + workload number):
  1 tiny            lengths [17, 33, 64], block 16, 4 q / 2 KV heads, d 64,
                    blocks drawn from a 32-block pool in permuted order
  2 batched GQA     32 sequences, L ~ U{1..4096}, block 16, 32 q / 8 KV heads,
                    d 128, pool = used blocks + 10 %, permuted placement
  3 batching mix    256 sequences, L = clip(round(exp(ln 512 + N(0,1))), 1, 8192),
                    block 16, 32 q / 8 KV heads, d 128, 32 layers with a pool each
  4 shared prefix   64 prompts x 8 samples, 2048-token shared prefix,
                    suffix ~ U{0..512}, block 16, 32 q / 8 KV heads, d 128
  5 long context    16 x 32768 tokens, block 16 and 32, 64 q / 8 KV heads,
                    d 128, 512-token partitions, plus a 16-token causal chunk

Chunked-prefill workloads (``PREFILL_WORKLOADS``; each sequence is (context
length L including its chunk, chunk length c)):
  prefill_long_context  16 sequences, the last 1,024 tokens of a 32,768-token
                        prompt (L 32768, c 1024), block 16, 64 q / 8 KV heads, d 128
  prefill_prompts       8 prompts of 4,096 tokens prefilled whole from an empty
                        cache (L = c = 4096), block 16, 64 q / 8 KV heads, d 128
  prefill_mixed         one scheduler step: 256 single-token decodes with
                        L ~ U{1..4096} and two 1,024-token prompt chunks at
                        L 8192 and 16384, block 16, 32 q / 8 KV heads, d 128
  prefill_short_chunk   one 128-token chunk behind 32,640 cached tokens
                        (L 32768, c 128), block 16, 64 q / 8 KV heads, d 128,
                        its keys split into 8192-token partitions
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    number: int
    name: str
    num_seqs: int
    block_size: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    q_len: int = 1
    layers: int = 1
    partition_size: int = 0  # 0: the library's default; the long-context workload names 512
    extra: dict = field(default_factory=dict)

    @property
    def seed(self) -> int:
        return 1000 + self.number

    @property
    def scale(self) -> float:
        return float(np.float32(1.0 / math.sqrt(self.head_dim)))


WORKLOADS = {
    1: Workload(1, "tiny paged decode", 3, 16, 4, 2, 64, extra={"pool": 32}),
    2: Workload(2, "batched decode, GQA 32q/8kv", 32, 16, 32, 8, 128,
                extra={"len_max": 4096, "pool_extra": 0.10}),
    3: Workload(3, "continuous-batching mix, 32 layers", 256, 16, 32, 8, 128, layers=32,
                extra={"median": 512, "sigma": 1.0, "clip": (1, 8192), "pool_extra": 0.10}),
    4: Workload(4, "shared-prefix parallel sampling", 512, 16, 32, 8, 128,
                extra={"prompts": 64, "samples": 8, "prefix": 2048, "suffix_max": 512}),
    5: Workload(5, "long-context decode", 16, 16, 64, 8, 128, partition_size=512,
                extra={"len": 32768, "chunk": 16}),
}


@dataclass(frozen=True)
class PrefillWorkload:
    tag: str
    name: str
    block_size: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    seed: int
    extra: dict = field(default_factory=dict)

    @property
    def scale(self) -> float:
        return float(np.float32(1.0 / math.sqrt(self.head_dim)))


PREFILL_WORKLOADS = {
    "prefill_long_context": PrefillWorkload("prefill_long_context", "chunked prefill behind a 31,744-token context",
                                            16, 64, 8, 128, 2001, extra={"seqs": 16, "len": 32768, "chunk": 1024}),
    "prefill_prompts": PrefillWorkload("prefill_prompts", "whole 4,096-token prompts from an empty cache",
                                       16, 64, 8, 128, 2002, extra={"seqs": 8, "len": 4096, "chunk": 4096}),
    "prefill_mixed": PrefillWorkload("prefill_mixed", "256 decodes + two 1,024-token prompt chunks in one call",
                                     16, 32, 8, 128, 2003,
                                     extra={"decodes": 256, "len_max": 4096, "chunks": ((8192, 1024), (16384, 1024))}),
    # one short chunk behind a long context: 8 query tiles x 8 KV heads, fewer units
    # of work than SMs unless the keys are split (partitions of 8192 keys: 4 pairs
    # of query tiles x 8 KV heads x 4 partitions = 128 items, one per CTA)
    "prefill_short_chunk": PrefillWorkload("prefill_short_chunk", "one 128-token chunk behind a 32,640-token context",
                                           16, 64, 8, 128, 2004,
                                           extra={"seqs": 1, "len": 32768, "chunk": 128, "split": 8192}),
}


def prefill_shape(pw: PrefillWorkload):
    """(lengths L, chunk lengths c) of a prefill workload's sequences, int32."""
    e = pw.extra
    if "decodes" in e:
        rng = np.random.default_rng(pw.seed)
        lens = list(rng.integers(1, e["len_max"] + 1, size=e["decodes"]))
        chunks = [1] * e["decodes"]
        for L, c in e["chunks"]:
            lens.append(L)
            chunks.append(c)
        return np.asarray(lens, dtype=np.int32), np.asarray(chunks, dtype=np.int32)
    return (np.full(e["seqs"], e["len"], dtype=np.int32), np.full(e["seqs"], e["chunk"], dtype=np.int32))


def rng_for(w: Workload, salt: int = 0) -> np.random.Generator:
    return np.random.default_rng(w.seed + 7919 * salt)


def lengths(w: Workload, rng: np.random.Generator | None = None) -> np.ndarray:
    """Context lengths (tokens, including the newest) of the workload's sequences."""
    rng = rng_for(w) if rng is None else rng
    if w.number == 1:
        return np.array([17, 33, 64], dtype=np.int32)
    if w.number == 2:
        return rng.integers(1, w.extra["len_max"] + 1, size=w.num_seqs).astype(np.int32)
    if w.number == 3:
        lo, hi = w.extra["clip"]
        x = np.exp(np.log(w.extra["median"]) + w.extra["sigma"] * rng.standard_normal(w.num_seqs))
        return np.clip(np.rint(x), lo, hi).astype(np.int32)
    if w.number == 4:
        suffix = rng.integers(0, w.extra["suffix_max"] + 1, size=w.num_seqs)
        return (w.extra["prefix"] + suffix).astype(np.int32)
    if w.number == 5:
        return np.full(w.num_seqs, w.extra["len"], dtype=np.int32)
    raise KeyError(w.number)


def entries_to_fill(length: int, block_size: int) -> int:
    """Table entries that cover ``length`` tokens."""
    return -(-int(length) // block_size)


def permuted_tables(seq_lens, block_size: int, num_blocks: int, rng: np.random.Generator,
                    max_blocks: int | None = None):
    """Block tables whose entries come from a random permutation of the pool, in order.

    Returns (tables int32 [B, max_blocks] padded with -1, permutation).
    """
    counts = [entries_to_fill(n, block_size) for n in seq_lens]
    if sum(counts) > num_blocks:
        raise ValueError("pool too small")
    if max_blocks is None:
        max_blocks = max(counts) if counts else 1
    perm = rng.permutation(num_blocks).astype(np.int32)
    tables = np.full((len(counts), max(1, max_blocks)), -1, dtype=np.int32)
    pos = 0
    for i, c in enumerate(counts):
        tables[i, :c] = perm[pos:pos + c]
        pos += c
    return tables, perm


def pool_size(seq_lens, block_size: int, extra_fraction: float) -> int:
    used = sum(entries_to_fill(n, block_size) for n in seq_lens)
    return int(math.ceil(used * (1.0 + extra_fraction)))


def randn_bf16(shape, seed: int, device="cpu", chunk_rows: int = 1 << 14) -> torch.Tensor:
    """bf16 N(0,1) tensor drawn from torch's generator on ``device`` (chunked along dim 0)."""
    shape = tuple(int(s) for s in shape)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    rows = shape[0] if shape else 1
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        out[r0:r1] = torch.randn((r1 - r0,) + shape[1:], generator=g, device=device,
                                 dtype=torch.float32).to(torch.bfloat16)
    return out


def distinct_slots(num_tokens: int, num_slots: int, rng: np.random.Generator,
                   skip_fraction: float = 0.0) -> np.ndarray:
    """``num_tokens`` distinct slots in [0, num_slots); a fraction replaced by -1 (skip)."""
    slots = rng.choice(num_slots, size=num_tokens, replace=False).astype(np.int64)
    if skip_fraction > 0:
        mask = rng.random(num_tokens) < skip_fraction
        slots[mask] = -1
    return slots
