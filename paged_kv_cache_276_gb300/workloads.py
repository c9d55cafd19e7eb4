"""Decode workloads driven through the public API, as a serving step would use it.

A ``DecodeSession`` owns the per-layer cache pools on the device, a block
allocator (the native ``BlockAllocator``, or any object with the same methods),
and the sequences.  ``plan_steps`` runs the allocator for a number of decode
steps ahead of time and uploads each step's slot mapping, block tables and
lengths, so timed steps start with every input resident in HBM.  ``run_step``
is one pass of the hot path: for every layer, ``pkv_write`` the new tokens'
K/V, then ``paged_attention_decode`` (plus ``pkv_block_copy`` for any
copy-on-write pairs the step produced).

Random numbers come from ``inputs``; this module does no attention, write or
copy arithmetic itself.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import inputs, native
from .inputs import Workload


def permute_free_blocks(alloc, num_blocks: int, rng: np.random.Generator) -> np.ndarray:
    """Leave the allocator's free stack in a random order using only its public calls.

    Each block is taken by a throw-away one-token sequence, then the sequences
    are freed in a random order; later allocations pop blocks in the reverse of
    that order.  Returns the free order.
    """
    for b in range(num_blocks):
        alloc.seq_add(-(b + 1))
        alloc.seq_append(-(b + 1), 1)
    order = rng.permutation(num_blocks)
    for b in order:
        alloc.seq_free(-(int(b) + 1))
    return order


@dataclass
class StepInputs:
    slots: torch.Tensor         # [B * q_len] int64, device
    tables: torch.Tensor        # [B, max_blocks] int32, device
    lens: torch.Tensor          # [B] int32, device
    max_len: int
    cow_pairs: torch.Tensor | None  # [n, 2] int32, device, or None
    host_tables: np.ndarray
    host_lens: np.ndarray
    items: torch.Tensor | None = None  # single-token steps: the decode's work list [1 + n, 4] int32, device
    partition: int = 0                 # the partition size that list was built for


class DecodeSession:
    def __init__(self, w: Workload, device, allocator_factory=None, block_size: int | None = None,
                 q_len: int | None = None, layers: int | None = None, seq_lens=None,
                 extra_steps: int = 64, prefix_len: int | None = None, seed_salt: int = 0):
        self.w = w
        self.device = torch.device(device)
        self.bs = block_size or w.block_size
        self.q_len = q_len or w.q_len
        self.layers = layers or w.layers
        self.Hq, self.Hkv, self.d = w.num_q_heads, w.num_kv_heads, w.head_dim
        self.scale = w.scale
        self.partition_size = w.partition_size
        self.seed_salt = seed_salt  # offsets every tensor seed (independent replicas)
        factory = allocator_factory or native.BlockAllocator
        rng = inputs.rng_for(w)
        target = np.asarray(inputs.lengths(w, rng) if seq_lens is None else seq_lens, dtype=np.int64)
        self.B = len(target)
        self.extra_steps = extra_steps
        # tokens already cached before the first step; the step adds q_len more.
        # Shared-prefix sampling: prefix + suffix are cached, the step generates
        # the next token of every sample.
        ctx = target.copy() if w.number == 4 else np.maximum(target - self.q_len, 0)
        growth = self.q_len * extra_steps
        if w.number == 4:
            self._init_shared_prefix(factory, ctx, growth, prefix_len or w.extra["prefix"])
        else:
            if w.number == 1:
                self.num_blocks = w.extra["pool"]
            else:
                used = sum(inputs.entries_to_fill(int(n) + growth, self.bs) for n in ctx)
                frac = w.extra.get("pool_extra", 0.10)
                self.num_blocks = int(np.ceil(used * (1 + frac)))
            self.alloc = factory(self.num_blocks, self.bs)
            permute_free_blocks(self.alloc, self.num_blocks, inputs.rng_for(w, salt=1))
            for i, n in enumerate(ctx):
                self.alloc.seq_add(i)
                if n:
                    self.alloc.seq_append(i, int(n))
            self.setup_cow_pairs = np.zeros((0, 2), dtype=np.int32)
        self.max_blocks = max(inputs.entries_to_fill(int(n) + growth, self.bs) for n in ctx) + 1
        self.k_caches, self.v_caches = [], []
        for layer in range(self.layers):
            shape = (self.num_blocks, self.Hkv, self.bs, self.d)
            base = w.seed * 100 + 2 * layer + 7777 * seed_salt
            self.k_caches.append(inputs.randn_bf16(shape, base, self.device))
            self.v_caches.append(inputs.randn_bf16(shape, base + 1, self.device))
        self.step_index = 0

    def _init_shared_prefix(self, factory, ctx, growth, prefix):
        """64 prompts x 8 samples: the prefix blocks are shared by refcount, the
        last prefix block is copied on write for each sample, suffixes follow."""
        w = self.w
        prompts, samples = w.extra["prompts"], w.extra["samples"]
        assert prompts * samples == self.B
        prefix_blocks = inputs.entries_to_fill(prefix, self.bs)
        suffix_blocks = sum(inputs.entries_to_fill(int(n) + growth, self.bs) for n in ctx) \
            - self.B * (prefix // self.bs)
        self.num_blocks = prompts * prefix_blocks + self.B + suffix_blocks + self.B
        self.alloc = factory(self.num_blocks, self.bs)
        pairs = []
        for p in range(prompts):
            parent = 10 ** 9 + p
            self.alloc.seq_add(parent)
            self.alloc.seq_append(parent, prefix)
            for s in range(samples):
                self.alloc.seq_fork(parent, p * samples + s)
            self.alloc.seq_free(parent)
            if prefix % self.bs == 0:
                # The prefix fills its last block, so no write would ever land in
                # it; copy it on each sample's first write anyway, standing in for
                # the partially filled last prefix block of the workload.
                for s in range(samples):
                    pair = self.alloc.seq_cow(p * samples + s, prefix_blocks - 1)
                    if pair is not None:
                        pairs.append(pair)
        for i, n in enumerate(ctx):
            extra = int(n) - prefix
            if extra > 0:
                pair = self.alloc.seq_cow(i)  # no-op unless the next write lands in a shared block
                if pair is not None:
                    pairs.append(pair)
                self.alloc.seq_append(i, extra)
        self.setup_cow_pairs = np.asarray(pairs, dtype=np.int32).reshape(-1, 2)

    # ------------------------------------------------------------ planning
    def plan_step(self) -> StepInputs:
        """Allocator work of one step (host), then upload its inputs."""
        slots = np.empty(self.B * self.q_len, dtype=np.int64)
        pairs = []
        for i in range(self.B):
            pair = self.alloc.seq_cow(i)
            if pair is not None:
                pairs.append(pair)
            slots[i * self.q_len:(i + 1) * self.q_len] = self.alloc.seq_append(i, self.q_len)
        tables, lens = self.alloc.block_table(range(self.B), self.max_blocks)
        tables = np.asarray(tables, dtype=np.int32)
        lens = np.asarray(lens, dtype=np.int32)
        dev = self.device
        cow = torch.as_tensor(np.asarray(pairs, dtype=np.int32).reshape(-1, 2), device=dev) if pairs else None
        items, partition = None, self.partition_size
        if self.q_len == 1:  # the host knows every length: the decode's longest-first work list
            host_items = native.pkv_decode_items(lens, tables, self.Hkv, self.bs, self.partition_size, self.d)
            items, partition = torch.as_tensor(host_items, device=dev), int(host_items[0, 1])
        return StepInputs(torch.as_tensor(slots, device=dev), torch.as_tensor(tables, device=dev),
                          torch.as_tensor(lens, device=dev), int(lens.max()) if len(lens) else 0, cow,
                          tables, lens, items, partition)

    def plan_steps(self, n: int):
        return [self.plan_step() for _ in range(n)]

    def new_token_tensors(self, n_steps: int, seed: int):
        """Per-step q [B, q_len, Hq, d] and new-token k, v [B*q_len, Hkv, d] (per layer)."""
        out = []
        for s in range(n_steps):
            base = seed * 1000 + s * 97 + 7777 * self.seed_salt
            q = inputs.randn_bf16((self.B, self.q_len, self.Hq, self.d), base, self.device)
            ks = [inputs.randn_bf16((self.B * self.q_len, self.Hkv, self.d), base + 1 + 2 * l, self.device)
                  for l in range(self.layers)]
            vs = [inputs.randn_bf16((self.B * self.q_len, self.Hkv, self.d), base + 2 + 2 * l, self.device)
                  for l in range(self.layers)]
            out.append((q, ks, vs))
        return out

    def workspace(self, max_len: int):
        n = native.paged_attention_workspace_size(self.B, self.q_len, self.Hq, self.d, max_len,
                                                  self.partition_size)
        return torch.empty(max(n, 16), dtype=torch.uint8, device=self.device) if n else None

    def apply_setup_copies(self, d_status=None):
        if len(self.setup_cow_pairs):
            pairs = torch.as_tensor(self.setup_cow_pairs, device=self.device)
            for l in range(self.layers):
                native.pkv_block_copy(self.k_caches[l], self.v_caches[l], pairs, d_status=d_status)

    # ------------------------------------------------------------ one step
    def run_step(self, step: StepInputs, q, ks, vs, out, workspace, d_status=None, stream=None,
                 per_layer_out=None, fused=False, planned=False):
        """One pass of the hot path over every layer.  fused (single-token steps):
        the new tokens' store runs inside the decode grid (paged_attention_decode_write);
        planned: that grid runs the host-built work list (paged_attention_decode_items),
        each layer overlapping the one before (PKV_DECODE_OVERLAP; not behind the
        layer's copy-on-write copies, which it reads)."""
        fused = fused and self.q_len == 1
        for l in range(self.layers):
            if step.cow_pairs is not None:
                native.pkv_block_copy(self.k_caches[l], self.v_caches[l], step.cow_pairs, d_status, stream)
            o = out if per_layer_out is None else per_layer_out[l]
            if fused and planned:
                native.paged_attention_decode_items(q, ks[l], vs[l], step.slots, self.k_caches[l], self.v_caches[l],
                                                    step.tables, step.lens, step.max_len, self.scale, o, step.items,
                                                    workspace=workspace, partition_size=step.partition,
                                                    d_status=d_status, stream=stream, overlap=step.cow_pairs is None)
                continue
            if fused:
                native.paged_attention_decode_write(q, ks[l], vs[l], step.slots, self.k_caches[l], self.v_caches[l],
                                                    step.tables, step.lens, step.max_len, self.scale, o, workspace,
                                                    self.partition_size, d_status, stream)
                continue
            native.pkv_write(ks[l], vs[l], step.slots, self.k_caches[l], self.v_caches[l], d_status, stream)
            native.paged_attention_decode(q, self.k_caches[l], self.v_caches[l], step.tables, step.lens,
                                          step.max_len, self.scale, o, workspace, self.partition_size,
                                          d_status, stream)

    def kv_bytes(self, step: StepInputs) -> int:
        """Valid K and V bytes one step's decodes read over all layers."""
        return int(step.host_lens.astype(np.int64).sum()) * 2 * self.Hkv * self.d * 2 * self.layers


# ------------------------------------------------------------ chunked prefill
def causal_visible_keys(lens, chunks) -> int:
    """Sum over every chunk row of the keys it sees: row r of a chunk of c
    tokens in a sequence of L sees max(0, L - c + 1 + r) keys."""
    total = 0
    for L, c in zip(np.asarray(lens, dtype=np.int64), np.asarray(chunks, dtype=np.int64)):
        r0 = max(0, int(c - L))               # rows before r0 see nothing
        n = int(c) - r0
        if n > 0:
            first = int(L - c + 1 + r0)       # keys of row r0; the last row sees L
            total += n * (first + int(L)) // 2
    return total


# Rates of the two halves of a mixed step on one GB300 (measured): chunked
# prefill on the tensor cores (whole GPU, and per prefill-list cost unit on one
# CTA per SM: a pair's 128-key tile, a lone query tile's 0.55, 2 per item), the
# decode kernel over the whole GPU and per SM when only part of the GPU streams
# (the rest busy, HBM not saturated).
PREFILL_FLOPS_PER_S = 1.4e15
CHUNK_UNIT_S = 1.68e-6
DECODE_BYTES_PER_S = 6.3e12
DECODE_SM_BYTES_PER_S = 75e9


def prefill_item_costs(lens, q_start, total_q: int, num_q_heads: int, num_kv_heads: int) -> np.ndarray:
    """Cost of every item of a prefill launch, in the kernel's item order, by
    the model pkv_prefill_items balances: per sequence, per KV head, the pairs
    of query tiles (or lone tiles) from the last one back; an item costs its
    128-key tiles (a lone tile's at 0.55 of a pair's) plus 2."""
    group = num_q_heads // num_kv_heads
    tile_tok = 128 // group
    pairs = total_q >= 2 * tile_tok * len(lens)  # the launch's schedule, as prefill_entry picks it
    span = 2 * tile_tok if pairs else tile_tok
    out = []
    for s in range(len(lens)):
        c, L = int(q_start[s + 1]) - int(q_start[s]), max(0, int(lens[s]))
        nparts = -(-c // span)
        qt = np.arange(nparts - 1, -1, -1)
        k_hi = np.minimum(L, np.maximum(0, L - c + np.minimum(c, span * (qt + 1))))
        pair = pairs & ((2 * qt + 1) * tile_tok < c)
        cost = np.where(pair, 1.0, 0.55) * -(-k_hi // 128) + 2.0
        out.extend([cost] * num_kv_heads)
    return np.concatenate(out) if out else np.zeros(0)


def mixed_step_time(case, prefill_ctas: int, sms: int = 152) -> float:
    """Estimated seconds of a mixed step with the chunks on a grid of
    prefill_ctas CTAs over their host-built list: the chunks end with their
    most loaded CTA; until then the decodes stream on the other SMs, after that
    on the whole GPU."""
    nd = case.num_decodes
    work = native.pkv_prefill_items(case.lens[nd:], case.q_start[nd:], case.total_q, case.Hq, case.Hkv,
                                    prefill_ctas)
    cost = prefill_item_costs(case.lens[nd:], case.q_start[nd:], case.total_q, case.Hq, case.Hkv)
    off = work[2:3 + prefill_ctas]
    items = work[3 + prefill_ctas:]
    t_chunks = max(float(cost[items[off[g]:off[g + 1]]].sum()) for g in range(prefill_ctas)) * CHUNK_UNIT_S
    bytes_dec = float(case.lens[:nd].astype(np.int64).sum()) * 2 * case.Hkv * case.d * 2
    beside = (sms - prefill_ctas) * DECODE_SM_BYTES_PER_S
    if beside > 0 and bytes_dec <= beside * t_chunks:
        return max(t_chunks, bytes_dec / beside)
    return t_chunks + (bytes_dec - max(0, beside) * t_chunks) / DECODE_BYTES_PER_S


def mixed_prefill_ctas(case, sms: int = 152) -> int:
    """Chunk grid of a mixed step: the size from half the SMs up whose
    estimated step (mixed_step_time) is shortest.  The estimate follows the
    host list's packing, which moves in steps (the items are few and large
    against a CTA's share).  Measured on the mixed workload: 0.499 ms at 96
    CTAs, 0.512 at 104, 0.533 at 112, 0.554 at 90, 0.567 at 84."""
    nd = case.num_decodes
    if nd == case.B:
        return 0
    return min(range(sms // 2, sms + 1), key=lambda g: mixed_step_time(case, g, sms))


# One decode CTA streams at most this many bytes per second (its ring's bytes
# in flight over the copy latency; three CTAs share an SM).
DECODE_CTA_BYTES_PER_S = 25e9


def mixed_decode_partition(case, prefill_ctas: int, sms: int = 152) -> int:
    """Partition size of the decodes of a mixed step.  Beside a chunk grid the
    decodes run on the SMs the chunks leave for most of the step, so their
    longest item only has to end before the chunks do: when one whole decode
    (a sequence's KV head, unsplit) streams in under half the chunks' estimated
    time, the decodes run unsplit (no merge kernel, fewer and longer items);
    otherwise the work list picks its partition (0).  Measured on the mixed
    workload (decodes staged one 16-row block per stage): unsplit 0.531-0.539
    ms at 84-89 chunk CTAs, 2048-token partitions 0.551-0.553 ms."""
    nd = case.num_decodes
    if nd == 0 or nd == case.B or prefill_ctas <= 0:
        return 0
    flops_chunks = 4 * case.d * case.Hq * causal_visible_keys(case.lens[nd:], case.chunks[nd:])
    t_chunks = flops_chunks / PREFILL_FLOPS_PER_S * sms / min(sms, prefill_ctas)
    longest = int(case.lens[:nd].max())
    t_item = longest * 2 * case.d * 2 / DECODE_CTA_BYTES_PER_S
    if t_item >= t_chunks / 2:
        return 0
    return -(-longest // case.bs) * case.bs  # whole blocks: one partition per sequence


class PrefillCase:
    """One chunked-prefill batch resident on the device.

    The caches hold every sequence's L tokens, the chunk's own keys and values
    included, as seeded N(0,1) bf16 in a permuted block placement (the state
    after the chunk's ``pkv_write``).  ``step`` is one pass of the hot path: the
    chunk's keys and values written into their slots (``chunk_k``/``chunk_v``,
    fresh seeded values) and ``paged_attention_prefill`` over all sequences.
    """

    def __init__(self, pw: inputs.PrefillWorkload, device, pool_extra: float = 0.05):
        self.pw = pw
        self.device = torch.device(device)
        self.bs, self.Hq, self.Hkv, self.d = pw.block_size, pw.num_q_heads, pw.num_kv_heads, pw.head_dim
        self.scale = pw.scale
        self.lens, self.chunks = inputs.prefill_shape(pw)
        self.B = len(self.lens)
        rng = np.random.default_rng(pw.seed)
        NB = inputs.pool_size(self.lens, self.bs, pool_extra)
        self.num_blocks = NB
        self.tables, _ = inputs.permuted_tables(self.lens, self.bs, NB, rng)
        self.k_cache = inputs.randn_bf16((NB, self.Hkv, self.bs, self.d), pw.seed * 10 + 1, self.device)
        self.v_cache = inputs.randn_bf16((NB, self.Hkv, self.bs, self.d), pw.seed * 10 + 2, self.device)
        self.q_start = np.concatenate([[0], np.cumsum(self.chunks)]).astype(np.int32)
        self.total_q = int(self.q_start[-1])
        self.q = inputs.randn_bf16((self.total_q, self.Hq, self.d), pw.seed * 10 + 3, self.device)
        # slot of every chunk token: positions L - c .. L - 1 of its sequence
        slots = np.empty(self.total_q, dtype=np.int64)
        for i, (L, c) in enumerate(zip(self.lens, self.chunks)):
            t = np.arange(L - c, L)
            slots[self.q_start[i]:self.q_start[i + 1]] = self.tables[i, t // self.bs].astype(np.int64) * self.bs \
                + t % self.bs
        self.slots = torch.as_tensor(slots, device=self.device)
        self.chunk_k = inputs.randn_bf16((self.total_q, self.Hkv, self.d), pw.seed * 10 + 4, self.device)
        self.chunk_v = inputs.randn_bf16((self.total_q, self.Hkv, self.d), pw.seed * 10 + 5, self.device)
        self.d_tables = torch.as_tensor(self.tables, device=self.device)
        self.d_lens = torch.as_tensor(self.lens, device=self.device)
        self.d_q_start = torch.as_tensor(self.q_start, device=self.device)
        self.out = torch.empty_like(self.q)

    def attend(self, d_status=None, stream=None):
        native.paged_attention_prefill(self.q, self.k_cache, self.v_cache, self.d_tables, self.d_lens,
                                       self.d_q_start, self.scale, self.out, d_status, stream)

    # A batch whose leading sequences are single-token decodes (rows 0..nd-1)
    # can run as one mixed step: the decodes over their work list beside the chunks.
    @property
    def num_decodes(self) -> int:
        nd = 0
        while nd < self.B and int(self.chunks[nd]) == 1 and int(self.q_start[nd]) == nd:
            nd += 1
        return nd

    def prepare_mixed(self, prefill_ctas=None, partition_size=0, chunk_list=True):
        """Work list and workspace of the leading decodes (partition_size 0:
        mixed_decode_partition's choice); the chunks' grid cap (default:
        mixed_prefill_ctas) and, with chunk_list, their host-built work list
        for that grid."""
        nd = self.num_decodes
        self.mixed_nd = nd
        self.mixed_max_len = int(self.lens[:nd].max()) if nd else 0
        self.mixed_ctas = mixed_prefill_ctas(self) if prefill_ctas is None else prefill_ctas
        if partition_size == 0:
            partition_size = mixed_decode_partition(self, self.mixed_ctas)
        host_items = native.pkv_decode_items(self.lens[:nd], self.tables[:nd], self.Hkv, self.bs, partition_size,
                                             self.d)
        self.mixed_part = int(host_items[0, 1])
        self.mixed_items = torch.as_tensor(host_items, device=self.device)
        n = native.paged_attention_workspace_size(nd, 1, self.Hq, self.d, self.mixed_max_len, self.mixed_part)
        self.mixed_ws = torch.empty(max(n, 16), dtype=torch.uint8, device=self.device)
        self.mixed_chunk_items = None
        if chunk_list and nd < self.B and self.mixed_ctas > 0:
            w = native.pkv_prefill_items(self.lens[nd:], self.q_start[nd:], self.total_q, self.Hq, self.Hkv,
                                         self.mixed_ctas)
            self.mixed_chunk_items = torch.as_tensor(w, device=self.device)

    def prepare_split(self, partition_size: int):
        """Workspace of the prefill split over keys into partition_size-token partitions."""
        self.split_part = partition_size
        self.split_max_len = int(self.lens.max())
        n = native.paged_attention_prefill_workspace_size(self.total_q, self.Hq, self.d, self.split_max_len,
                                                          partition_size)
        self.split_ws = torch.empty(max(n, 16), dtype=torch.uint8, device=self.device)

    def attend_split(self, d_status=None, stream=None):
        native.paged_attention_prefill_ex(self.q, self.k_cache, self.v_cache, self.d_tables, self.d_lens,
                                          self.d_q_start, self.scale, self.out, self.split_max_len, self.split_part,
                                          self.split_ws, d_status, stream)

    def attend_mixed(self, d_status=None, stream=None):
        native.paged_attention_mixed(self.q, self.k_cache, self.v_cache, self.d_tables, self.d_lens, self.d_q_start,
                                     self.scale, self.out, self.mixed_nd, self.mixed_items, self.mixed_max_len,
                                     self.mixed_part, self.mixed_ws, self.mixed_ctas, d_status=d_status,
                                     stream=stream, prefill_items=self.mixed_chunk_items)

    def write(self, d_status=None, stream=None):
        """The chunk tokens' keys and values into their slots."""
        native.pkv_write(self.chunk_k, self.chunk_v, self.slots, self.k_cache, self.v_cache, d_status, stream)

    def step(self, d_status=None, stream=None):
        self.write(d_status, stream)
        self.attend(d_status, stream)

    def flops(self) -> int:
        """Algorithmic FLOPs of the attention: per query head and visible key,
        d multiply-adds for q.k and d for p.v."""
        return 4 * self.d * self.Hq * causal_visible_keys(self.lens, self.chunks)

    def kv_bytes(self) -> int:
        """Distinct K and V bytes the call needs (every cached token once)."""
        return int(self.lens.astype(np.int64).sum()) * 2 * self.Hkv * self.d * 2
