"""KV-cache memory accounting: paged blocks versus one contiguous reservation per request.

The pages weigh the two layouts.  A contiguous region reserved for the most a
request might generate wastes what it never generates (4,096 tokens reserved
for a request that stops after 287; 2,048 for one that stops after 200), and
regions with different lifetimes leave holes that later requests do not fit
(x321.org "The serving bottleneck is not just FLOPs", section "Why naive
allocation wastes so much memory"; praveentn.live "PagedAttention KV-cache
constraint", section "The situation").  Fixed-size blocks waste at most one
partial block per request and every free block fits every request (same
page, "What the change bought"); smaller blocks waste less but cost more
addressing and bookkeeping, which slot arithmetic alone cannot price
(chenhuiyu.github.io "A complete explanation from first principles", section
"Calculate a block-allocation example").

``simulate`` runs both layouts on the same stream of requests through the same
memory: every request has a prompt and a final length; each step every
running request that has room appends one token; finished requests free their
memory; waiting requests are admitted first come first served while they fit.
The paged side runs on the library's own block allocator (``BlockAllocator``,
through the C ABI); the contiguous side on a first-fit allocator of intervals
kept here.  Both report, per step, the tokens of KV state held, the memory they
pin, the requests running, and the tokens generated.
"""
from __future__ import annotations

import bisect
import math
from dataclasses import dataclass

import numpy as np


@dataclass
class SimResult:
    layout: str               # "paged" or "contiguous"
    block_size: int           # paged block size (contiguous: 1)
    capacity_tokens: int
    steps: int
    generated: int            # tokens appended over the run
    token_state_fraction: float  # mean over steps of (tokens held) / capacity
    pinned_fraction: float       # mean over steps of (memory pinned) / capacity
    utilisation: float           # sum of tokens held / sum of memory pinned
    mean_running: float
    peak_running: int
    preemptions: int

    @property
    def tokens_per_step(self) -> float:
        return self.generated / max(1, self.steps)


class FirstFit:
    """Contiguous allocator over [0, capacity): sorted free intervals, first fit."""

    def __init__(self, capacity: int):
        self.free = [(0, capacity)]  # (start, length), sorted by start, coalesced

    def alloc(self, n: int):
        for i, (s, ln) in enumerate(self.free):
            if ln >= n:
                if ln == n:
                    del self.free[i]
                else:
                    self.free[i] = (s + n, ln - n)
                return s
        return None

    def release(self, start: int, n: int):
        i = bisect.bisect_left(self.free, (start, 0))
        self.free.insert(i, (start, n))
        # coalesce with the neighbours
        if i + 1 < len(self.free) and self.free[i][0] + self.free[i][1] == self.free[i + 1][0]:
            self.free[i] = (self.free[i][0], self.free[i][1] + self.free[i + 1][1])
            del self.free[i + 1]
        if i > 0 and self.free[i - 1][0] + self.free[i - 1][1] == self.free[i][0]:
            self.free[i - 1] = (self.free[i - 1][0], self.free[i - 1][1] + self.free[i][1])
            del self.free[i]

    def largest_hole(self) -> int:
        return max((ln for _, ln in self.free), default=0)

    def total_free(self) -> int:
        return sum(ln for _, ln in self.free)


def contiguous_used_fraction(final_tokens: int, reserved_tokens: int) -> float:
    """Share of a contiguous reservation that ends up holding tokens."""
    if not 0 < final_tokens <= reserved_tokens:
        raise ValueError("need 0 < final <= reserved")
    return final_tokens / reserved_tokens


def paged_slots(tokens: int, block_size: int) -> int:
    """Slots of the blocks a request of `tokens` tokens holds (the unused ones are
    the tail of its last block)."""
    return -(-int(tokens) // int(block_size)) * int(block_size)


def simulate(prompts, finals, capacity_tokens: int, layout: str, block_size: int = 16, reserve=None,
             max_steps: int = 10 ** 7, trace: list | None = None) -> SimResult:
    """Run the request stream to completion.

    prompts, finals: per request, tokens at admission and at completion
    (1 <= prompt <= final).  capacity_tokens: the KV memory, in token slots.
    layout "contiguous" reserves ``reserve`` slots at admission (one size for
    all, a size per request, or by default the largest final length); "paged" takes ceil(prompt / block_size) blocks at
    admission and one block whenever a token starts a new block.  A paged
    request is admitted only while one free block per running request stays
    in reserve, so running requests can grow; one that still cannot get its
    next block waits, and when no running request can make progress the most
    recently admitted one is preempted (its blocks freed, the request sent
    back to the head of the queue to start over).  ``trace``, when given,
    receives (tokens held, memory pinned, requests running) after every step.
    """
    prompts = [int(x) for x in prompts]
    finals = [int(x) for x in finals]
    if any(p < 1 or p > f for p, f in zip(prompts, finals)):
        raise ValueError("need 1 <= prompt <= final for every request")
    n = len(prompts)
    queue = list(range(n))
    running = {}  # request -> current length
    order = []    # admission order of running requests
    held_sum = pinned_sum = 0.0
    steps = generated = preemptions = peak = 0
    run_sum = 0

    if layout == "contiguous":
        if reserve is None:
            sizes = [max(finals)] * n
        elif np.ndim(reserve) == 0:
            sizes = [int(reserve)] * n
        else:
            sizes = [int(x) for x in reserve]
        if len(sizes) != n or any(sz < f for sz, f in zip(sizes, finals)):
            raise ValueError("every contiguous reservation must hold its request's final length")
        ff = FirstFit(capacity_tokens)
        where = {}

        def admit(r):
            s = ff.alloc(sizes[r])
            if s is None:
                return False
            where[r] = s
            return True

        def grow(r):
            return True

        def release(r):
            ff.release(where.pop(r), sizes[r])

        def pinned():
            return sum(sizes[r] for r in running)

        def admit_possible(r):
            return sizes[r] <= capacity_tokens
    elif layout == "paged":
        from .native import BlockAllocator, PkvError
        nblocks = capacity_tokens // block_size
        alloc = BlockAllocator(nblocks, block_size)

        def admit(r):
            need = math.ceil(prompts[r] / block_size)
            if alloc.num_free() < need + len(running):
                return False
            alloc.seq_add(r)
            alloc.seq_append(r, prompts[r])
            return True

        def grow(r):
            try:
                alloc.seq_append(r, 1)
                return True
            except PkvError:
                return False

        def release(r):
            alloc.seq_free(r)

        def pinned():
            return (nblocks - alloc.num_free()) * block_size

        def admit_possible(r):
            return math.ceil(finals[r] / block_size) <= nblocks
    else:
        raise ValueError(layout)

    try:
        while (queue or running) and steps < max_steps:
            if not running and queue and not admit_possible(queue[0]):
                raise ValueError("a request does not fit in the memory at all")
            while queue and admit(queue[0]):
                r = queue.pop(0)
                running[r] = prompts[r]
                order.append(r)
            progressed = False
            for r in list(order):
                if running[r] >= finals[r]:
                    continue
                if grow(r):
                    running[r] += 1
                    generated += 1
                    progressed = True
            peak = max(peak, len(running))  # requests that ran this step
            done = [r for r in order if running[r] >= finals[r]]
            for r in done:
                release(r)
                del running[r]
                order.remove(r)
                progressed = True
            if not progressed and order:  # out of blocks: send the youngest request back
                r = order.pop()
                release(r)
                del running[r]
                queue.insert(0, r)
                preemptions += 1
            steps += 1
            held = sum(running.values())
            pin = pinned()
            if trace is not None:
                trace.append((held, pin, len(running)))
            held_sum += held
            pinned_sum += pin
            run_sum += len(running)
    finally:
        if layout == "paged":
            alloc.close()
    return SimResult(layout=layout, block_size=block_size if layout == "paged" else 1,
                     capacity_tokens=capacity_tokens, steps=steps, generated=generated,
                     token_state_fraction=held_sum / max(1, steps) / capacity_tokens,
                     pinned_fraction=pinned_sum / max(1, steps) / capacity_tokens,
                     utilisation=held_sum / pinned_sum if pinned_sum else 1.0,
                     mean_running=run_sum / max(1, steps), peak_running=peak, preemptions=preemptions)


def request_stream(final_lengths, rng: np.random.Generator, prompt_fraction: float = 0.5):
    """Prompts for a list of final lengths: each request's prompt is a fraction
    of its final length (at least one token), the rest is generated."""
    finals = np.asarray(final_lengths, dtype=np.int64)
    prompts = np.maximum(1, np.floor(finals * prompt_fraction)).astype(np.int64)
    return prompts.tolist(), finals.tolist()
