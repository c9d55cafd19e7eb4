"""Dictionary restatement of the block manager: pool, block tables, refcounts, copy-on-write.

TEST INFRASTRUCTURE ONLY.  It shares no code with the native allocator; the
tests drive both with the same call sequence and compare every table, length,
refcount and free count bit for bit.

What the pages fix:
* a sequence's cache is split into fixed-size blocks anywhere in a pool, a
  per-sequence block table keeps the logical order, a request grows by taking
  more free blocks, and a finished request returns its blocks to the pool
  (x321.org "The serving bottleneck is not just FLOPs", section
  "PagedAttention borrows an operating-system trick");
* blocks holding an identical prefix may be referenced by several sequences
  and are copied on write (praveentn.live "PagedAttention KV-cache
  constraint", section "What the change bought");
* under memory pressure a sequence's blocks are swapped out to host memory
  and back (same page, "What it cost").

Readings of ours where the pages leave the policy open:
* free blocks form a LIFO stack that starts as [NB-1, ..., 1, 0] (top last),
  so the first block handed out is 0; blocks whose refcount falls to zero are
  pushed back in logical order;
* an append that would write into a partially filled block with refcount > 1
  is refused ("shared"); the caller first asks for the copy-on-write;
* a failed call (out of blocks, bad id) leaves the state unchanged;
* a swapped-out sequence keeps its id and length, releases its blocks like a
  free does, refuses append / fork / cow / table until it is swapped back in,
  and comes back with fresh private blocks in logical order;
* prefix caching (tokens appended with their ids): a full block is known by
  its whole token prefix; a block about to be stored whose prefix is already
  known is shared instead (slot -1, nothing to store); a known block nobody
  holds stays known and counts as free, and when the free stack is empty the
  one released longest ago is reused (forgotten).  Lookups of a call are made
  before any block is taken.  A plain append or a swap-in ends prefix
  tracking for that sequence.
"""
from __future__ import annotations


class AllocError(Exception):
    """Raised with ``kind`` in {"arg", "oom", "range", "shared"}."""

    def __init__(self, kind: str, msg: str = ""):
        super().__init__(f"{kind}: {msg}")
        self.kind = kind


class OracleAllocator:
    def __init__(self, num_blocks: int, block_size: int):
        if num_blocks < 0 or block_size < 1:
            raise AllocError("arg", "bad pool shape")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free = list(range(num_blocks - 1, -1, -1))  # top of stack = end of list
        self.refcount = [0] * num_blocks
        self.seqs: dict[int, dict] = {}
        self.known: dict[tuple, int] = {}        # whole token prefix of a full block -> block
        self.prefix_of: dict[int, tuple] = {}    # known block -> its prefix
        self.unheld: list[int] = []              # known blocks nobody holds, released longest ago first

    # -- helpers -----------------------------------------------------------
    def _blocks_for(self, length: int) -> int:
        n = 0
        while n * self.block_size < length:
            n += 1
        return n

    def _get(self, seq_id: int, resident: bool = True) -> dict:
        if seq_id not in self.seqs:
            raise AllocError("arg", f"unknown sequence {seq_id}")
        s = self.seqs[seq_id]
        if resident and s["swapped"]:
            raise AllocError("arg", f"sequence {seq_id} is swapped out")
        return s

    def _take(self) -> int:
        if self.free:
            b = self.free.pop()
        else:
            b = self.unheld.pop(0)
            del self.known[self.prefix_of.pop(b)]
        self.refcount[b] = 1
        return b

    def _release(self, b: int) -> None:
        self.refcount[b] -= 1
        if self.refcount[b] == 0:
            if b in self.prefix_of:
                self.unheld.append(b)
            else:
                self.free.append(b)

    def _remember(self, b: int, prefix: tuple) -> None:
        if b in self.prefix_of or prefix in self.known:
            return
        self.known[prefix] = b
        self.prefix_of[b] = prefix

    # -- operations --------------------------------------------------------
    def seq_add(self, seq_id: int) -> None:
        if seq_id in self.seqs:
            raise AllocError("arg", f"sequence {seq_id} exists")
        self.seqs[seq_id] = {"blocks": [], "len": 0, "swapped": False, "tokens": []}

    def seq_append(self, seq_id: int, n_tokens: int) -> list[int]:
        s = self._get(seq_id)
        if n_tokens < 0:
            raise AllocError("arg", "negative token count")
        if n_tokens == 0:
            return []
        old_len = s["len"]
        if old_len % self.block_size != 0:
            last = s["blocks"][-1]
            if self.refcount[last] > 1:
                raise AllocError("shared", f"block {last} is shared; copy it first")
        new_len = old_len + n_tokens
        need = self._blocks_for(new_len) - len(s["blocks"])
        if need > self.num_free():
            raise AllocError("oom", f"need {need} blocks, {self.num_free()} free")
        for _ in range(need):
            s["blocks"].append(self._take())
        slots = []
        for pos in range(old_len, new_len):
            logical, offset = divmod(pos, self.block_size)
            slots.append(s["blocks"][logical] * self.block_size + offset)
        s["len"] = new_len
        s["tokens"] = None  # token ids unknown from here on
        return slots

    def seq_append_tokens(self, seq_id: int, token_ids) -> tuple[list[int], int]:
        """Append tokens with their ids; returns (slots, tokens found already stored)."""
        s = self._get(seq_id)
        toks = [int(t) for t in token_ids]
        if not toks:
            return [], 0
        bs = self.block_size
        old_len = s["len"]
        if old_len % bs != 0 and self.refcount[s["blocks"][-1]] > 1:
            raise AllocError("shared", "the open block is shared; copy it first")
        new_len = old_len + len(toks)
        tracked = s["tokens"] is not None
        prefix = (s["tokens"] + toks) if tracked else None
        first_new = self._blocks_for(old_len)          # index of the first block this call adds
        last_full = new_len // bs                      # blocks complete after the call
        plan = []                                      # (block index, known block or None)
        for j in range(first_new, last_full):
            plan.append((j, self.known.get(tuple(prefix[:(j + 1) * bs])) if tracked else None))
        tail_new = 1 if new_len % bs and new_len // bs >= first_new else 0  # a new, partial last block
        fresh = sum(1 for _, b in plan if b is None) + tail_new
        revive = sum(1 for _, b in plan if b is not None and self.refcount[b] == 0)
        if fresh > self.num_free() - revive:
            raise AllocError("oom", "not enough free blocks")
        for _, b in plan:  # hold the known blocks first
            if b is not None:
                if self.refcount[b] == 0:
                    self.unheld.remove(b)
                self.refcount[b] += 1
        slots, cached = [], 0
        pos = old_len
        if old_len % bs:
            while pos < new_len and pos % bs:
                slots.append(s["blocks"][-1] * bs + pos % bs)
                pos += 1
            if tracked and pos % bs == 0:
                self._remember(s["blocks"][-1], tuple(prefix[:pos]))
        for j, b in plan:
            if b is not None:
                s["blocks"].append(b)
                slots.extend([-1] * bs)
                cached += bs
            else:
                b = self._take()
                s["blocks"].append(b)
                slots.extend(b * bs + i for i in range(bs))
                if tracked:
                    self._remember(b, tuple(prefix[:(j + 1) * bs]))
            pos += bs
        if pos < new_len:
            b = self._take()
            s["blocks"].append(b)
            while pos < new_len:
                slots.append(b * bs + pos % bs)
                pos += 1
        s["len"] = new_len
        if tracked:
            s["tokens"] = prefix
        return slots, cached

    def seq_fork(self, parent: int, child: int) -> None:
        p = self._get(parent)
        if child in self.seqs:
            raise AllocError("arg", f"sequence {child} exists")
        for b in p["blocks"]:
            self.refcount[b] += 1
        self.seqs[child] = {"blocks": list(p["blocks"]), "len": p["len"], "swapped": False,
                            "tokens": None if p["tokens"] is None else list(p["tokens"])}

    def seq_cow(self, seq_id: int, logical: int = -1):
        """Give ``seq_id`` a private copy of one shared block.

        ``logical = -1`` picks the block the next append would write into (none
        when the last block is full).  Returns ``(src, dst)`` when a copy is
        needed, else ``None``.
        """
        s = self._get(seq_id)
        if logical == -1:
            if s["len"] % self.block_size == 0:
                return None
            logical = s["len"] // self.block_size
        if not (0 <= logical < len(s["blocks"])):
            raise AllocError("range", f"logical block {logical} out of range")
        old = s["blocks"][logical]
        if self.refcount[old] <= 1:
            return None
        if self.num_free() == 0:
            raise AllocError("oom", "no free block for the copy")
        new = self._take()
        self.refcount[old] -= 1
        s["blocks"][logical] = new
        return (old, new)

    def seq_free(self, seq_id: int) -> None:
        s = self._get(seq_id, resident=False)
        for b in s["blocks"]:
            self._release(b)
        del self.seqs[seq_id]

    def seq_swap_out(self, seq_id: int, max_blocks: int) -> list[int]:
        """Release the sequence's blocks (returned in logical order for the copy out)."""
        s = self._get(seq_id)
        if len(s["blocks"]) > max_blocks:
            raise AllocError("range", f"sequence {seq_id} has more than {max_blocks} blocks")
        out = list(s["blocks"])
        for b in out:
            self._release(b)
        s["blocks"] = []
        s["swapped"] = True
        return out

    def seq_swap_in(self, seq_id: int, max_blocks: int) -> list[int]:
        """Fresh blocks for a swapped-out sequence (logical order), for the copy in."""
        s = self._get(seq_id, resident=False)
        if not s["swapped"]:
            raise AllocError("arg", f"sequence {seq_id} is resident")
        need = self._blocks_for(s["len"])
        if need > max_blocks:
            raise AllocError("range", f"sequence {seq_id} needs more than {max_blocks} blocks")
        if need > self.num_free():
            raise AllocError("oom", f"need {need} blocks, {self.num_free()} free")
        for _ in range(need):
            s["blocks"].append(self._take())
        s["swapped"] = False
        s["tokens"] = None
        return list(s["blocks"])

    def block_table(self, seq_ids, max_blocks: int):
        """Rows of physical ids (-1 past each sequence's blocks) and lengths."""
        table, lens = [], []
        for sid in seq_ids:
            s = self._get(sid)
            if len(s["blocks"]) > max_blocks:
                raise AllocError("range", f"sequence {sid} has more than {max_blocks} blocks")
            table.append(list(s["blocks"]) + [-1] * (max_blocks - len(s["blocks"])))
            lens.append(s["len"])
        return table, lens

    def num_free(self) -> int:
        return len(self.free) + len(self.unheld)
