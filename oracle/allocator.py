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
  and comes back with fresh private blocks in logical order.
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

    # -- operations --------------------------------------------------------
    def seq_add(self, seq_id: int) -> None:
        if seq_id in self.seqs:
            raise AllocError("arg", f"sequence {seq_id} exists")
        self.seqs[seq_id] = {"blocks": [], "len": 0, "swapped": False}

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
        if need > len(self.free):
            raise AllocError("oom", f"need {need} blocks, {len(self.free)} free")
        for _ in range(need):
            b = self.free.pop()
            self.refcount[b] = 1
            s["blocks"].append(b)
        slots = []
        for pos in range(old_len, new_len):
            logical, offset = divmod(pos, self.block_size)
            slots.append(s["blocks"][logical] * self.block_size + offset)
        s["len"] = new_len
        return slots

    def seq_fork(self, parent: int, child: int) -> None:
        p = self._get(parent)
        if child in self.seqs:
            raise AllocError("arg", f"sequence {child} exists")
        for b in p["blocks"]:
            self.refcount[b] += 1
        self.seqs[child] = {"blocks": list(p["blocks"]), "len": p["len"], "swapped": False}

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
        if not self.free:
            raise AllocError("oom", "no free block for the copy")
        new = self.free.pop()
        self.refcount[new] = 1
        self.refcount[old] -= 1
        s["blocks"][logical] = new
        return (old, new)

    def seq_free(self, seq_id: int) -> None:
        s = self._get(seq_id, resident=False)
        for b in s["blocks"]:
            self.refcount[b] -= 1
            if self.refcount[b] == 0:
                self.free.append(b)
        del self.seqs[seq_id]

    def seq_swap_out(self, seq_id: int, max_blocks: int) -> list[int]:
        """Release the sequence's blocks (returned in logical order for the copy out)."""
        s = self._get(seq_id)
        if len(s["blocks"]) > max_blocks:
            raise AllocError("range", f"sequence {seq_id} has more than {max_blocks} blocks")
        out = list(s["blocks"])
        for b in out:
            self.refcount[b] -= 1
            if self.refcount[b] == 0:
                self.free.append(b)
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
        if need > len(self.free):
            raise AllocError("oom", f"need {need} blocks, {len(self.free)} free")
        for _ in range(need):
            b = self.free.pop()
            self.refcount[b] = 1
            s["blocks"].append(b)
        s["swapped"] = False
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
        return len(self.free)
