"""Plain Python model of the paged KV block manager -- TEST INFRASTRUCTURE ONLY.

It restates, step by step, the bookkeeping rules the pages give, and is the
oracle the C++ allocator in the product library is compared against:

* fixed-size physical blocks of B token slots in one shared pool
  ("Paged Attention and vLLM", "Block Table and Logical-to-Physical Mapping");
* a per-sequence block table; token ``pos`` lives at offset ``pos % B`` of
  physical block ``table[pos // B]`` ("PagedAttention: Virtual Memory for the
  KV Cache", "A block table preserves token order");
* growth: a new block is taken from the free pool only when the last block
  is full, and existing entries never move (same page, "Growing a request");
* a reference count per block; a block returns to the free pool only when its
  count reaches zero ("KV Cache Optimization and Management", "PagedAttention:
  borrowing virtual memory" and active-recall answer A6);
* prefix sharing by forking a table; copy-on-write of a *partially filled*
  shared last block before a sequence writes into it: allocate p', copy
  p -> p', redirect the writer's table, adjust counts, write into p'
  ("PagedAttention: Virtual Memory for the KV Cache", "Sharing a prefix and
  copying a partial block"; "Paged Attention and vLLM", "Continuous Batching
  and Scheduler").  A full shared block needs no copy: the next token goes to a
  new private block.

Readings where the pages leave the policy open:

* which free block is handed out: the pool keeps a FIFO free list, initialised
  from a caller-supplied order (ascending ids by default); allocations pop the
  front, freed blocks are pushed at the back;
* the first writer into a shared partial block gets the private copy; the
  other sharers keep the original;
* an append that cannot get all the blocks it needs fails as a whole and
  changes nothing (out-of-memory with rollback); the policy for what to do
  next belongs to a scheduler ("Growing a request", last paragraph);
* within one append, the copy-on-write block is allocated before any new
  growth block;
* sequence ids are handed out 0, 1, 2, ... and never reused;
* swapping a sequence out ("Paged Attention and vLLM", "Continuous Batching
  and Scheduler": evict its physical blocks to CPU, bring them back later)
  gives every table entry a private host block -- blocks it shared stay with
  their other users on the device and are duplicated on the host -- and
  swapping in gives every entry a fresh private device block.
"""
from __future__ import annotations

from collections import deque
from dataclasses import dataclass, field


class OutOfBlocks(Exception):
    """The pool cannot supply the blocks an operation needs; nothing was changed."""


@dataclass
class _Seq:
    table: list = field(default_factory=list)
    length: int = 0


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of the block ids")
        self.num_blocks = num_blocks
        self.B = block_size
        self.free = deque(order)
        self.ref = [0] * num_blocks
        self.seqs: dict[int, _Seq] = {}
        self._next_id = 0
        self._fail_budget = None      # allocations allowed before injected failure
        self.cow_copies = 0

    # -- helpers --------------------------------------------------------------
    def _alloc(self) -> int:
        b = self.free.popleft()
        self.ref[b] = 1
        if self._fail_budget is not None:
            self._fail_budget -= 1
        return b

    def _release(self, b: int) -> None:
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free.append(b)

    def set_fail_after(self, n):
        """Let only ``n`` more block allocations succeed (None: no limit)."""
        self._fail_budget = None if n is None or n < 0 else int(n)

    # -- sequence operations ----------------------------------------------------
    def create(self) -> int:
        sid = self._next_id
        self._next_id += 1
        self.seqs[sid] = _Seq()
        return sid

    def fork(self, parent: int) -> int:
        p = self.seqs[parent]
        sid = self.create()
        self.seqs[sid].table = list(p.table)
        self.seqs[sid].length = p.length
        for b in p.table:
            self.ref[b] += 1
        return sid

    def append(self, sid: int, n: int):
        """Store n more tokens; return (slots, cow_pairs)."""
        s = self.seqs[sid]
        if n < 0:
            raise ValueError("n must be >= 0")
        B = self.B
        # blocks to add for growth: ceil((len+n)/B) - ceil(len/B)
        grow = -(-(s.length + n) // B) - (-(-s.length // B))
        # copy-on-write if the next token lands in a partially filled shared block
        cow = n > 0 and s.length % B != 0 and self.ref[s.table[-1]] > 1
        need = grow + (1 if cow else 0)
        if need > len(self.free) or (self._fail_budget is not None and need > self._fail_budget):
            raise OutOfBlocks(f"need {need} blocks, {len(self.free)} free")
        pairs = []
        if cow:
            old = s.table[-1]
            new = self._alloc()
            pairs.append((old, new))
            self.ref[old] -= 1          # stays >= 1: another sequence still holds it
            s.table[-1] = new
            self.cow_copies += 1
        slots = []
        for pos in range(s.length, s.length + n):
            logical, offset = divmod(pos, B)
            if logical == len(s.table):
                s.table.append(self._alloc())
            slots.append(s.table[logical] * B + offset)
        s.length += n
        return slots, pairs

    def free_seq(self, sid: int) -> None:
        s = self.seqs.pop(sid)
        for b in s.table:
            self._release(b)

    # -- preemption: swap a sequence to another pool and back ---------------------
    def swap_out(self, sid: int, host: "BlockManager"):
        """Move sequence `sid` into `host`: a private host block per table entry,
        then release the device sequence.  Returns (host id, [(device, host)]).
        All-or-nothing: OutOfBlocks if `host` is short."""
        s = self.seqs[sid]
        if len(s.table) > len(host.free) or (host._fail_budget is not None and len(s.table) > host._fail_budget):
            raise OutOfBlocks("host pool too small")
        hid = host.create()
        pairs = []
        for b in s.table:
            hb = host._alloc()
            host.seqs[hid].table.append(hb)
            pairs.append((b, hb))
        host.seqs[hid].length = s.length
        self.free_seq(sid)
        return hid, pairs

    def swap_in(self, hid: int, host: "BlockManager"):
        """Move host sequence `hid` back: fresh private blocks here, then release
        it in `host`.  Returns (new id, [(host, device)])."""
        hs = host.seqs[hid]
        if len(hs.table) > len(self.free) or (self._fail_budget is not None and len(hs.table) > self._fail_budget):
            raise OutOfBlocks("device pool too small")
        sid = self.create()
        pairs = []
        for hb in hs.table:
            b = self._alloc()
            self.seqs[sid].table.append(b)
            pairs.append((hb, b))
        self.seqs[sid].length = hs.length
        host.free_seq(hid)
        return sid, pairs

    # -- queries ----------------------------------------------------------------
    def table(self, sid: int) -> list:
        return list(self.seqs[sid].table)

    def length(self, sid: int) -> int:
        return self.seqs[sid].length

    def num_free(self) -> int:
        return len(self.free)

    def refcount(self, b: int) -> int:
        return self.ref[b]

    def stats(self) -> dict:
        """Pool-wide counts used by the fragmentation analysis."""
        used = sum(1 for r in self.ref if r > 0)
        shared = sum(1 for r in self.ref if r > 1)
        tokens = sum(s.length for s in self.seqs.values())
        slots = sum(len(s.table) for s in self.seqs.values()) * self.B   # per-sequence view
        return {"free": len(self.free), "used": used, "shared": shared,
                "cow_copies": self.cow_copies, "tokens": tokens,
                "table_slots": slots, "padded_slots": slots - tokens}
