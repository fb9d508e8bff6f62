"""Plain model of the block-level prefix cache -- TEST INFRASTRUCTURE ONLY.

"KV Cache Optimization and Management", "RadixAttention: caching, not just
packing, the prefix": requests that start with the same tokens reuse the
blocks already computed for them; when memory runs low the least recently
used cached leaves are dropped, and reference counts keep anything a running
request still uses.  Only whole blocks are reused ("PagedAttention: Virtual
Memory for the KV Cache", "Sharing a prefix and copying a partial block";
answer A3 of the chapter above counts whole shareable blocks).

This model keeps no tree: it stores every cached block-aligned prefix (a
tuple of tokens) with its block and a last-use stamp, which is the plain
statement of what the radix tree in the library represents.  Rules:

* match: the longest cached prefix of the request; its prefixes get a new stamp;
* insert: every missing prefix of the first min(len(blocks), len(tokens) // B)
  blocks is cached with the caller's block (the cache takes a reference);
  prefixes already cached keep their block; all of them get a new stamp; a
  block already cached, or given twice among the new ones, is refused and
  nothing changes (a physical block holds the K/V of one prefix);
* evict(n): repeatedly drop a cached prefix that no longer prefix extends and
  whose block only the cache references, smallest (stamp, block) first.
"""
from __future__ import annotations

from .block_manager import BlockManager


class PrefixCache:
    def __init__(self, bm: BlockManager):
        self.bm = bm
        self.B = bm.B
        self.entries: dict[tuple, list] = {}   # prefix -> [block, stamp]
        self.clock = 0

    def match(self, tokens) -> list:
        self.clock += 1
        out = []
        k = 1
        while k * self.B <= len(tokens):
            e = self.entries.get(tuple(tokens[:k * self.B]))
            if e is None:
                break
            e[1] = self.clock
            out.append(e[0])
            k += 1
        return out

    def insert(self, tokens, blocks) -> int:
        m = min(len(blocks), len(tokens) // self.B)
        if any(not 0 <= int(b) < self.bm.num_blocks or self.bm.ref[int(b)] < 1 for b in blocks[:m]):
            raise IndexError("insert: block not allocated")
        new = [int(blocks[k - 1]) for k in range(1, m + 1) if tuple(tokens[:k * self.B]) not in self.entries]
        held = {e[0] for e in self.entries.values()}
        if len(set(new)) != len(new) or any(b in held for b in new):
            raise ValueError("insert: a block may be cached under one prefix only")
        self.clock += 1
        added = 0
        for k in range(1, m + 1):
            p = tuple(tokens[:k * self.B])
            if p in self.entries:
                self.entries[p][1] = self.clock
            else:
                self.entries[p] = [int(blocks[k - 1]), self.clock]
                self.bm.ref[int(blocks[k - 1])] += 1
                added += 1
        return added

    def evict(self, n) -> int:
        freed = 0
        while freed < n:
            extended = {p[:-self.B] for p in self.entries}
            leaves = [p for p in self.entries if p not in extended and self.bm.ref[self.entries[p][0]] == 1]
            if not leaves:
                break
            victim = min(leaves, key=lambda p: (self.entries[p][1], self.entries[p][0]))
            block = self.entries.pop(victim)[0]
            self.bm._release(block)
            freed += 1
        return freed

    def cached_blocks(self) -> int:
        return len(self.entries)


def create_from_prefix(bm: BlockManager, blocks) -> int:
    """A new sequence starting with existing blocks (one more reference each)."""
    sid = bm.create()
    bm.seqs[sid].table = [int(b) for b in blocks]
    bm.seqs[sid].length = len(blocks) * bm.B
    for b in blocks:
        bm.ref[int(b)] += 1
    return sid
