"""Pins for the Python block-manager model (the allocator's oracle)."""
import json
import os

import pytest

from oracle.block_manager import BlockManager, OutOfBlocks
from paged_kv_cache_127_gb300 import synth

G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "block_tables.json")))


def _pool_example():
    g = G["pool"]
    order = [b for t in g["tables"] for b in t] + [g["allocated"]]
    order += [b for b in range(g["num_blocks"]) if b not in order]
    bm = BlockManager(g["num_blocks"], g["block_size"], order)
    seqs = []
    for n in g["lengths"]:
        s = bm.create()
        bm.append(s, n)
        seqs.append(s)
    return g, bm, seqs


def test_three_requests_tables_and_free_count():
    g, bm, seqs = _pool_example()
    assert [bm.table(s) for s in seqs] == g["tables"]
    assert bm.num_free() == g["free_after"]


def test_pool_statistics_of_the_three_requests():
    # "Where contiguous allocation wastes space": 25, 47 and 12 tokens take 96 slots
    # in 16-token blocks, 12 of them padding; a fork shares every block of its parent
    f = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "fragmentation.json")))["cases"][0]
    g, bm, seqs = _pool_example()
    st = bm.stats()
    assert (st["tokens"], st["table_slots"], st["padded_slots"]) == (f["tokens"], f["paged_slots"], f["paged_waste"])
    assert (st["used"], st["shared"], st["free"]) == (sum(f["blocks"]), 0, g["free_after"])
    bm.fork(seqs[1])
    st = bm.stats()
    assert (st["used"], st["shared"]) == (sum(f["blocks"]), f["blocks"][1])


def test_growth_adds_one_block_and_keeps_entries():
    g, bm, seqs = _pool_example()
    s = seqs[g["grow_seq"]]
    before = bm.table(s)
    slots, pairs = bm.append(s, g["grow_by"])
    assert bm.length(s) == g["grown_len"]
    assert bm.table(s) == g["grown_table"]
    assert bm.table(s)[:len(before)] == before
    assert len(bm.table(s)) == g["grown_blocks"] and pairs == []
    # slots of the 10 new tokens: positions 47..56 through [0, 5, 9, 11]
    assert slots == [9 * 16 + 15] + [11 * 16 + o for o in range(9)]


def test_twenty_more_tokens_need_five_blocks():
    g, bm, seqs = _pool_example()
    bm.append(seqs[g["grow_seq"]], g["grow_by_alt"])
    assert len(bm.table(seqs[g["grow_seq"]])) == g["grown_blocks_alt"]


def test_full_shared_prefix_needs_no_copy():
    g = G["full_prefix"]
    bm = BlockManager(64, g["block_size"])
    a = bm.create()
    bm.append(a, g["prefix"])
    assert len(bm.table(a)) == g["prefix_blocks"]
    b = bm.fork(a)
    slots, pairs = bm.append(b, 1)
    assert len(pairs) == g["cow_pairs_on_next_token"]
    assert bm.table(b)[:50] == bm.table(a) and len(bm.table(b)) == 51
    assert bm.refcount(bm.table(b)[-1]) == 1
    assert all(bm.refcount(x) == 2 for x in bm.table(a))


def test_partial_shared_block_is_copied_on_write():
    g = G["partial_cow"]
    bm = BlockManager(8, g["block_size"])
    a = bm.create()
    bm.append(a, g["shared_tokens"])
    assert bm.table(a) == g["shared_table"]
    b = bm.fork(a)
    slots, pairs = bm.append(b, 1)
    assert pairs == [tuple(g["copy_pair"])]
    assert bm.table(b) == g["b_table_after"]
    assert bm.table(a) == g["a_table_after"]
    assert {str(k): bm.refcount(k) for k in (0, 1, 2)} == g["refcounts_after"]
    assert divmod(slots[0], g["block_size"]) == (g["b_new_slot_block"], g["b_new_slot_offset"])
    # A's next write lands in P1 in place: it is no longer shared
    slots_a, pairs_a = bm.append(a, 1)
    assert pairs_a == [] and slots_a == [1 * 16 + 8]


def test_refcount_teardown():
    g = G["refcount_teardown"]
    bm = BlockManager(4, 16)
    a = bm.create()
    bm.append(a, 16)
    b = bm.fork(a)
    p0 = bm.table(a)[0]
    assert bm.refcount(p0) == g["refcount_before"]
    bm.free_seq(a)
    assert bm.refcount(p0) == g["refcount_after_a"]
    assert (p0 in bm.free) == g["freed_after_a"]
    bm.free_seq(b)
    assert (p0 in bm.free) == g["freed_after_b"]



def test_freed_blocks_rejoin_the_back_of_the_free_list():
    # the pages leave the choice of free block open ("Growing a request" hands out
    # P11); the reading taken is a FIFO list: a freed block is handed out again only
    # after every block that was already free
    bm = BlockManager(4, 16)
    a, b = bm.create(), bm.create()
    bm.append(a, 16)
    bm.append(b, 16)
    assert (bm.table(a), bm.table(b)) == ([0], [1])
    bm.free_seq(a)
    assert list(bm.free) == [2, 3, 0]
    c = bm.create()
    bm.append(c, 48)
    assert bm.table(c) == [2, 3, 0]


def test_appending_nothing_changes_nothing():
    # zero new tokens write no slot, so even a shared, partly filled last block is
    # not copied; a negative count is refused
    bm = BlockManager(8, 16)
    a = bm.create()
    bm.append(a, 24)
    b = bm.fork(a)
    snap = (bm.table(a), bm.table(b), list(bm.free), list(bm.ref))
    assert bm.append(b, 0) == ([], [])
    assert (bm.table(a), bm.table(b), list(bm.free), list(bm.ref)) == snap
    with pytest.raises(ValueError):
        bm.append(b, -1)
    assert (bm.table(a), bm.table(b), list(bm.free), list(bm.ref)) == snap


def test_bad_pools_are_refused_and_copies_counted():
    with pytest.raises(ValueError):
        BlockManager(0, 16)
    with pytest.raises(ValueError):
        BlockManager(4, 16, [0, 1, 1, 2])          # not a permutation of the ids
    # one copy-on-write ("Sharing a prefix and copying a partial block") is one copy
    bm = BlockManager(8, 16)
    a = bm.create()
    bm.append(a, 24)
    b = bm.fork(a)
    bm.append(b, 1)
    bm.append(b, 1)                                 # b's block is private now: no second copy
    assert bm.stats()["cow_copies"] == 1


def test_fault_injection_counts_down():
    # after set_fail_after(2) exactly two more block allocations succeed
    bm = BlockManager(8, 16)
    a = bm.create()
    bm.set_fail_after(2)
    bm.append(a, 32)
    with pytest.raises(OutOfBlocks):
        bm.append(a, 1)
    assert bm.length(a) == 32 and bm.num_free() == 6
    bm.set_fail_after(None)
    bm.append(a, 1)
    assert bm.num_free() == 5


def test_out_of_blocks_changes_nothing():
    bm = BlockManager(3, 4)
    a = bm.create()
    bm.append(a, 6)
    b = bm.fork(a)
    snap = (bm.table(a), bm.table(b), list(bm.free), list(bm.ref))
    with pytest.raises(OutOfBlocks):
        bm.append(b, 7)                    # needs a copy + 2 new blocks, only 1 free
    assert (bm.table(a), bm.table(b), list(bm.free), list(bm.ref)) == snap
    bm.set_fail_after(0)
    with pytest.raises(OutOfBlocks):
        bm.append(a, 3)
    assert (bm.table(a), bm.table(b), list(bm.free), list(bm.ref)) == snap


def test_random_operations_keep_the_invariants():
    rng = synth.make_rng(21)
    bm = BlockManager(200, 8, synth.free_order(rng, 200))
    live = []
    for step in range(3000):
        op = rng.integers(0, 10)
        try:
            if op == 0 or not live:
                live.append(bm.create())
            elif op == 1:
                live.append(bm.fork(live[rng.integers(len(live))]))
            elif op == 2:
                bm.free_seq(live.pop(rng.integers(len(live))))
            else:
                bm.append(live[rng.integers(len(live))], int(rng.integers(0, 20)))
        except OutOfBlocks:
            pass
        # refcount = number of tables listing the block; free <=> refcount 0
        counts = [0] * 200
        for s in live:
            t = bm.table(s)
            assert len(t) == -(-bm.length(s) // 8)
            for x in t:
                counts[x] += 1
        assert counts == bm.ref
        assert sorted(bm.free) == [x for x in range(200) if counts[x] == 0]


def test_swap_out_and_in_keeps_tables_and_sharing_rules():
    dev = BlockManager(12, 4)
    host = BlockManager(8, 4)
    a = dev.create()
    dev.append(a, 10)                       # blocks 0, 1, 2
    b = dev.fork(a)                         # shares all three
    dev.append(b, 3)                        # b copies block 2 (partial) and grows
    shared = dev.table(a)[:2]
    b_table = dev.table(b)
    hid, pairs = dev.swap_out(b, host)
    assert [p[0] for p in pairs] == b_table          # every entry, in table order
    assert len(pairs) == 4 and host.length(hid) == 13
    assert [p[1] for p in pairs] == host.table(hid)
    # the blocks b shared with a stay on the device, with a's reference only
    assert all(dev.refcount(x) == 1 for x in shared)
    assert b not in dev.seqs and dev.table(a)[:2] == shared
    # the blocks only b used are free again on the device
    assert dev.num_free() == 12 - 3
    sid, back = dev.swap_in(hid, host)
    assert [p[0] for p in back] == [p[1] for p in pairs]
    assert dev.table(sid) == [p[1] for p in back] and dev.length(sid) == 13
    assert all(dev.refcount(x) == 1 for x in dev.table(sid))     # private after swap-in
    assert host.num_free() == 8 and hid not in host.seqs


def test_swap_is_all_or_nothing():
    dev = BlockManager(8, 4)
    host = BlockManager(2, 4)
    a = dev.create()
    dev.append(a, 12)                       # 3 blocks, host has 2
    snap = (dev.table(a), list(dev.free), list(host.free))
    with pytest.raises(OutOfBlocks):
        dev.swap_out(a, host)
    assert (dev.table(a), list(dev.free), list(host.free)) == snap
