"""The C++ host allocator in libpa: the pages' worked examples, and bit-exact
agreement with the Python block-manager oracle on random operation streams."""
import json
import os

import numpy as np
import pytest

from oracle import bookkeeping as bk
from oracle.block_manager import BlockManager, OutOfBlocks
from paged_kv_cache_127_gb300 import build as pa_build
from paged_kv_cache_127_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
G = json.load(open(os.path.join(GOLDEN, "block_tables.json")))


@pytest.fixture(scope="module")
def pa():
    pa_build.build()
    from paged_kv_cache_127_gb300 import binding
    return binding


def test_three_requests_and_growth(pa):
    g = G["pool"]
    order = [b for t in g["tables"] for b in t] + [g["allocated"]]
    order += [b for b in range(g["num_blocks"]) if b not in order]
    with pa.Pool(g["num_blocks"], g["block_size"], order) as p:
        seqs = [pa.pa_seq_create(p.handle) for _ in g["lengths"]]
        for s, n in zip(seqs, g["lengths"]):
            pa.pa_seq_append(p.handle, s, n)
        assert [pa.pa_seq_table(p.handle, s).tolist() for s in seqs] == g["tables"]
        assert pa.pa_pool_num_free(p.handle) == g["free_after"]
        s = seqs[g["grow_seq"]]
        slots, pairs = pa.pa_seq_append(p.handle, s, g["grow_by"])
        assert pa.pa_seq_len(p.handle, s) == g["grown_len"]
        assert pa.pa_seq_table(p.handle, s).tolist() == g["grown_table"]
        assert len(pairs) == 0
        # position 37 of this sequence is at (9, 5)
        t = g["grown_table"]
        assert t[37 // 16] * 16 + 37 % 16 == 9 * 16 + 5


def test_full_prefix_and_partial_cow(pa):
    gf = G["full_prefix"]
    with pa.Pool(64, 16) as p:
        a = pa.pa_seq_create(p.handle)
        pa.pa_seq_append(p.handle, a, gf["prefix"])
        b = pa.pa_seq_fork(p.handle, a)
        _, pairs = pa.pa_seq_append(p.handle, b, 1)
        assert len(pairs) == gf["cow_pairs_on_next_token"]
        assert len(pa.pa_seq_table(p.handle, a)) == gf["prefix_blocks"]
    gc = G["partial_cow"]
    with pa.Pool(8, gc["block_size"]) as p:
        a = pa.pa_seq_create(p.handle)
        pa.pa_seq_append(p.handle, a, gc["shared_tokens"])
        b = pa.pa_seq_fork(p.handle, a)
        slots, pairs = pa.pa_seq_append(p.handle, b, 1)
        assert pairs.tolist() == [gc["copy_pair"]]
        assert pa.pa_seq_table(p.handle, b).tolist() == gc["b_table_after"]
        assert pa.pa_seq_table(p.handle, a).tolist() == gc["a_table_after"]
        assert {str(k): pa.pa_block_refcount(p.handle, k) for k in (0, 1, 2)} == gc["refcounts_after"]
        assert divmod(int(slots[0]), 16) == (gc["b_new_slot_block"], gc["b_new_slot_offset"])


def test_refcount_teardown(pa):
    with pa.Pool(4, 16) as p:
        a = pa.pa_seq_create(p.handle)
        pa.pa_seq_append(p.handle, a, 16)
        b = pa.pa_seq_fork(p.handle, a)
        p0 = int(pa.pa_seq_table(p.handle, a)[0])
        pa.pa_seq_free(p.handle, a)
        assert pa.pa_block_refcount(p.handle, p0) == 1 and pa.pa_pool_num_free(p.handle) == 3
        pa.pa_seq_free(p.handle, b)
        assert pa.pa_block_refcount(p.handle, p0) == 0 and pa.pa_pool_num_free(p.handle) == 4


def test_stats_match_worked_example_1(pa):
    lengths = [47, 612, 130, 1900]
    with pa.Pool(200, 16) as p:
        for n in lengths:
            pa.pa_seq_append(p.handle, pa.pa_seq_create(p.handle), n)
        st = pa.pa_pool_get_stats(p.handle)
    ref = bk.fragmentation(lengths, 16, 2048)
    assert st["used_blocks"] == ref["total_blocks"] == 170
    assert st["table_slots"] == ref["paged_slots"] == 2720
    assert st["tokens"] == ref["tokens"] == 2689
    assert st["padded_slots"] == ref["paged_waste"] == 31


def test_oom_rolls_back_and_fault_injection(pa):
    with pa.Pool(3, 4) as p:
        a = pa.pa_seq_create(p.handle)
        pa.pa_seq_append(p.handle, a, 6)
        b = pa.pa_seq_fork(p.handle, a)
        before = (pa.pa_seq_table(p.handle, a).tolist(), pa.pa_seq_table(p.handle, b).tolist(),
                  pa.pa_pool_num_free(p.handle), pa.pa_seq_len(p.handle, b))
        with pytest.raises(pa.PaError) as e:
            pa.pa_seq_append(p.handle, b, 7)
        assert e.value.status == pa.PA_ERR_OOM
        after = (pa.pa_seq_table(p.handle, a).tolist(), pa.pa_seq_table(p.handle, b).tolist(),
                 pa.pa_pool_num_free(p.handle), pa.pa_seq_len(p.handle, b))
        assert before == after
        pa.pa_pool_set_fail_after(p.handle, 0)
        with pytest.raises(pa.PaError):
            pa.pa_seq_append(p.handle, a, 3)
        pa.pa_pool_set_fail_after(p.handle, None)
        pa.pa_seq_append(p.handle, a, 2)          # fits in block 1 after the limit is lifted


def test_bad_ids_and_arguments(pa):
    assert pa.lib.pa_pool_create(0, 16, None) is None
    with pytest.raises(pa.PaError):
        pa.pa_pool_create(4, 16, [0, 1, 1, 2])    # not a permutation
    with pa.Pool(4, 16) as p:
        with pytest.raises(pa.PaError) as e:
            pa.pa_seq_fork(p.handle, 5)
        assert e.value.status == pa.PA_ERR_BAD_INDEX
        s = pa.pa_seq_create(p.handle)
        pa.pa_seq_free(p.handle, s)
        with pytest.raises(pa.PaError):
            pa.pa_seq_free(p.handle, s)           # already freed
        with pytest.raises(pa.PaError):
            pa.pa_block_refcount(p.handle, 4)
        s2 = pa.pa_seq_create(p.handle)
        with pytest.raises(pa.PaError) as e:
            pa.pa_seq_append_batch(p.handle, [s2, s2], 1)
        assert e.value.status == pa.PA_ERR_INVALID
        with pytest.raises(pa.PaError) as e:
            pa.pa_seq_append_batch(p.handle, [s2, s], 1)   # s was freed
        assert e.value.status == pa.PA_ERR_BAD_INDEX
        assert pa.pa_seq_len(p.handle, s2) == 0 and pa.pa_pool_num_free(p.handle) == 4
        pa.pa_seq_append(p.handle, s2, 20)
        with pytest.raises(pa.PaError) as e:
            pa.pa_pool_export(p.handle, [s2], 1)            # two blocks do not fit one column
        assert e.value.status == pa.PA_ERR_INVALID


def test_copy_pairs_check(pa):
    # a copy-on-write copy goes to a fresh block: ids in range, destinations distinct
    # and never a source; several copies may read one source
    pa.pa_copy_pairs_check([[3, 7], [3, 9], [0, 11]], 12)
    pa.pa_copy_pairs_check(np.zeros((0, 2), np.int64), 12)
    for bad, status in (([[3, 7], [4, 7]], pa.PA_ERR_INVALID),     # destination twice
                        ([[3, 7], [7, 9]], pa.PA_ERR_INVALID),     # a destination is also a source
                        ([[5, 5]], pa.PA_ERR_INVALID),
                        ([[3, 12]], pa.PA_ERR_BAD_INDEX),
                        ([[-1, 2]], pa.PA_ERR_BAD_INDEX)):
        with pytest.raises(pa.PaError) as e:
            pa.pa_copy_pairs_check(bad, 12)
        assert e.value.status == status
    assert pa.lib.pa_copy_pairs_check(None, 1, 12) == pa.PA_ERR_INVALID
    assert pa.lib.pa_copy_pairs_check(None, -1, 12) == pa.PA_ERR_INVALID
    assert pa.lib.pa_copy_pairs_check(None, 0, 0) == pa.PA_ERR_INVALID


def test_batch_counts_a_copy_that_spares_the_next_sharer(pa):
    # two sequences share a partly filled block and both append in one batch: the
    # first copies it, after which the second holds it alone and writes in place,
    # so one free block is enough (the model, appending one after the other, agrees)
    bm = BlockManager(3, 16)
    a = bm.create()
    bm.append(a, 24)
    b = bm.fork(a)
    want = [bm.append(a, 1), bm.append(b, 1)]
    with pa.Pool(3, 16) as p:
        pa_a = pa.pa_seq_create(p.handle)
        pa.pa_seq_append(p.handle, pa_a, 24)
        pa_b = pa.pa_seq_fork(p.handle, pa_a)
        slots, pairs = pa.pa_seq_append_batch(p.handle, [pa_a, pa_b], 1)
        assert slots.tolist() == [w[0] for w in want]
        assert [tuple(x) for x in pairs.tolist()] == want[0][1] + want[1][1]
        assert pa.pa_pool_num_free(p.handle) == bm.num_free() == 0


def _run_stream(pa, seed, num_blocks, B, steps, batch):
    """Drive the C++ pool and the oracle model with one random operation stream."""
    rng = synth.make_rng(seed)
    order = synth.free_order(rng, num_blocks)
    bm = BlockManager(num_blocks, B, order)
    p = pa.Pool(num_blocks, B, order)
    live = []
    ops = 0
    for _ in range(steps):
        op = int(rng.integers(0, 12))
        if op == 0 or not live:
            a, b = bm.create(), pa.pa_seq_create(p.handle)
            assert a == b
            live.append(a)
        elif op == 1:
            par = live[int(rng.integers(len(live)))]
            a, b = bm.fork(par), pa.pa_seq_fork(p.handle, par)
            assert a == b
            live.append(a)
        elif op == 2:
            s = live.pop(int(rng.integers(len(live))))
            bm.free_seq(s)
            pa.pa_seq_free(p.handle, s)
        elif op == 3:
            n = int(rng.integers(0, 3))
            bm.set_fail_after(n)
            pa.pa_pool_set_fail_after(p.handle, n)
        elif op == 4:
            bm.set_fail_after(None)
            pa.pa_pool_set_fail_after(p.handle, None)
        elif batch and op >= 9:
            k = int(rng.integers(1, len(live) + 1))
            seqs = [int(x) for x in rng.choice(live, size=k, replace=False)]
            n = int(rng.integers(0, 5))
            snap = ([list(bm.table(s)) for s in live], list(bm.free), list(bm.ref),
                    {s: bm.length(s) for s in live}, bm._fail_budget, bm.cow_copies)
            try:
                want_slots, want_pairs = [], []
                for s in seqs:
                    sl, pr = bm.append(s, n)
                    want_slots.append(sl)
                    want_pairs += pr
                ok = True
            except OutOfBlocks:
                ok = False
                # batch is all-or-nothing: undo the model's partial progress
                for s, t in zip(live, snap[0]):
                    bm.seqs[s].table = t
                    bm.seqs[s].length = snap[3][s]
                bm.free = type(bm.free)(snap[1])
                bm.ref = snap[2]
                bm._fail_budget = snap[4]
                bm.cow_copies = snap[5]
            try:
                slots, pairs = pa.pa_seq_append_batch(p.handle, seqs, n)
                got = True
            except pa.PaError as e:
                assert e.status == pa.PA_ERR_OOM
                got = False
            assert ok == got
            if ok:
                assert slots.tolist() == want_slots
                assert [tuple(x) for x in pairs.tolist()] == want_pairs
                pa.pa_copy_pairs_check(pairs, num_blocks)
        else:
            s = live[int(rng.integers(len(live)))]
            n = int(rng.integers(0, 2 * B + 3))
            try:
                want = bm.append(s, n)
            except OutOfBlocks:
                want = None
            try:
                slots, pairs = pa.pa_seq_append(p.handle, s, n)
                got = (slots.tolist(), [tuple(x) for x in pairs.tolist()])
            except pa.PaError as e:
                assert e.status == pa.PA_ERR_OOM
                got = None
            assert got == want
        ops += 1
        for s in live:
            assert pa.pa_seq_table(p.handle, s).tolist() == bm.table(s)
            assert pa.pa_seq_len(p.handle, s) == bm.length(s)
        assert pa.pa_pool_num_free(p.handle) == bm.num_free()
        if live and ops % 50 == 0:
            width = max(len(bm.table(s)) for s in live) + 2
            tables, lens = pa.pa_pool_export(p.handle, live, width, pad=-7)
            assert tables.tolist() == [bm.table(s) + [-7] * (width - len(bm.table(s))) for s in live]
            assert lens.tolist() == [bm.length(s) for s in live]
    for blk in range(num_blocks):
        assert pa.pa_block_refcount(p.handle, blk) == bm.refcount(blk)
    st = pa.pa_pool_get_stats(p.handle)
    ref = bm.stats()
    for k in ("free", "used", "shared", "cow_copies", "tokens", "table_slots", "padded_slots"):
        assert st[{"free": "free_blocks", "used": "used_blocks", "shared": "shared_blocks"}.get(k, k)] == ref[k]
    assert st["live_seqs"] == len(bm.seqs) == len(live)
    p.close()
    return ops


@pytest.mark.parametrize("seed,num_blocks,B,batch", [(1, 64, 16, False), (2, 40, 4, True),
                                                      (3, 300, 32, True), (4, 12, 1, True)])
def test_matches_block_manager_oracle(pa, seed, num_blocks, B, batch):
    assert _run_stream(pa, seed, num_blocks, B, 1500, batch) == 1500


def test_swap_matches_block_manager_oracle(pa):
    """Random create / fork / append / free / swap-out / swap-in streams on a device
    pool and a host pool: the C++ pools and the oracle model agree exactly."""
    rng = synth.make_rng(77)
    B = 8
    order_d = synth.free_order(rng, 60)
    order_h = synth.free_order(rng, 40)
    bd, bh = BlockManager(60, B, order_d), BlockManager(40, B, order_h)
    pd, ph = pa.Pool(60, B, order_d), pa.Pool(40, B, order_h)
    live, swapped = [], []
    for _ in range(2000):
        op = int(rng.integers(0, 8))
        if op == 0 or not live:
            a, b = bd.create(), pa.pa_seq_create(pd.handle)
            assert a == b
            live.append(a)
        elif op == 1:
            par = live[int(rng.integers(len(live)))]
            a, b = bd.fork(par), pa.pa_seq_fork(pd.handle, par)
            assert a == b
            live.append(a)
        elif op == 2:
            s = live.pop(int(rng.integers(len(live))))
            bd.free_seq(s)
            pa.pa_seq_free(pd.handle, s)
        elif op == 3:
            s = live[int(rng.integers(len(live)))]
            try:
                want = bd.swap_out(s, bh)
            except OutOfBlocks:
                want = None
            try:
                hid, pairs = pa.pa_seq_swap_out(pd.handle, ph.handle, s)
                got = (hid, [tuple(x) for x in pairs.tolist()])
            except pa.PaError as e:
                assert e.status == pa.PA_ERR_OOM
                got = None
            assert got == want
            if got:
                live.remove(s)
                swapped.append(got[0])
        elif op == 4 and swapped:
            h = swapped[int(rng.integers(len(swapped)))]
            try:
                want = bd.swap_in(h, bh)
            except OutOfBlocks:
                want = None
            try:
                sid, pairs = pa.pa_seq_swap_in(pd.handle, ph.handle, h)
                got = (sid, [tuple(x) for x in pairs.tolist()])
            except pa.PaError as e:
                assert e.status == pa.PA_ERR_OOM
                got = None
            assert got == want
            if got:
                swapped.remove(h)
                live.append(got[0])
        else:
            s = live[int(rng.integers(len(live)))]
            n = int(rng.integers(0, 2 * B + 3))
            try:
                want = bd.append(s, n)
            except OutOfBlocks:
                want = None
            try:
                slots, pairs = pa.pa_seq_append(pd.handle, s, n)
                got = (slots.tolist(), [tuple(x) for x in pairs.tolist()])
            except pa.PaError as e:
                assert e.status == pa.PA_ERR_OOM
                got = None
            assert got == want
        for s in live:
            assert pa.pa_seq_table(pd.handle, s).tolist() == bd.table(s)
        for h in swapped:
            assert pa.pa_seq_table(ph.handle, h).tolist() == bh.table(h)
            assert pa.pa_seq_len(ph.handle, h) == bh.length(h)
        assert pa.pa_pool_num_free(pd.handle) == bd.num_free()
        assert pa.pa_pool_num_free(ph.handle) == bh.num_free()
    pd.close()
    ph.close()
