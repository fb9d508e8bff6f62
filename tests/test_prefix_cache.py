"""The C++ radix-tree prefix cache against the plain prefix-cache model."""
import numpy as np
import pytest

from oracle.block_manager import BlockManager, OutOfBlocks
from oracle.prefix_cache import PrefixCache, create_from_prefix
from paged_kv_cache_127_gb300 import build as pa_build
from paged_kv_cache_127_gb300 import synth


@pytest.fixture(scope="module")
def pa():
    pa_build.build()
    from paged_kv_cache_127_gb300 import binding
    return binding


@pytest.mark.parametrize("seed,B", [(1, 4), (2, 16), (3, 1)])
def test_radix_tree_matches_model(pa, seed, B):
    rng = synth.make_rng(seed)
    N = 400
    order = synth.free_order(rng, N)
    bm, pool = BlockManager(N, B, order), pa.Pool(N, B, order)
    model, cache = PrefixCache(bm), pa.pa_prefix_cache_create(pool.handle)
    # a few prompt families sharing prefixes of varying length, so edges split
    bases = [list(rng.integers(0, 50, size=int(rng.integers(1, 12)) * B)) for _ in range(5)]
    live = []
    for _ in range(1500):
        op = int(rng.integers(0, 10))
        if op <= 4:                                   # a request arrives
            base = bases[int(rng.integers(len(bases)))]
            cut = int(rng.integers(0, len(base) + 1))
            toks = base[:cut] + list(rng.integers(0, 50, size=int(rng.integers(0, 3 * B + 2))))
            want = model.match(toks)
            got = pa.pa_prefix_match(cache, toks).tolist()
            assert got == want
            extra = len(toks) - len(want) * B
            try:
                bm_ok = True
                sid_m = create_from_prefix(bm, want)
                bm.append(sid_m, extra)
            except OutOfBlocks:
                bm_ok = False
                bm.free_seq(sid_m)
            sid_p = pa.pa_seq_create_from_prefix(pool.handle, got)
            assert sid_p == sid_m
            try:
                pa.pa_seq_append(pool.handle, sid_p, extra)
                pool_ok = True
            except pa.PaError:
                pool_ok = False
                pa.pa_seq_free(pool.handle, sid_p)
            assert bm_ok == pool_ok
            if bm_ok:
                assert pa.pa_seq_table(pool.handle, sid_p).tolist() == bm.table(sid_m)
                if rng.random() < 0.7:
                    assert pa.pa_prefix_insert(cache, toks, pa.pa_seq_table(pool.handle, sid_p)) == \
                        model.insert(toks, bm.table(sid_m))
                live.append(sid_m)
        elif op <= 6 and live:                        # a request finishes
            s = live.pop(int(rng.integers(len(live))))
            bm.free_seq(s)
            pa.pa_seq_free(pool.handle, s)
        elif op == 7:                                 # memory pressure
            n = int(rng.integers(0, 6))
            assert pa.pa_prefix_evict(cache, n) == model.evict(n)
        assert pa.pa_prefix_cached_blocks(cache) == model.cached_blocks()
        assert pa.pa_pool_num_free(pool.handle) == bm.num_free()
    for b in range(N):
        assert pa.pa_block_refcount(pool.handle, b) == bm.refcount(b)
    # destroying the cache drops its references; freeing the live sequences empties the pool
    pa.pa_prefix_cache_destroy(cache)
    for s in live:
        pa.pa_seq_free(pool.handle, s)
    assert pa.pa_pool_num_free(pool.handle) == N
    pool.close()


def test_prefix_cache_rejects_bad_blocks(pa):
    with pa.Pool(8, 4) as p:
        c = pa.pa_prefix_cache_create(p.handle)
        with pytest.raises(pa.PaError):
            pa.pa_prefix_insert(c, list(range(8)), [0, 1])      # blocks not allocated
        with pytest.raises(pa.PaError):
            pa.pa_seq_create_from_prefix(p.handle, [9])
        pa.pa_prefix_cache_destroy(c)


def test_a_block_is_cached_under_one_prefix_only(pa):
    with pa.Pool(8, 2) as p:
        bm = BlockManager(8, 2)
        c, model = pa.pa_prefix_cache_create(p.handle), PrefixCache(bm)
        s = pa.pa_seq_create(p.handle)
        pa.pa_seq_append(p.handle, s, 4)
        m = bm.create()
        bm.append(m, 4)
        t = pa.pa_seq_table(p.handle, s)
        assert t.tolist() == bm.table(m)
        assert pa.pa_prefix_insert(c, [1, 2, 3, 4], t) == model.insert([1, 2, 3, 4], bm.table(m)) == 2
        u = pa.pa_seq_create(p.handle)
        pa.pa_seq_append(p.handle, u, 2)
        mu = bm.create()
        bm.append(mu, 2)
        f = int(pa.pa_seq_table(p.handle, u)[0])            # allocated, not cached
        assert f == bm.table(mu)[0]
        for toks, blocks in (([9, 9, 3, 4], t), ([1, 2, 7, 7], [t[0], t[0]]), ([5, 5, 6, 6], [f, f])):
            with pytest.raises(pa.PaError):
                pa.pa_prefix_insert(c, toks, blocks)
            with pytest.raises(ValueError):
                model.insert(toks, blocks)
            assert pa.pa_prefix_cached_blocks(c) == model.cached_blocks() == 2
        pa.pa_seq_free(p.handle, s)
        bm.free_seq(m)
        pa.pa_seq_free(p.handle, u)
        bm.free_seq(mu)
        assert pa.pa_prefix_evict(c, 5) == model.evict(5) == 2
        assert pa.pa_pool_num_free(p.handle) == bm.num_free() == 8
        pa.pa_prefix_cache_destroy(c)


class _Twin:
    """The C++ pool and cache driven in lockstep with the block manager and cache models."""

    def __init__(self, pa, num_blocks, B):
        self.pa = pa
        self.pool = pa.Pool(num_blocks, B)
        self.cache = pa.pa_prefix_cache_create(self.pool.handle)
        self.bm = BlockManager(num_blocks, B)
        self.model = PrefixCache(self.bm)

    def serve(self, toks):
        """A request: reuse the cached prefix, store the rest; returns (sequence, blocks)."""
        got = self.pa.pa_prefix_match(self.cache, toks).tolist()
        assert got == self.model.match(toks)
        sid = self.pa.pa_seq_create_from_prefix(self.pool.handle, got)
        assert sid == create_from_prefix(self.bm, got)
        self.pa.pa_seq_append(self.pool.handle, sid, len(toks) - len(got) * self.bm.B)
        self.bm.append(sid, len(toks) - len(got) * self.bm.B)
        blocks = self.pa.pa_seq_table(self.pool.handle, sid).tolist()
        assert blocks == self.bm.table(sid)
        return sid, blocks

    def insert(self, toks, blocks):
        got = self.pa.pa_prefix_insert(self.cache, toks, blocks)
        assert got == self.model.insert(toks, blocks)
        return got

    def free(self, sid):
        self.pa.pa_seq_free(self.pool.handle, sid)
        self.bm.free_seq(sid)

    def evict(self, n):
        got = self.pa.pa_prefix_evict(self.cache, n)
        assert got == self.model.evict(n)
        return got

    def match(self, toks):
        got = self.pa.pa_prefix_match(self.cache, toks).tolist()
        assert got == self.model.match(toks)
        return got

    def close(self):
        self.pa.pa_prefix_cache_destroy(self.cache)
        self.pool.close()


def test_reinserting_a_prompt_makes_it_recent(pa):
    # an insert stamps the prefixes it finds cached as well as the ones it adds
    t = _Twin(pa, 8, 2)
    p, q = [1, 1, 2, 2], [7, 7]
    s, bp = t.serve(p)
    t.insert(p, bp)
    t.free(s)
    s, bq = t.serve(q)
    t.insert(q, bq)
    t.free(s)
    assert t.insert(p, bp) == 0                 # nothing new: only stamps
    assert t.evict(1) == 1
    assert t.match(q) == [] and t.match(p) == bp
    t.close()


def test_an_edge_split_keeps_the_stamps_of_its_upper_part(pa):
    # the shared first block of two prompts keeps the stamp of its last use when the
    # edge holding it is split, and is evicted after an older, once-held prompt
    t = _Twin(pa, 10, 2)
    held, bh = t.serve([5, 5])
    t.insert([5, 5], bh)
    s, b1 = t.serve([1, 1, 2, 2])
    t.insert([1, 1, 2, 2], b1)
    t.free(s)
    s, b2 = t.serve([1, 1, 3, 3])                # shares b1[0]; its insert splits the edge
    assert b2[0] == b1[0]
    t.insert([1, 1, 3, 3], b2)
    t.free(s)
    assert t.evict(2) == 2                      # the two tails; [5, 5] is still held
    t.free(held)
    assert t.evict(1) == 1                      # the older prompt goes, the shared block stays
    assert t.match([5, 5]) == [] and t.match([1, 1]) == [b1[0]]
    t.close()


def test_a_refused_insert_leaves_no_trace(pa):
    # an insert refused because one of its blocks is cached elsewhere changes nothing:
    # the same prefix with a proper block is accepted afterwards
    t = _Twin(pa, 8, 2)
    sq, bq = t.serve([9, 9])
    t.insert([9, 9], bq)
    sa, ba = t.serve([1, 1, 2, 2])
    with pytest.raises(pa.PaError):
        pa.pa_prefix_insert(t.cache, [1, 1, 2, 2], [ba[0], bq[0]])
    with pytest.raises(ValueError):
        t.model.insert([1, 1, 2, 2], [ba[0], bq[0]])
    assert t.insert([1, 1, 2, 2], ba) == 2
    t.free(sq)
    t.free(sa)
    t.close()
