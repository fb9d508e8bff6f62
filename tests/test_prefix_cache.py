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
