"""Pins for the prefix-cache model against the pages' sharing arithmetic."""
import json
import os

import pytest

from oracle import bookkeeping as bk
from oracle.block_manager import BlockManager
from oracle.prefix_cache import PrefixCache, create_from_prefix

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "sharing.json")))


def _serve(bm, cache, prompt, suffix_tokens):
    """One request: reuse the cached prompt blocks, store the rest, cache the prompt."""
    blocks = cache.match(prompt)
    sid = create_from_prefix(bm, blocks)
    bm.append(sid, len(prompt) + suffix_tokens - len(blocks) * bm.B)
    cache.insert(prompt, bm.table(sid))
    return sid


@pytest.mark.parametrize("case", GOLDEN["full_blocks"], ids=lambda c: str(c["block_size"]))
def test_a_repeated_prompt_reuses_its_whole_blocks(case):
    # answer A3: of a 380-token prompt, 23 blocks of 16 (368 tokens) or 5 of 64 (320) are reusable
    B = case["block_size"]
    bm = BlockManager(200, B)
    cache = PrefixCache(bm)
    prompt = list(range(1000, 1000 + case["prompt"]))
    _serve(bm, cache, prompt, 90)
    assert len(cache.match(prompt + [7] * 90)) == case["full_blocks"]
    assert len(cache.match(prompt)) * B == case["tokens"]
    # the partly filled last prompt block is not cached at all
    assert cache.cached_blocks() == case["full_blocks"]


def test_q5_shared_prompt_block_count():
    # answer A5: 512-token prompt, 1,000 requests with 60 own tokens, B = 16:
    # 32 shared + 4 per request = 4,032 blocks, against 36,000 unshared
    case = GOLDEN["shared_prompt"][1]
    B, n = case["block_size"], case["requests"]
    bm = BlockManager(5000, B)
    cache = PrefixCache(bm)
    prompt = list(range(case["prompt"]))
    for _ in range(n):
        _serve(bm, cache, prompt, case["suffix"])
    used = bm.num_blocks - bm.num_free()
    assert used == case["with"] == 4032
    assert round(case["without"] / used, 2) == case["reduction_2dp"]


def test_worked_example_2_under_whole_block_reuse():
    # 380-token prompt + 90 tokens, 500 requests: with whole-block reuse the
    # 12-token tail of the prompt is stored per request (23 + 7 * 500 blocks),
    # the page's 3,024 assumes the partial 24th block is shared as well
    case = GOLDEN["shared_prompt"][0]
    B = case["block_size"]
    bm = BlockManager(5000, B)
    cache = PrefixCache(bm)
    prompt = list(range(case["prompt"]))
    for _ in range(case["requests"]):
        _serve(bm, cache, prompt, case["suffix"])
    used = bm.num_blocks - bm.num_free()
    ref = bk.shared_prompt_blocks(case["prompt"], case["suffix"], B, case["requests"], share_partial=False)
    assert used == ref["with"] == 23 + 7 * 500


def test_lru_leaf_goes_first_and_running_requests_are_protected():
    bm = BlockManager(40, 4)
    cache = PrefixCache(bm)
    a = list(range(100, 112))      # 3 blocks
    b = list(range(200, 212))      # 3 blocks
    sa = _serve(bm, cache, a, 0)
    sb = _serve(bm, cache, b, 0)
    bm.free_seq(sa)
    cache.match(a)                 # a is now the more recently used prompt
    # b's blocks are still used by sequence sb: nothing of b can go
    assert cache.evict(1) == 1 and len(cache.match(a)) == 2 and len(cache.match(b)) == 3
    bm.free_seq(sb)
    # both prompts are now evictable; b was looked up after a, so a's tail is older
    assert cache.evict(1) == 1
    assert len(cache.match(a)) == 1 and len(cache.match(b)) == 3
    assert cache.evict(10) == 4 and cache.cached_blocks() == 0
    assert bm.num_free() == 40


def test_a_lookup_counts_as_a_use():
    # least recently *used*: a prompt looked up after another one was cached is the newer
    bm = BlockManager(20, 4)
    cache = PrefixCache(bm)
    a, b = list(range(100, 108)), list(range(200, 208))
    bm.free_seq(_serve(bm, cache, a, 0))
    bm.free_seq(_serve(bm, cache, b, 0))
    cache.match(a)
    assert cache.evict(1) == 1
    assert len(cache.match(a)) == 2 and len(cache.match(b)) == 1


def test_insert_refuses_free_and_repeated_blocks():
    # a cached block holds the K/V of one prefix, and only allocated blocks can be cached
    bm = BlockManager(8, 4)
    cache = PrefixCache(bm)
    s = bm.create()
    bm.append(s, 8)
    b0, b1 = bm.table(s)
    toks = list(range(8))
    free_block = next(b for b in range(8) if bm.refcount(b) == 0)
    with pytest.raises(IndexError):
        cache.insert(toks, [b0, free_block])
    with pytest.raises(ValueError):
        cache.insert(toks, [b0, b0])
    assert cache.cached_blocks() == 0 and (bm.refcount(b0), bm.refcount(b1)) == (1, 1)
    assert cache.insert(toks, [b0, b1]) == 2 and (bm.refcount(b0), bm.refcount(b1)) == (2, 2)


def test_a_sequence_started_from_a_prefix_holds_its_blocks():
    bm = BlockManager(8, 4)
    cache = PrefixCache(bm)
    s = bm.create()
    bm.append(s, 8)
    cache.insert(list(range(8)), bm.table(s))
    bm.free_seq(s)
    blocks = cache.match(list(range(10)))
    t = create_from_prefix(bm, blocks)
    assert bm.length(t) == 8 and [bm.refcount(b) for b in blocks] == [2, 2]
    assert cache.evict(2) == 0           # held by the new sequence
    bm.free_seq(t)
    assert [bm.refcount(b) for b in blocks] == [1, 1] and cache.evict(2) == 2
