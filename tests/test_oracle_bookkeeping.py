"""The pages' block-count, fragmentation and sharing numbers (tests/golden/)."""
import json
import os
from fractions import Fraction

import pytest

from oracle import bookkeeping as bk

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    return json.load(open(os.path.join(GOLDEN, name)))


def _pct2(fr: Fraction) -> float:
    return round(float(fr) * 100, 2)


@pytest.mark.parametrize("case", _load("fragmentation.json")["cases"], ids=lambda c: c["citation"][:40])
def test_fragmentation_examples(case):
    r = bk.fragmentation(case["lengths"], case["block_size"], case["max_len"])
    assert r["blocks"] == case["blocks"]
    assert r["paged_slots"] == case["paged_slots"]
    assert r["paged_waste"] == case["paged_waste"]
    for key in ("total_blocks", "tokens", "naive_slots", "naive_waste"):
        if key in case:
            assert r[key] == case[key], key
    if "paged_frag_pct_2dp" in case:
        assert _pct2(r["paged_frag"]) == case["paged_frag_pct_2dp"]
    if "naive_frag_pct_2dp" in case:
        assert _pct2(r["naive_frag"]) == case["naive_frag_pct_2dp"]
    if "reduction_2dp" in case:
        assert round(float(r["reduction"]), 2) == case["reduction_2dp"]
    if "reduction_exact" in case:
        assert r["reduction"] == Fraction(*case["reduction_exact"])


@pytest.mark.parametrize("case", _load("sharing.json")["shared_prompt"], ids=lambda c: c["citation"][:40])
def test_shared_prompt_examples(case):
    r = bk.shared_prompt_blocks(case["prompt"], case["suffix"], case["block_size"],
                                case["requests"], case["share_partial"])
    assert r["per_request_unshared"] == case["per_request_unshared"]
    assert r["without"] == case["without"]
    assert r["with"] == case["with"]
    assert round(float(r["reduction"]), 2) == case["reduction_2dp"]


@pytest.mark.parametrize("case", _load("sharing.json")["full_blocks"], ids=lambda c: str(c["block_size"]))
def test_full_shareable_blocks(case):
    n = bk.full_shareable_blocks(case["prompt"], case["block_size"])
    assert n == case["full_blocks"]
    assert n * case["block_size"] == case["tokens"]


def test_table_entries_by_block_size():
    g = _load("sharing.json")["table_entries"]
    for B, entries in g["entries"].items():
        assert sum(bk.blocks_for(n, int(B)) for n in g["lengths"]) == entries


def test_kv_bytes_per_token():
    g = _load("block_tables.json")["kv_bytes_per_token"]
    assert bk.kv_bytes_per_token(g["layers"], g["heads"], g["head_dim"], g["dtype_bytes"]) == g["bytes"]


def test_waste_below_one_block_and_eta_bound():
    # waste < B slots per sequence; eta_paged >= 1 - (B - 1) / L for each sequence
    for B in (1, 2, 16, 32, 64):
        for L in range(1, 300):
            slots = bk.blocks_for(L, B) * B
            assert 0 <= slots - L < B
            assert bk.eta_paged([L], B) >= bk.eta_paged_lower_bound(L, B)


def test_block_count_refuses_negative_sizes():
    with pytest.raises(ValueError):
        bk.blocks_for(-1, 16)
    with pytest.raises(ValueError):
        bk.blocks_for(5, 0)
    assert bk.blocks_for(0, 16) == 0


def test_eta_bound_closed_forms():
    # one-slot blocks waste nothing: the bound is exactly 1
    for L in (1, 7, 300):
        assert bk.eta_paged_lower_bound(L, 1) == 1 == bk.eta_paged([L], 1)
    # a sequence one token into its last block wastes the full B - 1 slots, so
    # eta = L / (L + B - 1), and L / (L + B - 1) - (1 - (B - 1) / L) = (B - 1)^2 / (L (L + B - 1))
    for B in (2, 16, 64):
        for k in (0, 1, 5, 40):
            L = k * B + 1
            gap = bk.eta_paged([L], B) - bk.eta_paged_lower_bound(L, B)
            assert gap == Fraction((B - 1) ** 2, L * (L + B - 1))


def test_pool_slots_and_naive_reservation_do_not_fit():
    g = _load("block_tables.json")["pool"]
    assert g["num_blocks"] * g["block_size"] == g["pool_slots"]
    assert bk.fragmentation(g["lengths"], 16, 2048)["naive_slots"] > g["pool_slots"]
