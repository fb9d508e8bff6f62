"""The seeded input generators produce the workloads their recipes state.

These check the shapes, ranges and distributions of the synthetic inputs (the
stand-ins for the pages' workloads), and the bfloat16 rounding of the input
helper against PyTorch's own conversion.  No attention arithmetic is involved.
"""
import math

import numpy as np
import pytest

from paged_kv_cache_127_gb300 import synth

# name: (dtype, Hq, Hkv, D, B, S)
SHAPES = {
    "tiny": ("f32", 4, 4, 64, 16, 3),
    "mha7b": ("f16", 32, 32, 128, 16, 64),
    "gqa8b_b16": ("bf16", 32, 8, 128, 16, 256),
    "gqa8b_b32": ("bf16", 32, 8, 128, 32, 256),
    "prefix_cow": ("bf16", 32, 8, 128, 16, 192),
    "long70b": ("bf16", 64, 8, 128, 16, 32),
    "verify8b": ("bf16", 32, 8, 128, 16, 256),
    "prefill8b": ("bf16", 32, 8, 128, 16, 16),
}


@pytest.mark.parametrize("name", list(SHAPES))
def test_workload_shapes(name):
    w = synth.workload(name, 0)
    assert (w.dtype, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, w.num_seqs) == SHAPES[name]
    assert w.num_q_heads % w.num_kv_heads == 0
    # the same seed gives the same workload; another seed another one
    np.testing.assert_array_equal(synth.workload(name, 0).lengths, w.lengths)
    if name != "tiny":
        assert not np.array_equal(synth.workload(name, 1).lengths, w.lengths)


def test_length_ranges():
    assert synth.workload("tiny").lengths.tolist() == [25, 47, 12]
    m = synth.workload("mha7b").lengths
    assert m.min() >= 1 and m.max() <= 2048
    for name in ("gqa8b_b16", "gqa8b_b32"):
        g = synth.workload(name).lengths
        assert g.min() >= 1 and g.max() <= 4096
        # the lognormal tail reaches past 2048 (P ~ 6 % a sequence): the clip is at 4096, not lower
        assert (g > 2048).sum() >= 5
    p = synth.workload("prefix_cow")
    assert p.lengths.shape == (128,) and p.lengths.min() >= 1 and p.lengths.max() <= 512
    assert (p.prefix_len, p.prefix_group, p.pair_count, p.pair_prefix) == (800, 128, 32, 24)
    lg = synth.workload("long70b").lengths
    assert lg.min() >= 8192 and lg.max() <= 32768
    v = synth.workload("verify8b")
    assert v.query_len == 5 and v.lengths.min() >= 6 and v.lengths.max() <= 4096
    f = synth.workload("prefill8b")
    assert f.query_len == 512 and f.lengths.min() >= 512 and f.lengths.max() <= 4096


def test_lognormal_lengths_have_the_stated_median_and_spread():
    # round(600 exp(0.8 Z)) clipped to [1, 4096]: median 600; the quartiles (untouched
    # by the clip) are 600 exp(-+0.8 z75), z75 = 0.6745 the normal's upper quartile
    x = synth.lognormal_lengths(synth.make_rng(3), 200_000, 600, 0.8, 1, 4096)
    assert abs(np.median(x) - 600) <= 6
    q1, q3 = np.percentile(x, [25, 75])
    assert abs(math.log(q3 / q1) - 2 * 0.6745 * 0.8) < 0.02
    # P(600 exp(0.8 Z) > 4096) = P(Z > ln(4096 / 600) / 0.8)
    p = 0.5 * math.erfc(math.log(4096 / 600) / 0.8 / math.sqrt(2))
    assert abs((x == 4096).mean() - p) < 0.002


def test_uniform_lengths_cover_their_range():
    x = synth.uniform_lengths(synth.make_rng(4), 100_000, 8192, 32768)
    assert x.min() == 8192 and x.max() == 32768
    assert abs(x.mean() - (8192 + 32768) / 2) < 100


def test_normal_values_have_the_stated_spread():
    for dtype in synth.DTYPES:
        x = synth.storage_to_f32(synth.normal(synth.make_rng(5), (400, 256), 0.5, dtype), dtype)
        assert abs(x.mean()) < 0.01 and abs(x.std() - 0.5) < 0.01


def test_pool_and_placement():
    rng = synth.make_rng(6)
    lens = synth.uniform_lengths(rng, 64, 1, 2048)
    demand = int(synth.blocks_needed(lens, 16).sum())
    N = synth.pool_blocks(lens, 16, 1.25)
    assert N == math.ceil(1.25 * demand)
    tables, used = synth.scattered_tables(rng, lens, 16, N)
    nb = synth.blocks_needed(lens, 16)
    ids = np.concatenate([tables[s, :n] for s, n in enumerate(nb)])
    assert len(ids) == demand and len(np.unique(ids)) == demand       # every block at most once
    assert ids.min() >= 0 and ids.max() < N
    assert all((tables[s, n:] == -1).all() for s, n in enumerate(nb))
    assert used.sum() == demand and used[ids].all()
    # a seeded permutation of the pool, not the blocks in order: another seed places
    # them differently, and consecutive table entries are rarely consecutive ids
    steps = np.concatenate([np.diff(tables[s_, :n]) for s_, n in enumerate(nb)])
    assert np.mean(steps == 1) < 0.05
    other, _ = synth.scattered_tables(synth.make_rng(60), lens, 16, N)
    assert not np.array_equal(other, tables)
    ordered, _ = synth.scattered_tables(rng, lens, 16, N, shuffle=False)
    assert ordered[0, :nb[0]].tolist() == list(range(nb[0]))
    with pytest.raises(ValueError):
        synth.scattered_tables(rng, lens, 16, demand - 1)


def test_slots_and_copy_pairs():
    rng = synth.make_rng(7)
    s = synth.distinct_slots(rng, 500, 4096, frac_skip=0.1)
    kept = s[s >= 0]
    assert len(np.unique(kept)) == len(kept) and kept.max() < 4096 and 0 < (s < 0).sum() < 100
    pairs = synth.copy_pairs(rng, 32, 100)
    assert len(set(pairs[:, 1])) == 32 and not set(pairs[:, 0]) & set(pairs[:, 1])
    with pytest.raises(ValueError):
        synth.copy_pairs(rng, 51, 100)


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = synth.make_rng(8)
    x = np.concatenate([
        rng.standard_normal(100_000).astype(np.float32) * np.float32(3.0),
        np.array([0.0, -0.0, 1.0, 65504.0, 3.0e38, -3.0e38, 1e-40, -1e-40, np.inf, -np.inf], np.float32),
        # halfway cases: the bits just above, at and below a bfloat16 rounding boundary
        (np.array([0x3F808000, 0x3F818000, 0x3F807FFF, 0x3F808001], np.uint32)).view(np.float32),
    ])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(synth.f32_to_bf16_bits(x), want)
    nan = synth.f32_to_bf16_bits(np.array([np.nan], np.float32))
    assert np.isnan(synth.bf16_bits_to_f32(nan)).all()
    np.testing.assert_array_equal(synth.bf16_bits_to_f32(want), torch.from_numpy(want.view(np.int16)).view(
        torch.bfloat16).float().numpy())
