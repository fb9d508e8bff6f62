"""Test-side helpers: an independent scatter into a paged pool and an unpaged
brute-force attention, used to pin the oracle and to build GPU parity inputs.

These restate the pages' rules in numpy on contiguous data:
token i of a sequence goes to offset i % B of physical block table[i // B]
("PagedAttention: Virtual Memory for the KV Cache", "A block table preserves
token order"), and unpaged attention is softmax(scale q K^T) V over the
contiguous rows, computed with scipy's softmax.
"""
from __future__ import annotations

import numpy as np
from scipy.special import softmax

from paged_kv_cache_127_gb300 import synth


def widen(a: np.ndarray, dtype: str) -> np.ndarray:
    """Storage array -> float64 (numpy's own conversions)."""
    with np.errstate(invalid="ignore"):
        if dtype == "bf16":
            return synth.bf16_bits_to_f32(a).astype(np.float64)
        return a.astype(np.float64)


def scatter(seq_rows, tables, block_size: int, num_blocks: int, dtype: str, fill=None):
    """Build a [N, Hkv, B, D] pool from contiguous per-sequence rows [len, Hkv, D].

    Slots that no sequence writes hold `fill` (default: NaN in the storage type).
    """
    first = next(r for r in seq_rows if r is not None)
    Hkv, D = first.shape[1], first.shape[2]
    fill = synth.nan_value(dtype) if fill is None else fill
    pool = np.full((num_blocks, Hkv, block_size, D), fill, dtype=synth.STORAGE[dtype])
    for s, rows in enumerate(seq_rows):
        for i in range(rows.shape[0]):
            pool[tables[s][i // block_size], :, i % block_size, :] = rows[i]
    return pool


def brute_attention(q64: np.ndarray, K64, V64, lens, scale: float) -> np.ndarray:
    """Unpaged attention: q [S, Hq, D]; K/V lists of contiguous [len, Hkv, D] float64."""
    S, Hq, D = q64.shape
    out = np.zeros((S, Hq, D))
    for s in range(S):
        n = int(lens[s])
        if n == 0:
            continue
        Hkv = K64[s].shape[1]
        G = Hq // Hkv
        for h in range(Hq):
            k = K64[s][:n, h // G, :]
            v = V64[s][:n, h // G, :]
            w = softmax(scale * (k @ q64[s, h]))
            out[s, h] = w @ v
    return out


def random_case(rng, dtype: str, S: int, Hq: int, Hkv: int, D: int, B: int, lens,
                extra_blocks: int = 3, std: float = 1.0):
    """Random contiguous K/V per sequence, scattered into a shuffled pool."""
    lens = np.asarray(lens, dtype=np.int32)
    nb = synth.blocks_needed(lens, B)
    N = int(nb.sum()) + extra_blocks
    tables, _ = synth.scattered_tables(rng, lens, B, N, shuffle=True,
                                       max_blocks=int(max(1, nb.max())) + 1)
    K = [synth.normal(rng, (int(n), Hkv, D), std, dtype) for n in lens]
    V = [synth.normal(rng, (int(n), Hkv, D), std, dtype) for n in lens]
    q = synth.normal(rng, (S, Hq, D), std, dtype)
    kc = scatter(K, tables, B, N, dtype)
    vc = scatter(V, tables, B, N, dtype)
    return q, K, V, kc, vc, tables, lens


def assert_attention_close(got, ref, atol=2e-3, rtol=1e-2, floor=0.05):
    """The decode tolerance: every |d| <= atol, and |d|/|ref| <= rtol where |ref| >= floor."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), "non-finite output"
    d = np.abs(got - ref)
    worst = float(d.max()) if d.size else 0.0
    assert worst <= atol, f"max abs error {worst:.3e} > {atol}"
    big = np.abs(ref) >= floor
    if big.any():
        rel = float((d[big] / np.abs(ref[big])).max())
        assert rel <= rtol, f"max rel error {rel:.3e} > {rtol}"
    return worst
