"""Pins for the oracle's chunk attention (several query tokens per sequence).

The n_s query tokens of a sequence are its last n_s positions; the query at
position pos sees keys 0..pos, the cache that one-token-at-a-time decoding
would hold at that point.  The pins: a closed form, an unpaged causal brute
force with scipy's softmax, the equality with n_s separate decodes, causality
(keys after a query's position cannot change it), and the reduction to decode
when every sequence has one query.
"""
import math

import numpy as np
import pytest
from scipy.special import softmax

import oracle
from paged_helpers import random_case, scatter, widen
from paged_kv_cache_127_gb300 import synth


def _chunk_case(rng, dtype, Hq, Hkv, D, B, lens, nq):
    q_unused, K, V, kc, vc, tables, lens = random_case(rng, dtype, len(lens), Hq, Hkv, D, B, lens)
    qs = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    q = synth.normal(rng, (int(qs[-1]), Hq, D), 1.0, dtype)
    return q, K, V, kc, vc, tables, lens, qs


def _brute_causal(q64, K64, V64, lens, qs, scale):
    """Unpaged: for each sequence, scores of its query rows against all its
    keys, future keys masked to -inf, scipy softmax along the keys."""
    T, Hq, D = q64.shape
    out = np.zeros((T, Hq, D))
    for s in range(len(lens)):
        n, L = int(qs[s + 1] - qs[s]), int(lens[s])
        if n == 0:
            continue
        G = Hq // K64[s].shape[1]
        allowed = np.arange(L)[None, :] <= (L - n + np.arange(n))[:, None]      # [n, L]
        for h in range(Hq):
            k, v = K64[s][:L, h // G, :], V64[s][:L, h // G, :]
            z = scale * (q64[qs[s]:qs[s + 1], h, :] @ k.T)
            z = np.where(allowed, z, -np.inf)
            out[qs[s]:qs[s + 1], h] = softmax(z, axis=1) @ v
    return out


def test_closed_form_first_query_sees_one_token():
    # two stored tokens, both queried: query 0 (position 0) sees only token 0 and
    # returns v0 exactly; query 1 sees both with keys 0 and ln 3 -> weights 1/4, 3/4
    k = np.array([0.0, math.log(3.0)], dtype=np.float32).reshape(2, 1, 1)
    v = np.array([1.0, 5.0], dtype=np.float32).reshape(2, 1, 1)
    tables = np.array([[2, 0]], np.int32)                       # B = 1, reversed placement
    kc = scatter([k], tables, 1, 3, "f32")
    vc = scatter([v], tables, 1, 3, "f32")
    q = np.ones((2, 1, 1), np.float32)
    out = oracle.chunk_attention(q, kc, vc, tables, np.array([2], np.int32), np.array([0, 2], np.int32), 1.0, "f32")
    assert out[0, 0, 0] == 1.0
    assert out[1, 0, 0] == pytest.approx(4.0, abs=1e-6)


@pytest.mark.parametrize("dtype", synth.DTYPES)
def test_matches_unpaged_causal_brute_force(dtype):
    rng = synth.make_rng(41)
    lens = [9, 1, 23, 16]
    nq = [3, 1, 23, 5]                 # a partial chunk, one token, the whole sequence, a block-aligned one
    q, K, V, kc, vc, tables, lens, qs = _chunk_case(rng, dtype, 4, 2, 16, 4, lens, nq)
    got = oracle.chunk_attention(q, kc, vc, tables, lens, qs, 0.3, dtype)
    ref = _brute_causal(widen(q, dtype), [widen(x, dtype) for x in K], [widen(x, dtype) for x in V], lens, qs, 0.3)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_equals_one_decode_per_query(dtype):
    # verifying n drafted tokens at once gives what n sequential decode steps give
    rng = synth.make_rng(42)
    lens, nq = [40, 17], [6, 17]
    q, K, V, kc, vc, tables, lens, qs = _chunk_case(rng, dtype, 8, 2, 32, 8, lens, nq)
    got = oracle.chunk_attention(q, kc, vc, tables, lens, qs, 1 / 8, dtype)
    for s in range(2):
        n = nq[s]
        for t in range(n):
            one = oracle.decode(q[qs[s] + t][None], kc, vc, tables[s:s + 1],
                                np.array([lens[s] - n + t + 1], np.int32), 1 / 8, dtype)
            np.testing.assert_allclose(got[qs[s] + t], one[0], rtol=1e-13, atol=1e-15)


def test_future_keys_cannot_change_a_query():
    rng = synth.make_rng(43)
    lens, nq = [30], [8]
    q, K, V, kc, vc, tables, lens, qs = _chunk_case(rng, "f16", 4, 4, 16, 8, lens, nq)
    base = oracle.chunk_attention(q, kc, vc, tables, lens, qs, 0.25, "f16")
    cut = 30 - 8 + 3                    # query 3's position: tokens after it are its future
    K2 = K[0].copy()
    V2 = V[0].copy()
    K2[cut + 1:] = synth.normal(rng, K2[cut + 1:].shape, 3.0, "f16")
    V2[cut + 1:] = synth.normal(rng, V2[cut + 1:].shape, 3.0, "f16")
    N = kc.shape[0]
    kc2 = scatter([K2], tables, 8, N, "f16")
    vc2 = scatter([V2], tables, 8, N, "f16")
    moved = oracle.chunk_attention(q, kc2, vc2, tables, lens, qs, 0.25, "f16")
    np.testing.assert_array_equal(moved[:4], base[:4])          # queries 0..3
    assert (np.abs(moved[4:] - base[4:]).max(axis=(1, 2)) > 1e-3).all()   # 4..7 see the change


@pytest.mark.parametrize("dtype", synth.DTYPES)
def test_one_query_per_sequence_is_decode(dtype):
    rng = synth.make_rng(44)
    lens = [5, 33, 64, 2]
    q, K, V, kc, vc, tables, lens = random_case(rng, dtype, 4, 8, 4, 16, 16, lens)
    qs = np.arange(5, dtype=np.int32)
    np.testing.assert_allclose(oracle.chunk_attention(q, kc, vc, tables, lens, qs, 0.2, dtype),
                               oracle.decode(q, kc, vc, tables, lens, 0.2, dtype), rtol=1e-14, atol=1e-15)


def test_rejects_inconsistent_query_ranges():
    rng = synth.make_rng(45)
    q, K, V, kc, vc, tables, lens, qs = _chunk_case(rng, "f32", 2, 1, 8, 4, [3, 5], [2, 2])
    with pytest.raises(ValueError):       # more queries than stored tokens
        oracle.chunk_attention(q, kc, vc, tables, lens, np.array([0, 4, 4], np.int32), 1.0, "f32")
    with pytest.raises(ValueError):       # ranges that do not end at T
        oracle.chunk_attention(q, kc, vc, tables, lens, np.array([0, 1, 3], np.int32), 1.0, "f32")
    with pytest.raises(ValueError):       # ranges that do not start at row 0
        oracle.chunk_attention(q, kc, vc, tables, lens, np.array([1, 2, 4], np.int32), 1.0, "f32")
