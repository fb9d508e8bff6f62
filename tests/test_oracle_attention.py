"""Pins for the fp64 decode oracle, against things other than itself.

Each test fixes the oracle to a closed form, an invariant the pages state, a
library routine, or an unpaged brute force on tiny inputs, chosen so that a
dropped term, a wrong sign, index or offset, or a swapped operand fails at
least one of them.
"""
import math
import zlib

import numpy as np
import pytest

import oracle
from paged_helpers import brute_attention, random_case, scatter, widen
from paged_kv_cache_127_gb300 import synth


def _one_seq(dtype, K, V, q, table, B, N, scale, fill=0):
    """Decode one sequence of contiguous rows K/V [len, Hkv, D] placed via `table`."""
    tables = np.array([table], dtype=np.int32)
    kc = scatter([K], tables, B, N, dtype, fill=fill)
    vc = scatter([V], tables, B, N, dtype, fill=fill)
    return oracle.decode(q, kc, vc, tables, np.array([K.shape[0]], np.int32), scale, dtype)


def test_closed_form_two_tokens_weights_one_to_three():
    # q = 1, keys 0 and ln 3 -> softmax weights 1/4, 3/4; values 1 and 5 -> output 4.
    # The two tokens sit in different physical blocks (B = 1), in reverse order.
    k = np.array([0.0, math.log(3.0)], dtype=np.float32).reshape(2, 1, 1)
    v = np.array([1.0, 5.0], dtype=np.float32).reshape(2, 1, 1)
    q = np.ones((1, 1, 1), dtype=np.float32)
    out = _one_seq("f32", k, v, q, [3, 1], 1, 4, 1.0)
    w1 = math.exp(float(np.float32(math.log(3.0))))
    assert out[0, 0, 0] == pytest.approx((1.0 + 5.0 * w1) / (1.0 + w1), rel=1e-15)
    assert out[0, 0, 0] == pytest.approx(4.0, abs=1e-6)
    # the scale multiplies the logits: scale 2 gives weights 1 : 9 -> (1 + 45) / 10
    out2 = _one_seq("f32", k, v, q, [3, 1], 1, 4, 2.0)
    assert out2[0, 0, 0] == pytest.approx(4.6, abs=1e-6)


def test_single_token_returns_its_value_exactly():
    rng = synth.make_rng(1)
    for dtype in synth.DTYPES:
        K = synth.normal(rng, (1, 2, 16), 1.0, dtype)
        V = synth.normal(rng, (1, 2, 16), 1.0, dtype)
        q = synth.normal(rng, (1, 4, 16), 1.0, dtype)
        out = _one_seq(dtype, K, V, q, [2], 4, 3, 0.25, fill=synth.nan_value(dtype))
        ref = widen(V, dtype)[0]
        # G = 2: query heads 0, 1 read KV head 0; heads 2, 3 read KV head 1
        np.testing.assert_array_equal(out[0, :2], np.stack([ref[0], ref[0]]))
        np.testing.assert_array_equal(out[0, 2:], np.stack([ref[1], ref[1]]))


@pytest.mark.parametrize("dtype", synth.DTYPES)
def test_zero_query_gives_mean_of_values(dtype):
    rng = synth.make_rng(2)
    n, B = 37, 8
    K = synth.normal(rng, (n, 1, 8), 1.0, dtype)
    V = synth.normal(rng, (n, 1, 8), 1.0, dtype)
    q = np.zeros((1, 1, 8), dtype=synth.STORAGE[dtype])
    table = list(rng.permutation(10)[:5])
    out = _one_seq(dtype, K, V, q, table, B, 10, 0.3, fill=synth.nan_value(dtype))
    np.testing.assert_allclose(out[0, 0], widen(V, dtype)[:, 0, :].mean(axis=0), rtol=1e-13, atol=1e-15)


def test_spike_key_selects_every_position():
    # For each position j, make k_j a large multiple of q: the output must be v_j.
    rng = synth.make_rng(3)
    n, B, D = 21, 4, 8
    q = rng.standard_normal((1, 1, D)).astype(np.float32)
    table = [7, 2, 5, 0, 3, 6]
    V = rng.standard_normal((n, 1, D)).astype(np.float32)
    for j in range(n):
        K = (0.01 * rng.standard_normal((n, 1, D))).astype(np.float32)
        K[j, 0] = 60.0 * q[0, 0] / float(q[0, 0] @ q[0, 0])
        out = _one_seq("f32", K, V, q, table, B, 8, 1.0)
        np.testing.assert_allclose(out[0, 0], V[j, 0].astype(np.float64), atol=1e-20, rtol=1e-12)


@pytest.mark.parametrize("j", range(10))
def test_large_logits_do_not_overflow(j):
    # scores near 1e4 overflow exp() unless the maximum over *all* logits is
    # subtracted first; the largest logit is placed at every position in turn
    rng = synth.make_rng(4)
    n, D = 10, 4
    q = rng.standard_normal((1, 1, D)).astype(np.float32)
    K = (0.1 * rng.standard_normal((n, 1, D))).astype(np.float32)
    K[j, 0] = q[0, 0] / float(q[0, 0] @ q[0, 0])
    V = rng.standard_normal((n, 1, D)).astype(np.float32)
    out = _one_seq("f32", K, V, q, [1, 0, 2], 4, 3, 5000.0)
    assert np.isfinite(out).all()
    np.testing.assert_allclose(out[0, 0], V[j, 0], rtol=1e-9, atol=1e-12)


@pytest.mark.parametrize("dtype", synth.DTYPES)
@pytest.mark.parametrize("G,B,D", [(1, 1, 8), (2, 4, 16), (4, 16, 64), (8, 16, 32), (1, 32, 64)])
def test_matches_unpaged_brute_force(dtype, G, B, D):
    rng = synth.make_rng(zlib.crc32(repr((dtype, G, B, D)).encode()))
    S, Hkv = 5, 2
    lens = [1, B, B + 1, 3 * B - 1, 41]
    q, K, V, kc, vc, tables, lens = random_case(rng, dtype, S, G * Hkv, Hkv, D, B, lens)
    scale = 1.0 / math.sqrt(D)
    got = oracle.decode(q, kc, vc, tables, lens, scale, dtype)
    ref = brute_attention(widen(q, dtype), [widen(k, dtype) for k in K],
                          [widen(v, dtype) for v in V], lens, scale)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_physical_placement_does_not_change_output():
    rng = synth.make_rng(5)
    dtype, B, Hkv, D, G = "bf16", 16, 2, 64, 2
    lens = np.array([70, 16, 3, 129], dtype=np.int32)
    K = [synth.normal(rng, (n, Hkv, D), 1.0, dtype) for n in lens]
    V = [synth.normal(rng, (n, Hkv, D), 1.0, dtype) for n in lens]
    q = synth.normal(rng, (4, G * Hkv, D), 1.0, dtype)
    outs = []
    for trial in range(3):
        N = 40
        tables, _ = synth.scattered_tables(synth.make_rng(100 + trial), lens, B, N)
        kc = scatter(K, tables, B, N, dtype)
        vc = scatter(V, tables, B, N, dtype)
        outs.append(oracle.decode(q, kc, vc, tables, lens, 0.125, dtype))
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], outs[2])


def test_poisoned_padding_and_free_blocks_are_never_read():
    rng = synth.make_rng(6)
    dtype = "f16"
    q, K, V, kc, vc, tables, lens = random_case(rng, dtype, 3, 4, 4, 32, 16, [5, 33, 16],
                                                extra_blocks=6)
    poisoned = oracle.decode(q, kc, vc, tables, lens, 0.2, dtype)   # NaN everywhere unused
    kz = scatter(K, tables, 16, kc.shape[0], dtype, fill=np.float16(0))
    vz = scatter(V, tables, 16, kc.shape[0], dtype, fill=np.float16(0))
    clean = oracle.decode(q, kz, vz, tables, lens, 0.2, dtype)
    assert np.isfinite(poisoned).all()
    np.testing.assert_array_equal(poisoned, clean)


def test_grouped_heads_equal_replicated_multi_head():
    # GQA stores fewer KV heads (first page, "A block table preserves token order");
    # query head h reads KV head h // G.  Replicating each KV head G times must give
    # the same output as plain multi-head attention.
    rng = synth.make_rng(7)
    dtype, G, Hkv, D, B = "f32", 4, 2, 16, 4
    q, K, V, kc, vc, tables, lens = random_case(rng, dtype, 3, G * Hkv, Hkv, D, B, [9, 1, 17])
    gqa = oracle.decode(q, kc, vc, tables, lens, 0.5, dtype)
    kr = np.repeat(kc, G, axis=1)
    vr = np.repeat(vc, G, axis=1)
    mha = oracle.decode(q, kr, vr, tables, lens, 0.5, dtype)
    np.testing.assert_array_equal(gqa, mha)


@pytest.mark.parametrize("psize", [1, 3, 16, 64, 512, 10**6])
def test_partitioned_merge_equals_plain_softmax(psize):
    # Merging per-partition (m_b, l_b, acc_b) with the log-sum-exp weights is exact:
    # "Paged Attention and vLLM", "Paged Attention CUDA Kernel", merge equation.
    rng = synth.make_rng(8)
    dtype = "bf16"
    q, K, V, kc, vc, tables, lens = random_case(rng, dtype, 4, 8, 2, 64, 16, [1, 200, 513, 77])
    plain = oracle.decode(q, kc, vc, tables, lens, 0.125, dtype)
    part = oracle.decode_partitioned(q, kc, vc, tables, lens, 0.125, dtype, psize)
    np.testing.assert_allclose(part, plain, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("psize", [4, 16])
def test_partitioned_merge_with_extreme_partition_maxima(psize):
    # The merge weights e^(m_b - m*) stay finite only when m* is the largest m_b and
    # every m_b is its own partition's maximum.  Two cases, each against the plain
    # softmax: every logit near -1000 (a partition maximum started at 0 rather than
    # -inf underflows every weight to 0), and a +1000 spike in the first partition
    # only (an m* taken from another partition overflows).
    rng = synth.make_rng(81)
    n, D, B = 40, 8, 4
    q = np.zeros((1, 1, D), np.float32)
    q[0, 0, 0] = 1.0
    V = rng.standard_normal((n, 1, D)).astype(np.float32)
    tables = np.array([[3, 0, 7, 5, 9, 1, 2, 6, 8, 4]], np.int32)
    lens = np.array([n], np.int32)
    for spike in (False, True):
        K = (0.25 * rng.standard_normal((n, 1, D))).astype(np.float32)
        if spike:
            K[1, 0, 0] = 1000.0
        else:
            K[:, 0, 0] -= np.float32(1000.0)
        kc = scatter([K], tables, B, 10, "f32", fill=0)
        vc = scatter([V], tables, B, 10, "f32", fill=0)
        plain = oracle.decode(q, kc, vc, tables, lens, 1.0, "f32")
        part = oracle.decode_partitioned(q, kc, vc, tables, lens, 1.0, "f32", psize)
        assert np.isfinite(plain).all() and np.isfinite(part).all()
        np.testing.assert_allclose(part, plain, rtol=1e-9, atol=1e-12)
        if spike:
            np.testing.assert_allclose(plain[0, 0], V[1, 0], rtol=1e-9, atol=1e-12)


def test_empty_context_gives_zeros():
    rng = synth.make_rng(9)
    q, K, V, kc, vc, tables, lens = random_case(rng, "f32", 2, 2, 2, 8, 4, [3, 5])
    lens = np.array([0, 5], dtype=np.int32)
    out = oracle.decode(q, kc, vc, tables, lens, 1.0, "f32")
    np.testing.assert_array_equal(out[0], 0.0)
    assert np.isfinite(out).all()


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_widening_of_every_16_bit_pattern(dtype):
    # One token, q = 0 and K = 0: the output is exactly V, so the oracle's own
    # f16/bf16 -> double conversion is compared with numpy's for all 65536 codes.
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    V = (bits.view(np.float16) if dtype == "f16" else bits).reshape(1, 1, 65536)
    K = np.zeros_like(V)
    q = np.zeros((1, 1, 65536), dtype=V.dtype)
    out = _one_seq(dtype, K, V, q, [0], 1, 1, 1.0)[0, 0]
    np.testing.assert_array_equal(out, widen(V[0, 0], dtype))


def test_context_longer_than_table_is_rejected():
    q = np.zeros((1, 1, 4), np.float32)
    kc = np.zeros((2, 1, 4, 4), np.float32)
    with pytest.raises(ValueError):
        oracle.decode(q, kc, kc, np.array([[0]], np.int32), np.array([5], np.int32), 1.0, "f32")


def test_query_heads_must_be_a_multiple_of_kv_heads():
    q = np.zeros((1, 3, 4), np.float32)
    kc = np.zeros((2, 2, 4, 4), np.float32)
    with pytest.raises(ValueError):
        oracle.decode(q, kc, kc, np.array([[0]], np.int32), np.array([2], np.int32), 1.0, "f32")
