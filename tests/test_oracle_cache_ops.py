"""Pins for the oracle's slot mapping, KV write and block copy."""
import json
import os

import numpy as np
import pytest

import oracle
from paged_helpers import scatter, widen
from paged_kv_cache_127_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_position_37_maps_to_block_9_offset_5():
    g = json.load(open(os.path.join(GOLDEN, "block_tables.json")))["translate"]
    slot = oracle.slot(g["table"], g["block_size"], g["position"])
    assert divmod(slot, g["block_size"]) == (g["physical_block"], g["offset"])


def test_slot_mapping_enumerates_every_slot_of_a_table_once():
    # walking positions 0..nB-1 through a table visits each slot of each listed block once,
    # in table order, offsets ascending
    B = 8
    table = np.array([[6, 1, 4, 0]], dtype=np.int32)
    pos = np.arange(4 * B, dtype=np.int32)
    slots = oracle.slot_mapping(table, B, np.zeros_like(pos), pos)
    expect = [b * B + o for b in table[0] for o in range(B)]
    assert slots.tolist() == expect
    neg = oracle.slot_mapping(table, B, np.zeros(2, np.int32), np.array([-1, 3], np.int32))
    assert neg.tolist() == [-1, 6 * B + 3]
    # a position past the table's last block, and a negative position asked of one
    # table row, are refused
    two = np.array([[6, 1, 4, 0], [2, 3, 5, 7]], dtype=np.int32)
    with pytest.raises(ValueError):
        oracle.slot_mapping(two, B, np.zeros(1, np.int32), np.array([4 * B], np.int32))
    with pytest.raises(ValueError):
        oracle.slot(table[0], B, -1)


@pytest.mark.parametrize("dtype", synth.DTYPES)
def test_written_rows_are_read_back_by_decode(dtype):
    # Write the rows of a sequence through its slots, then decode with q = 0: the
    # output must be the mean of exactly those value rows.
    rng = synth.make_rng(11)
    B, N, Hkv, D, n = 4, 9, 2, 8, 13
    table = np.array([[5, 8, 0, 2]], dtype=np.int32)
    K = synth.normal(rng, (n, Hkv, D), 1.0, dtype)
    V = synth.normal(rng, (n, Hkv, D), 1.0, dtype)
    kc = np.full((N, Hkv, B, D), synth.nan_value(dtype), synth.STORAGE[dtype])
    vc = kc.copy()
    slots = oracle.slot_mapping(table, B, np.zeros(n, np.int32), np.arange(n, dtype=np.int32))
    oracle.write_kv(K, V, slots, kc, vc, dtype)
    q = np.zeros((1, Hkv, D), synth.STORAGE[dtype])
    out = oracle.decode(q, kc, vc, table, np.array([n], np.int32), 1.0, dtype)
    np.testing.assert_allclose(out[0], widen(V, dtype).mean(axis=0), rtol=1e-13, atol=1e-15)
    # and the pool equals the independent scatter of the same rows
    np.testing.assert_array_equal(kc.view(np.uint8), scatter([K], table, B, N, dtype).view(np.uint8))


def test_negative_slots_are_skipped_and_others_untouched():
    rng = synth.make_rng(12)
    B, N, Hkv, D = 16, 6, 2, 8
    kc = synth.normal(rng, (N, Hkv, B, D), 1.0, "bf16")
    vc = synth.normal(rng, (N, Hkv, B, D), 1.0, "bf16")
    k0, v0 = kc.copy(), vc.copy()
    k = synth.normal(rng, (3, Hkv, D), 1.0, "bf16")
    v = synth.normal(rng, (3, Hkv, D), 1.0, "bf16")
    oracle.write_kv(k, v, np.array([-1, 17, -5]), kc, vc, "bf16")
    changed = np.argwhere((kc != k0).any(axis=-1))
    assert {tuple(c) for c in changed} <= {(1, 0, 1), (1, 1, 1)}
    np.testing.assert_array_equal(kc[1, :, 1, :], k[1])
    np.testing.assert_array_equal(vc[1, :, 1, :], v[1])
    mask = np.ones(kc.shape[:3], bool)
    mask[1, :, 1] = False
    np.testing.assert_array_equal(kc[mask], k0[mask])
    np.testing.assert_array_equal(vc[mask], v0[mask])
    with pytest.raises(ValueError):
        oracle.write_kv(k[:1], v[:1], np.array([N * B]), kc, vc, "bf16")


@pytest.mark.parametrize("dtype", synth.DTYPES)
def test_copy_blocks_copies_whole_blocks_only(dtype):
    rng = synth.make_rng(13)
    N, Hkv, B, D = 12, 2, 16, 8
    kc = synth.normal(rng, (N, Hkv, B, D), 1.0, dtype)
    vc = synth.normal(rng, (N, Hkv, B, D), 1.0, dtype)
    k0, v0 = kc.copy(), vc.copy()
    pairs = np.array([[3, 7], [3, 9], [0, 11]])
    oracle.copy_blocks(kc, vc, pairs, dtype)
    for src, dst in pairs:
        assert kc[dst].tobytes() == k0[src].tobytes()
        assert vc[dst].tobytes() == v0[src].tobytes()
    others = [b for b in range(N) if b not in (7, 9, 11)]
    assert kc[others].tobytes() == k0[others].tobytes()
    assert vc[others].tobytes() == v0[others].tobytes()
    for bad in ([0, N], [N, 0], [-1, 0], [0, -1]):
        with pytest.raises(ValueError):
            oracle.copy_blocks(kc, vc, np.array([bad]), dtype)


@pytest.mark.parametrize("dtype", synth.DTYPES)
def test_swap_blocks_moves_whole_blocks_between_pools(dtype):
    rng = synth.make_rng(14)
    Hkv, B, D = 2, 16, 8
    dev_k = synth.normal(rng, (10, Hkv, B, D), 1.0, dtype)
    dev_v = synth.normal(rng, (10, Hkv, B, D), 1.0, dtype)
    host_k = np.zeros((6, Hkv, B, D), synth.STORAGE[dtype])
    host_v = np.zeros((6, Hkv, B, D), synth.STORAGE[dtype])
    pairs = np.array([[7, 0], [2, 5], [9, 3]])
    oracle.swap_blocks(dev_k, dev_v, host_k, host_v, pairs, dtype)
    for src, dst in pairs:
        assert host_k[dst].tobytes() == dev_k[src].tobytes()
        assert host_v[dst].tobytes() == dev_v[src].tobytes()
    assert not host_k[[1, 2, 4]].view(np.uint8).any()        # untouched host blocks
    back_k, back_v = np.zeros_like(dev_k), np.zeros_like(dev_v)
    oracle.swap_blocks(host_k, host_v, back_k, back_v, pairs[:, ::-1], dtype)
    for src, dst in pairs:
        assert back_k[src].tobytes() == dev_k[src].tobytes()
    with pytest.raises(ValueError):
        oracle.swap_blocks(dev_k, dev_v, host_k, host_v, np.array([[0, 6]]), dtype)
