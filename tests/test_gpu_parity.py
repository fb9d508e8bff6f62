"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Bit-exact for the KV write, the block copy and the allocator's tables / slots /
pairs; for attention, every output element within |d| <= 2e-3, and within a
relative 1e-2 where |ref| >= 0.05 (fp32 accumulation of fp16 / bf16 data).
"""
import math

import numpy as np
import pytest

import oracle
from gpu_helpers import poison_unused, require_gpu, run_decode, to_dev, to_host
from oracle.block_manager import BlockManager
from paged_helpers import assert_attention_close, random_case, scatter
from paged_kv_cache_127_gb300 import synth, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gpu():
    return require_gpu()


def _check_no_device_errors(pa):
    assert pa.pa_device_errors(clear=True) == 0


# ----------------------------------------------------------------- decode, small shapes
SHAPES = [(D, B, G) for D in (64, 128) for B in (16, 32) for G in (1, 2, 4, 8)]


@pytest.mark.parametrize("dtype", synth.DTYPES)
@pytest.mark.parametrize("D,B,G", SHAPES)
def test_decode_small_shapes(gpu, dtype, D, B, G):
    torch, pa = gpu
    rng = synth.make_rng(1000 + D + B + G * 7 + synth.DTYPES.index(dtype) * 131)
    Hkv = 2
    # ragged lengths: single token, exact block, block + 1, several partitions + tail
    lens = [1, B, B + 1, 3 * B + 5, 200, 530, 0]
    q, K, V, kc, vc, tables, lens = random_case(rng, dtype, len(lens), G * Hkv, Hkv, D, B, lens)
    scale = 1.0 / math.sqrt(D)
    ref = oracle.decode(q, kc, vc, tables, lens, scale, dtype)
    for psize in (0, B, 4 * B):   # the automatic size (128 tokens at this batch), and split-K
        got = run_decode(torch, pa, dtype, q, kc, vc, tables, lens, scale, psize)
        assert_attention_close(got, ref)
        if dtype == "f32":
            assert np.abs(got - ref).max() < 1e-4
        np.testing.assert_array_equal(got[lens == 0], 0.0)
    _check_no_device_errors(pa)


def test_decode_tiny_worked_tables(gpu):
    # three sequences of 25/47/12 tokens in blocks [3, 7], [0, 5, 9], [4] of a 64-block pool
    torch, pa = gpu
    w = synth.workload("tiny")
    rng = synth.make_rng(5)
    tables = np.full((3, 4), -1, np.int32)
    for s, t in enumerate(w.fixed_tables):
        tables[s, :len(t)] = t
    kc = synth.normal(rng, (64, 4, 16, 64), 1.0, "f32")
    vc = synth.normal(rng, (64, 4, 16, 64), 1.0, "f32")
    poison_unused(kc, vc, tables, w.lengths, 16, "f32")
    q = synth.normal(rng, (3, 4, 64), 1.0, "f32")
    ref = oracle.decode(q, kc, vc, tables, w.lengths, w.scale, "f32")
    got = run_decode(torch, pa, "f32", q, kc, vc, tables, w.lengths, w.scale)
    assert np.abs(got - ref).max() < 1e-5
    _check_no_device_errors(pa)


def test_decode_placement_and_poison_invariance(gpu):
    torch, pa = gpu
    dtype, B, Hkv, D, G = "bf16", 16, 2, 128, 4
    rng = synth.make_rng(17)
    lens = np.array([700, 16, 3, 1029, 511], dtype=np.int32)
    K = [synth.normal(rng, (n, Hkv, D), 1.0, dtype) for n in lens]
    V = [synth.normal(rng, (n, Hkv, D), 1.0, dtype) for n in lens]
    q = synth.normal(rng, (5, G * Hkv, D), 0.1, dtype)
    outs = []
    for trial, fill in ((0, None), (1, None), (1, np.uint16(0))):
        N = 220
        tables, _ = synth.scattered_tables(synth.make_rng(300 + trial), lens, B, N)
        kc = scatter(K, tables, B, N, dtype, fill=fill)
        vc = scatter(V, tables, B, N, dtype, fill=fill)
        outs.append(run_decode(torch, pa, dtype, q, kc, vc, tables, lens, 1.0, 128))
    assert np.isfinite(outs[0]).all()
    np.testing.assert_array_equal(outs[0], outs[1])   # another placement: same bits
    np.testing.assert_array_equal(outs[1], outs[2])   # NaN vs zero in unused slots: same bits
    _check_no_device_errors(pa)


def test_decode_spike_selects_token(gpu):
    torch, pa = gpu
    dtype, B, D = "f16", 16, 128
    rng = synth.make_rng(23)
    n = 77
    base_q = rng.standard_normal(D).astype(np.float32)
    for j in (0, 15, 16, 40, 76):
        K = (0.01 * rng.standard_normal((n, 1, D))).astype(np.float16)
        K[j, 0] = (8.0 * base_q / np.linalg.norm(base_q)).astype(np.float16)
        V = synth.normal(rng, (n, 1, D), 1.0, dtype)
        q = (8.0 * base_q / np.linalg.norm(base_q)).astype(np.float16).reshape(1, 1, D)
        tables = np.array([[6, 2, 9, 0, 4]], np.int32)
        kc = scatter([K], tables, B, 10, dtype)
        vc = scatter([V], tables, B, 10, dtype)
        got = run_decode(torch, pa, dtype, q, kc, vc, tables, np.array([n], np.int32), 1.0, 32)
        ref = oracle.decode(q, kc, vc, tables, np.array([n], np.int32), 1.0, dtype)
        assert_attention_close(got, ref)
        np.testing.assert_allclose(got[0, 0], V[j, 0].astype(np.float64), atol=2e-3)


# ----------------------------------------------------------------- companion kernels
@pytest.mark.parametrize("dtype", synth.DTYPES)
@pytest.mark.parametrize("D,B", [(64, 16), (128, 16), (128, 32)])
def test_write_kv_bit_exact(gpu, dtype, D, B):
    torch, pa = gpu
    rng = synth.make_rng(31 + D + B)
    N, Hkv, T = 50, 8, 300
    kc = synth.normal(rng, (N, Hkv, B, D), 1.0, dtype)
    vc = synth.normal(rng, (N, Hkv, B, D), 1.0, dtype)
    k = synth.normal(rng, (T, Hkv, D), 1.0, dtype)
    v = synth.normal(rng, (T, Hkv, D), 1.0, dtype)
    slots = synth.distinct_slots(rng, T, N * B, frac_skip=0.1)
    dims = pa.make_dims(0, Hkv, Hkv, D, B, N, 1, 0, dtype)
    dkc, dvc = to_dev(torch, kc, dtype), to_dev(torch, vc, dtype)
    pa.pa_write_kv(dims, to_dev(torch, k, dtype), to_dev(torch, v, dtype),
                   torch.from_numpy(slots).cuda(), dkc, dvc)
    oracle.write_kv(k, v, slots, kc, vc, dtype)
    assert to_host(dkc, dtype).tobytes() == kc.tobytes()
    assert to_host(dvc, dtype).tobytes() == vc.tobytes()
    _check_no_device_errors(pa)


@pytest.mark.parametrize("dtype", synth.DTYPES)
def test_copy_blocks_bit_exact(gpu, dtype):
    torch, pa = gpu
    rng = synth.make_rng(41)
    N, Hkv, B, D = 96, 8, 16, 128
    kc = synth.normal(rng, (N, Hkv, B, D), 1.0, dtype)
    vc = synth.normal(rng, (N, Hkv, B, D), 1.0, dtype)
    pairs = synth.copy_pairs(rng, 32, N)
    dims = pa.make_dims(0, Hkv, Hkv, D, B, N, 1, 0, dtype)
    dkc, dvc = to_dev(torch, kc, dtype), to_dev(torch, vc, dtype)
    pa.pa_copy_blocks(dims, dkc, dvc, torch.from_numpy(pairs).cuda())
    oracle.copy_blocks(kc, vc, pairs, dtype)
    assert to_host(dkc, dtype).tobytes() == kc.tobytes()
    assert to_host(dvc, dtype).tobytes() == vc.tobytes()
    _check_no_device_errors(pa)


def test_bad_indices_are_flagged_not_faulted(gpu):
    # every bad index here is caught by the kernels' own range checks
    torch, pa = gpu
    dtype, N, Hkv, B, D = "bf16", 8, 2, 16, 64
    rng = synth.make_rng(51)
    kc = synth.normal(rng, (N, Hkv, B, D), 1.0, dtype)
    vc = synth.normal(rng, (N, Hkv, B, D), 1.0, dtype)
    dkc, dvc = to_dev(torch, kc, dtype), to_dev(torch, vc, dtype)
    dims = pa.make_dims(0, Hkv, Hkv, D, B, N, 1, 0, dtype)
    k = to_dev(torch, synth.normal(rng, (2, Hkv, D), 1.0, dtype), dtype)
    pa.pa_write_kv(dims, k, k, torch.tensor([N * B, 3], dtype=torch.int64, device="cuda"), dkc, dvc)
    assert pa.pa_device_errors(clear=True) == pa.PA_DEVERR_BAD_SLOT
    pa.pa_copy_blocks(dims, dkc, dvc, torch.tensor([[0, N]], dtype=torch.int64, device="cuda"))
    assert pa.pa_device_errors(clear=True) == pa.PA_DEVERR_BAD_PAIR
    # decode: one table entry out of range, one context longer than its table
    q = synth.normal(rng, (2, 2 * Hkv, D), 1.0, dtype)
    tables = np.array([[1, N + 5, 2], [3, 4, 5]], np.int32)
    lens = np.array([40, 10_000], np.int32)
    got = run_decode(torch, pa, dtype, q, kc, vc, tables, lens, 0.125)
    flags = pa.pa_device_errors(clear=True)
    assert flags == pa.PA_DEVERR_BAD_BLOCK | pa.PA_DEVERR_BAD_LEN
    # Sequence 0 loses block N+5 (tokens 16..31) and keeps tokens 0..15 of block 1
    # and 32..39 of block 2.  Decode has no positional term, so that equals
    # attention over table [1, 2] with 24 tokens.  Sequence 1 is clamped to its
    # 48-token table.
    ref0 = oracle.decode(q[:1], kc, vc, np.array([[1, 2]], np.int32), np.array([24], np.int32), 0.125, dtype)
    ref1 = oracle.decode(q[1:], kc, vc, tables[1:], np.array([48], np.int32), 0.125, dtype)
    assert_attention_close(got[:1], ref0)
    assert_attention_close(got[1:], ref1)


# ----------------------------------------------------------------- full-size workloads
@pytest.mark.parametrize("dtype", synth.DTYPES)
@pytest.mark.parametrize("B", [16, 32])
def test_decode_contexts_that_fill_the_whole_table(gpu, dtype, B):
    # the longest context a table row allows (max_blocks_per_seq * B tokens, no
    # spare column) next to shorter ones, with partitions of one block up to one
    # partition for the whole row
    torch, pa = gpu
    rng = synth.make_rng(4242 + B + 17 * synth.DTYPES.index(dtype))
    Hkv, G, D, mb = 2, 4, 128, 40
    lens = np.array([mb * B, 1, mb * B - 1, mb * B, B + 3], dtype=np.int32)
    N = int(synth.blocks_needed(lens, B).sum()) + 2
    tables, _ = synth.scattered_tables(rng, lens, B, N, shuffle=True, max_blocks=mb)
    assert tables.shape == (len(lens), mb) and (tables[lens == mb * B] >= 0).all()
    K = [synth.normal(rng, (int(n), Hkv, D), 1.0, dtype) for n in lens]
    V = [synth.normal(rng, (int(n), Hkv, D), 1.0, dtype) for n in lens]
    q = synth.normal(rng, (len(lens), G * Hkv, D), 1.0, dtype)
    kc, vc = scatter(K, tables, B, N, dtype), scatter(V, tables, B, N, dtype)
    scale = 1.0 / math.sqrt(D)
    ref = oracle.decode(q, kc, vc, tables, lens, scale, dtype)
    for psize in (0, B, 8 * B, mb * B):
        got = run_decode(torch, pa, dtype, q, kc, vc, tables, lens, scale, psize)
        assert_attention_close(got, ref)
    _check_no_device_errors(pa)


@pytest.mark.parametrize("name", ["mha7b", "gqa8b_b16", "gqa8b_b32", "long70b"])
def test_full_size_workloads_every_sequence(gpu, name):
    """The bench's own step at full size (allocator tables, KV write, then decode
    in the bench's launch configuration): every table and slot against the
    block-manager oracle, both caches byte for byte after the write, and every
    sequence's output against the fp64 oracle."""
    torch, pa = gpu
    st = workloads.build_step(name, seed=0, binding=pa)
    # the allocator's tables agree with the block-manager oracle driven the same way
    bm = BlockManager(st.num_blocks, st.block_size, st.free_order)
    w = synth.workload(name, 0)
    ids = []
    for n in w.lengths:
        s = bm.create()
        bm.append(s, int(n) - 1)
        ids.append(s)
    want_slots = [bm.append(s, 1)[0][0] for s in ids]
    assert st.slots.tolist() == want_slots
    for s in range(st.num_seqs):
        t = bm.table(ids[s])
        assert st.tables[s, :len(t)].tolist() == t and (st.tables[s, len(t):] == -1).all()
        assert st.lens[s] == bm.length(ids[s])

    dims = st.dims(pa)
    dq = to_dev(torch, st.q, st.dtype)
    dkc, dvc = to_dev(torch, st.k_cache, st.dtype), to_dev(torch, st.v_cache, st.dtype)
    dt = torch.from_numpy(st.tables).cuda()
    dl = torch.from_numpy(st.lens).cuda()
    out = torch.full((st.num_seqs, st.num_q_heads, st.head_dim), float("nan"), device="cuda")
    ws = torch.empty(max(pa.pa_decode_workspace_bytes(dims), 16), dtype=torch.uint8, device="cuda")
    pa.pa_write_kv(dims, to_dev(torch, st.k_new, st.dtype), to_dev(torch, st.v_new, st.dtype),
                   torch.from_numpy(st.slots).cuda(), dkc, dvc)
    pa.pa_decode(dims, dq, dkc, dvc, dt, dl, st.scale, out, ws)
    got = out.cpu().numpy().astype(np.float64)
    _check_no_device_errors(pa)
    assert np.isfinite(got).all()

    kc, vc = st.k_cache, st.v_cache
    oracle.write_kv(st.k_new, st.v_new, st.slots, kc, vc, st.dtype)
    assert to_host(dkc, st.dtype).tobytes() == kc.tobytes()
    assert to_host(dvc, st.dtype).tobytes() == vc.tobytes()
    del dkc, dvc
    ref = oracle.decode(st.q, kc, vc, st.tables, st.lens, st.scale, st.dtype)
    assert_attention_close(got, ref)


def test_prefix_sharing_and_copy_on_write_step(gpu):
    """Shared 800-token prefix + 32 pairs whose next write copies a partial block:
    allocator vs oracle model (bit-exact), then copy -> write -> decode vs the oracle."""
    torch, pa = gpu
    st = workloads.build_step("prefix_cow", seed=0, binding=pa)
    w = synth.workload("prefix_cow", 0)
    bm = BlockManager(st.num_blocks, st.block_size, st.free_order)
    root = bm.create()
    bm.append(root, w.prefix_len)
    ids = []
    for n in w.lengths:
        s = bm.fork(root)
        bm.append(s, int(n) - 1)
        ids.append(s)
    bm.free_seq(root)
    for _ in range(w.pair_count):
        a = bm.create()
        bm.append(a, w.pair_prefix)
        ids += [a, bm.fork(a)]
    want_slots, want_pairs = [], []
    for s in ids:
        sl, pr = bm.append(s, 1)
        want_slots += sl
        want_pairs += pr
    assert st.slots.tolist() == want_slots
    assert [tuple(p) for p in st.pairs.tolist()] == want_pairs
    assert len(want_pairs) == w.pair_count
    for i, s in enumerate(ids):
        assert st.tables[i, :len(bm.table(s))].tolist() == bm.table(s)
        assert st.lens[i] == bm.length(s)

    dims = st.dims(pa)
    dkc, dvc = to_dev(torch, st.k_cache, st.dtype), to_dev(torch, st.v_cache, st.dtype)
    pa.pa_copy_blocks(dims, dkc, dvc, torch.from_numpy(st.pairs).cuda())
    pa.pa_write_kv(dims, to_dev(torch, st.k_new, st.dtype), to_dev(torch, st.v_new, st.dtype),
                   torch.from_numpy(st.slots).cuda(), dkc, dvc)
    out = torch.full((st.num_seqs, st.num_q_heads, st.head_dim), float("nan"), device="cuda")
    ws = torch.empty(max(pa.pa_decode_workspace_bytes(dims), 16), dtype=torch.uint8, device="cuda")
    pa.pa_decode(dims, to_dev(torch, st.q, st.dtype), dkc, dvc, torch.from_numpy(st.tables).cuda(),
                 torch.from_numpy(st.lens).cuda(), st.scale, out, ws)
    got = out.cpu().numpy().astype(np.float64)
    _check_no_device_errors(pa)

    kc, vc = st.k_cache, st.v_cache
    oracle.copy_blocks(kc, vc, st.pairs, st.dtype)
    oracle.write_kv(st.k_new, st.v_new, st.slots, kc, vc, st.dtype)
    assert to_host(dkc, st.dtype).tobytes() == kc.tobytes()
    assert to_host(dvc, st.dtype).tobytes() == vc.tobytes()
    ref = oracle.decode(st.q, kc, vc, st.tables, st.lens, st.scale, st.dtype)
    assert_attention_close(got, ref)
