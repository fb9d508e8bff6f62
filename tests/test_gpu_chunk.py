"""GPU parity for chunk attention (several query tokens per sequence, causal)
through the C ABI, against the fp64 oracle; tolerance as for decode."""
import math

import numpy as np
import pytest

import oracle
from gpu_helpers import poison_unused, require_gpu, to_dev, to_host
from paged_helpers import assert_attention_close, random_case
from paged_kv_cache_127_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gpu():
    return require_gpu()


def run_chunk(torch, pa, dtype, q, kc, vc, tables, lens, qs, scale, max_q=None, partition_size=0, out_fill=float("nan")):
    T, Hq, D = q.shape
    N, Hkv, B, _ = kc.shape
    S = len(lens)
    max_q = int(np.diff(qs).max(initial=1)) if max_q is None else max_q
    dims = pa.make_dims(S, Hq, Hkv, D, B, N, tables.shape[1], partition_size, dtype)
    dq, dk, dv = to_dev(torch, q, dtype), to_dev(torch, kc, dtype), to_dev(torch, vc, dtype)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    out = torch.full((T, Hq, D), out_fill, dtype=torch.float32, device="cuda")
    nbytes = pa.pa_chunk_workspace_bytes(dims, T, max_q)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    pa.pa_chunk_attention(dims, dq, dk, dv, i32(tables), i32(lens), i32(qs), scale, out, max_q, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64)


def chunk_case(rng, dtype, Hq, Hkv, D, B, lens, nq, std=1.0):
    _, K, V, kc, vc, tables, lens = random_case(rng, dtype, len(lens), Hq, Hkv, D, B, lens, std=std)
    qs = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    q = synth.normal(rng, (int(qs[-1]), Hq, D), std, dtype)
    return q, kc, vc, tables, lens, qs


SHAPES = [(D, B, G) for D in (64, 128) for B in (16, 32) for G in (1, 2, 4, 8)]


# Short chunks (at most 7 tokens: fewer than 64 rows per KV head) take the
# mma.sync kernel with split-K; long ones (70 tokens) the tcgen05 kernel.
@pytest.mark.parametrize("path", ["mma", "umma"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D,B,G", SHAPES)
def test_chunk_small_shapes(gpu, dtype, D, B, G, path):
    torch, pa = gpu
    rng = synth.make_rng(3000 + D + B + 7 * G + 101 * (dtype == "bf16") + 13 * (path == "umma"))
    Hkv = 2
    # ragged: one query, a few drafted tokens, a query range crossing blocks and
    # partitions, a whole short sequence, an empty range
    lens = [1, 9, B + 3, 200, 530, 40, 7]
    nq = [1, 5, B + 3, 33, 70, 0, 7] if path == "umma" else [1, 5, 3, 7, 2, 0, 7]
    q, kc, vc, tables, lens, qs = chunk_case(rng, dtype, G * Hkv, Hkv, D, B, lens, nq)
    scale = 1.0 / math.sqrt(D)
    ref = oracle.chunk_attention(q, kc, vc, tables, lens, qs, scale, dtype)
    for psize in (0, B, 4 * B):
        got = run_chunk(torch, pa, dtype, q, kc, vc, tables, lens, qs, scale, partition_size=psize)
        assert_attention_close(got, ref)
    assert pa.pa_device_errors(clear=True) == 0


@pytest.mark.parametrize("nq,max_q", [(1, 1), (4, 4), (5, 5), (8, 8), (3, 16), (64, 64), (33, 33), (20, 64),
                                      (40, 64)])
def test_chunk_query_lengths_and_row_blocks(gpu, nq, max_q):
    # G = 4: 4 rows per token.  mma.sync path: one tile (<= 4 tokens), one block
    # of two tiles (5..8), a loose bound (3 of 16).  tcgen05 path: one 128-row
    # tile per CTA (33 tokens = 132 rows, two CTAs), two tiles per CTA (64
    # tokens), a CTA whose second tile has no row (20 of 64) and one whose
    # second tile is partly filled (40 of 64)
    torch, pa = gpu
    rng = synth.make_rng(3100 + nq)
    lens = [nq, nq + 1, 600, 1100, 64 + nq]
    q, kc, vc, tables, lens, qs = chunk_case(rng, "bf16", 32, 8, 128, 16, lens, [nq] * 5)
    ref = oracle.chunk_attention(q, kc, vc, tables, lens, qs, 1 / math.sqrt(128), "bf16")
    got = run_chunk(torch, pa, "bf16", q, kc, vc, tables, lens, qs, 1 / math.sqrt(128), max_q=max_q)
    assert_attention_close(got, ref)
    assert pa.pa_device_errors(clear=True) == 0


def test_chunk_poison_and_placement_invariance(gpu):
    torch, pa = gpu
    dtype, B = "bf16", 16
    rng = synth.make_rng(3200)
    lens = np.array([700, 16, 5, 1029], np.int32)
    nq = [6, 16, 5, 6]
    q, kc, vc, tables, lens, qs = chunk_case(rng, dtype, 16, 4, 128, B, lens, nq)
    base = run_chunk(torch, pa, dtype, q, kc, vc, tables, lens, qs, 0.1)
    # NaN in every slot no context covers changes nothing, bit for bit
    kc2, vc2 = kc.copy(), vc.copy()
    poison_unused(kc2, vc2, tables, lens, B, dtype)
    np.testing.assert_array_equal(run_chunk(torch, pa, dtype, q, kc2, vc2, tables, lens, qs, 0.1), base)
    # moving every block elsewhere in a bigger pool changes nothing either
    N = kc.shape[0]
    perm = synth.make_rng(9).permutation(N + 40)[:N]
    kc3 = np.full((N + 40,) + kc.shape[1:], synth.nan_value(dtype), kc.dtype)
    vc3 = kc3.copy()
    kc3[perm], vc3[perm] = kc, vc
    t3 = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1).astype(np.int32)
    np.testing.assert_array_equal(run_chunk(torch, pa, dtype, q, kc3, vc3, t3, lens, qs, 0.1), base)
    assert np.isfinite(base).all()
    assert pa.pa_device_errors(clear=True) == 0


def test_chunk_bad_ranges_are_flagged_and_skipped(gpu):
    torch, pa = gpu
    rng = synth.make_rng(3300)
    q, kc, vc, tables, lens, qs = chunk_case(rng, "f16", 8, 2, 64, 16, [10, 20, 30], [2, 3, 4])
    ref = oracle.chunk_attention(q, kc, vc, tables, lens, qs, 0.125, "f16")
    # sequence 2 has more queries than max_query_len: skipped, flagged, the others exact
    got = run_chunk(torch, pa, "f16", q, kc, vc, tables, lens, qs, 0.125, max_q=3, out_fill=7.0)
    assert pa.pa_device_errors(clear=True) == pa.PA_DEVERR_BAD_LEN
    assert_attention_close(got[:5], ref[:5])
    assert (got[5:] == 7.0).all()
    # more queries than stored tokens
    bad_lens = lens.copy()
    bad_lens[0] = 1
    got = run_chunk(torch, pa, "f16", q, kc, vc, tables, bad_lens, qs, 0.125, out_fill=7.0)
    assert pa.pa_device_errors(clear=True) == pa.PA_DEVERR_BAD_LEN
    assert (got[:2] == 7.0).all()
    assert_attention_close(got[2:], ref[2:])
    # decreasing query_start: every sequence skipped
    got = run_chunk(torch, pa, "f16", q, kc, vc, tables, lens, np.array([0, 4, 3, 9], np.int32), 0.125,
                    max_q=6, out_fill=7.0)
    assert pa.pa_device_errors(clear=True) == pa.PA_DEVERR_BAD_LEN
    assert (got == 7.0).all()


def test_chunk_large_logits_and_long_context(gpu):
    # one dominant key per query far from the chunk, across several partitions
    torch, pa = gpu
    rng = synth.make_rng(3400)
    q, kc, vc, tables, lens, qs = chunk_case(rng, "bf16", 8, 2, 128, 16, [3000, 2100], [8, 8], std=2.0)
    ref = oracle.chunk_attention(q, kc, vc, tables, lens, qs, 0.5, "bf16")
    got = run_chunk(torch, pa, "bf16", q, kc, vc, tables, lens, qs, 0.5)
    assert_attention_close(got, ref)
    assert pa.pa_device_errors(clear=True) == 0


@pytest.mark.parametrize("name", ["verify8b", "prefill8b"])
def test_chunk_full_size_workloads_every_sequence(gpu, name):
    """The bench's own chunk step at full size (allocator tables and slots, KV
    write of every new token, chunk attention).  Both caches are compared byte
    for byte after the write, and every sequence's output against the oracle:
    all query rows of verify8b's 5-token chunks; for prefill8b's 512-token
    chunks, three 8-row spans (first, middle, last) of every sequence, since
    all 8,192 rows would take the fp64 oracle several minutes."""
    from paged_kv_cache_127_gb300 import workloads
    torch, pa = gpu
    st = workloads.build_step(name, seed=0, binding=pa)
    dims = st.dims(pa)
    n = st.query_len
    dkc, dvc = to_dev(torch, st.k_cache, st.dtype), to_dev(torch, st.v_cache, st.dtype)
    pa.pa_write_kv(dims, to_dev(torch, st.k_new, st.dtype), to_dev(torch, st.v_new, st.dtype),
                   torch.from_numpy(st.slots).cuda(), dkc, dvc)
    out = torch.full((st.num_tokens, st.num_q_heads, st.head_dim), float("nan"), device="cuda")
    ws = torch.empty(max(pa.pa_chunk_workspace_bytes(dims, st.num_tokens, n), 16), dtype=torch.uint8, device="cuda")
    pa.pa_chunk_attention(dims, to_dev(torch, st.q, st.dtype), dkc, dvc, torch.from_numpy(st.tables).cuda(),
                          torch.from_numpy(st.lens).cuda(), torch.from_numpy(st.query_start()).cuda(), st.scale,
                          out, n, ws)
    got = out.cpu().numpy().astype(np.float64)
    assert pa.pa_device_errors(clear=True) == 0
    assert np.isfinite(got).all()
    kc, vc = st.k_cache, st.v_cache
    oracle.write_kv(st.k_new, st.v_new, st.slots, kc, vc, st.dtype)
    assert to_host(dkc, st.dtype).tobytes() == kc.tobytes()
    assert to_host(dvc, st.dtype).tobytes() == vc.tobytes()
    del dkc, dvc
    if n <= 16:
        ref = oracle.chunk_attention(st.q, kc, vc, st.tables, st.lens, st.query_start(), st.scale, st.dtype)
        assert_attention_close(got, ref)
        return
    # rows a..b-1 of a chunk are the last b - a queries of the context cut after
    # row b - 1 (causality), so the oracle checks a few rows of a long chunk cheaply
    for s in range(st.num_seqs):
        for a0, b0 in ((0, 8), (n // 2 - 4, n // 2 + 4), (n - 8, n)):
            cut = int(st.lens[s]) - n + b0
            ref = oracle.chunk_attention(st.q[s * n + a0:s * n + b0], kc, vc, st.tables[s:s + 1],
                                         np.array([cut], np.int32), np.array([0, b0 - a0], np.int32),
                                         st.scale, st.dtype)
            assert_attention_close(got[s * n + a0:s * n + b0], ref)


@pytest.mark.parametrize("path,nq", [("mma", 6), ("umma", 40)])
def test_chunk_bad_block_entry_is_flagged_and_skipped(gpu, path, nq):
    # a table entry outside the pool inside the context: its keys are skipped
    # (every query attends to the remaining keys), PA_DEVERR_BAD_BLOCK is raised
    # and the other sequence is untouched
    from scipy.special import softmax
    from paged_helpers import widen
    torch, pa = gpu
    rng = synth.make_rng(3500 + nq)
    B, Hq, Hkv, D = 16, 16, 4, 128
    q, kc, vc, tables, lens, qs = chunk_case(rng, "bf16", Hq, Hkv, D, B, [300, 300], [nq, nq])
    bad = tables.copy()
    bad[1, 10] = kc.shape[0] + 7                        # block 10 of sequence 1: tokens 160..175
    got = run_chunk(torch, pa, "bf16", q, kc, vc, bad, lens, qs, 0.1)
    assert pa.pa_device_errors(clear=True) & pa.PA_DEVERR_BAD_BLOCK
    ref = oracle.chunk_attention(q, kc, vc, tables, lens, qs, 0.1, "bf16")
    assert_attention_close(got[:nq], ref[:nq])          # sequence 0 is untouched
    # sequence 1: unpaged attention with tokens 160..175 removed
    K = widen(np.stack([kc[tables[1, t // B], :, t % B] for t in range(300)]), "bf16")
    V = widen(np.stack([vc[tables[1, t // B], :, t % B] for t in range(300)]), "bf16")
    q64 = widen(q[nq:], "bf16")
    keep = np.ones(300, bool)
    keep[160:176] = False
    want = np.zeros((nq, Hq, D))
    G = Hq // Hkv
    for t in range(nq):
        vis = keep & (np.arange(300) <= 300 - nq + t)
        for h in range(Hq):
            w = softmax(0.1 * (K[vis, h // G] @ q64[t, h]))
            want[t, h] = w @ V[vis, h // G]
    assert_attention_close(got[nq:], want)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_chunk_persistent_ctas_over_mixed_tiles(gpu, dtype):
    # The tcgen05 kernel is persistent: each CTA walks several work items and
    # keeps its TMEM, barriers and rings across them.  96 sequences with chunk
    # lengths cycling through 96, 64, 33, 80, 0 and 70 tokens (G = 4, so 384,
    # 256, 132, 320, 0 and 280 rows, two 128-row tiles per item) give 512 work
    # items for at most one CTA per SM: items with two full tiles, a full and a
    # partly filled tile, one tile (the second tile's roles skip the item), and
    # sequences with no item, mixed within each CTA's sequence of items.
    torch, pa = gpu
    rng = synth.make_rng(3300 + (dtype == "bf16"))
    Hq, Hkv, D, B = 16, 4, 128, 16
    nq = [96, 64, 33, 80, 0, 70] * 16
    lens = [n + int(x) for n, x in zip(nq, rng.integers(1, 300, len(nq)))]
    q, kc, vc, tables, lens, qs = chunk_case(rng, dtype, Hq, Hkv, D, B, lens, nq)
    scale = 1.0 / math.sqrt(D)
    ref = oracle.chunk_attention(q, kc, vc, tables, lens, qs, scale, dtype)
    got = run_chunk(torch, pa, dtype, q, kc, vc, tables, lens, qs, scale)
    assert_attention_close(got, ref)
    assert pa.pa_device_errors(clear=True) == 0
