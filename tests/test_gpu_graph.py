"""Multi-layer pools: the layered block copy and the captured L-layer decode step.

The step graph must reproduce, bit for bit, the same launches made one by one,
read its input buffers afresh at every launch, and match the oracle."""
import math

import numpy as np
import pytest

import oracle
from gpu_helpers import require_gpu, to_dev, to_host
from paged_helpers import assert_attention_close, random_case
from paged_kv_cache_127_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gpu():
    return require_gpu()


@pytest.mark.parametrize("dtype", synth.DTYPES)
def test_copy_blocks_layers_bit_exact(gpu, dtype):
    torch, pa = gpu
    rng = synth.make_rng(61)
    L, N, Hkv, B, D = 3, 40, 4, 16, 64
    kc = synth.normal(rng, (L, N, Hkv, B, D), 1.0, dtype)
    vc = synth.normal(rng, (L, N, Hkv, B, D), 1.0, dtype)
    pairs = synth.copy_pairs(rng, 9, N)
    dims = pa.make_dims(0, Hkv, Hkv, D, B, N, 1, 0, dtype)
    dkc, dvc = to_dev(torch, kc, dtype), to_dev(torch, vc, dtype)
    pa.pa_copy_blocks_layers(dims, dkc, dvc, torch.from_numpy(pairs).cuda())
    for layer in range(L):
        k_l, v_l = kc[layer].copy(), vc[layer].copy()
        oracle.copy_blocks(k_l, v_l, pairs, dtype)
        assert to_host(dkc[layer], dtype).tobytes() == k_l.tobytes()
        assert to_host(dvc[layer], dtype).tobytes() == v_l.tobytes()
    assert pa.pa_device_errors(clear=True) == 0


def test_step_graph_equals_eager_launches_and_oracle(gpu):
    torch, pa = gpu
    dtype, L, Hkv, G, D, B = "bf16", 3, 2, 4, 128, 16
    rng = synth.make_rng(62)
    lens = [1, 17, 300, 530, 64, 700]
    S = len(lens)
    _, _, _, kc0, _, tables, lens = random_case(rng, dtype, S, G * Hkv, Hkv, D, B, lens, extra_blocks=8)
    N = kc0.shape[0]
    kc = synth.normal(rng, (L, N, Hkv, B, D), 1.0, dtype)
    vc = synth.normal(rng, (L, N, Hkv, B, D), 1.0, dtype)
    # each sequence's newest token is written this step, at position len - 1
    pos = lens - 1
    slots = oracle.slot_mapping(tables, B, np.arange(S, dtype=np.int32), pos)
    dims = pa.make_dims(S, G * Hkv, Hkv, D, B, N, tables.shape[1], 64, dtype)   # split-K partitions
    scale = 1.0 / math.sqrt(D)

    def draw_inputs():
        return (synth.normal(rng, (L, S, G * Hkv, D), 1.0, dtype), synth.normal(rng, (L, S, Hkv, D), 1.0, dtype),
                synth.normal(rng, (L, S, Hkv, D), 1.0, dtype))

    # graph buffers (fixed) and an eager copy of everything
    q, kn, vn = draw_inputs()
    g_kc, g_vc = to_dev(torch, kc, dtype), to_dev(torch, vc, dtype)
    e_kc, e_vc = to_dev(torch, kc, dtype), to_dev(torch, vc, dtype)
    d_q, d_kn, d_vn = to_dev(torch, q, dtype), to_dev(torch, kn, dtype), to_dev(torch, vn, dtype)
    d_slots = torch.from_numpy(slots).cuda()
    d_tab = torch.from_numpy(tables).cuda()
    d_len = torch.from_numpy(lens).cuda()
    g_out = torch.full((L, S, G * Hkv, D), float("nan"), device="cuda")
    ws = torch.empty(pa.pa_decode_workspace_bytes(dims), dtype=torch.uint8, device="cuda")
    graph = pa.pa_step_graph_create(dims, g_kc, g_vc, d_q, d_kn, d_vn, d_slots, d_tab, d_len, scale, g_out, ws)
    e_ws = torch.empty_like(ws)
    for step in range(2):
        if step:                                       # new inputs in the same buffers
            q, kn, vn = draw_inputs()
            d_q.copy_(to_dev(torch, q, dtype))
            d_kn.copy_(to_dev(torch, kn, dtype))
            d_vn.copy_(to_dev(torch, vn, dtype))
        graph.launch()
        e_out = torch.full_like(g_out, float("nan"))
        for layer in range(L):
            pa.pa_write_kv(dims, d_kn[layer], d_vn[layer], d_slots, e_kc[layer], e_vc[layer])
            pa.pa_decode(dims, d_q[layer], e_kc[layer], e_vc[layer], d_tab, d_len, scale, e_out[layer], e_ws)
        torch.cuda.synchronize()
        assert torch.equal(g_out, e_out), "graph replay differs from the same launches made eagerly"
        assert torch.equal(g_kc.view(torch.int16), e_kc.view(torch.int16))
        assert torch.equal(g_vc.view(torch.int16), e_vc.view(torch.int16))
        # and layer L-1 against the oracle (each step rewrites the same slots, so
        # the initial pool plus this step's rows is the state the decode saw)
        k_l, v_l = kc[L - 1].copy(), vc[L - 1].copy()
        oracle.write_kv(kn[L - 1], vn[L - 1], slots, k_l, v_l, dtype)
        ref = oracle.decode(q[L - 1], k_l, v_l, tables, lens, scale, dtype)
        assert_attention_close(g_out[L - 1].cpu().numpy(), ref)
    graph.close()
    assert pa.pa_device_errors(clear=True) == 0


@pytest.mark.parametrize("psize", [0, 64])
def test_step_graph_plan_serves_every_layer(gpu, psize):
    """One work list per step: every layer matches the oracle, empty contexts
    give zero rows in every layer, and a second launch (counters reset by the
    decode kernel itself) gives the same bits."""
    torch, pa = gpu
    dtype, L, Hkv, G, D, B = "f16", 4, 4, 2, 64, 16
    rng = synth.make_rng(63)
    lens = [0, 40, 1, 333, 0, 129]
    S = len(lens)
    _, _, _, kc0, _, tables, lens = random_case(rng, dtype, S, G * Hkv, Hkv, D, B, lens, extra_blocks=4)
    N = kc0.shape[0]
    kc = synth.normal(rng, (L, N, Hkv, B, D), 1.0, dtype)
    vc = synth.normal(rng, (L, N, Hkv, B, D), 1.0, dtype)
    slots = oracle.slot_mapping(tables, B, np.arange(S, dtype=np.int32), lens - 1)   # -1: empty, skipped
    dims = pa.make_dims(S, G * Hkv, Hkv, D, B, N, tables.shape[1], psize, dtype)
    q = synth.normal(rng, (L, S, G * Hkv, D), 1.0, dtype)
    kn = synth.normal(rng, (L, S, Hkv, D), 1.0, dtype)
    vn = synth.normal(rng, (L, S, Hkv, D), 1.0, dtype)
    d_kc, d_vc = to_dev(torch, kc, dtype), to_dev(torch, vc, dtype)
    out = torch.full((L, S, G * Hkv, D), float("nan"), device="cuda")
    ws = torch.empty(max(pa.pa_decode_workspace_bytes(dims), 16), dtype=torch.uint8, device="cuda")
    graph = pa.pa_step_graph_create(dims, d_kc, d_vc, to_dev(torch, q, dtype), to_dev(torch, kn, dtype),
                                    to_dev(torch, vn, dtype), torch.from_numpy(slots).cuda(),
                                    torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(), 0.125, out, ws)
    graph.launch()
    torch.cuda.synchronize()
    first = out.clone()
    out.fill_(float("nan"))
    graph.launch()                                     # rewrites the same slots with the same rows
    torch.cuda.synchronize()
    assert torch.equal(out, first)
    got = first.cpu().numpy().astype(np.float64)
    for layer in range(L):
        k_l, v_l = kc[layer].copy(), vc[layer].copy()
        oracle.write_kv(kn[layer], vn[layer], slots, k_l, v_l, dtype)
        ref = oracle.decode(q[layer], k_l, v_l, tables, lens, 0.125, dtype)
        assert_attention_close(got[layer], ref)
        np.testing.assert_array_equal(got[layer][lens == 0], 0.0)
    graph.close()
    assert pa.pa_device_errors(clear=True) == 0
