"""Block swap (preemption) between the device pool and pinned host memory."""
import math

import numpy as np
import pytest

import oracle
from gpu_helpers import require_gpu, to_dev, to_host
from paged_kv_cache_127_gb300 import synth, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gpu():
    return require_gpu()


def _pinned(torch, arr, dtype):
    t = to_dev(torch, arr, dtype, device="cpu")
    return t.pin_memory()


@pytest.mark.parametrize("dtype", synth.DTYPES)
@pytest.mark.parametrize("layers", [1, 3])
def test_swap_blocks_bit_exact_both_ways(gpu, dtype, layers):
    torch, pa = gpu
    rng = synth.make_rng(81 + layers)
    N, NH, Hkv, B, D = 30, 12, 4, 16, 64
    shape_d = ((layers,) if layers > 1 else ()) + (N, Hkv, B, D)
    shape_h = ((layers,) if layers > 1 else ()) + (NH, Hkv, B, D)
    kc, vc = synth.normal(rng, shape_d, 1.0, dtype), synth.normal(rng, shape_d, 1.0, dtype)
    hk0 = np.zeros(shape_h, synth.STORAGE[dtype])
    dkc, dvc = to_dev(torch, kc, dtype), to_dev(torch, vc, dtype)
    hk, hv = _pinned(torch, hk0, dtype), _pinned(torch, hk0, dtype)
    dims = pa.make_dims(0, Hkv, Hkv, D, B, N, 1, 0, dtype)
    out_pairs = np.stack([rng.permutation(N)[:7], rng.permutation(NH)[:7]], axis=1).astype(np.int64)
    pa.pa_swap_blocks(dims, dkc, dvc, hk, hv, torch.from_numpy(out_pairs).cuda(), pa.PA_SWAP_OUT)
    torch.cuda.synchronize()
    for layer in range(layers):
        pick = (lambda a: a[layer]) if layers > 1 else (lambda a: a)
        ek, ev = pick(hk0).copy(), pick(hk0).copy()
        oracle.swap_blocks(np.ascontiguousarray(pick(kc)), np.ascontiguousarray(pick(vc)), ek, ev, out_pairs, dtype)
        assert to_host(pick(hk), dtype).tobytes() == ek.tobytes()
        assert to_host(pick(hv), dtype).tobytes() == ev.tobytes()
    # and back into other device blocks
    in_pairs = np.stack([out_pairs[:, 1], rng.permutation(N)[:7]], axis=1).astype(np.int64)
    back_k, back_v = torch.zeros_like(dkc), torch.zeros_like(dvc)
    pa.pa_swap_blocks(dims, back_k, back_v, hk, hv, torch.from_numpy(in_pairs).cuda(), pa.PA_SWAP_IN)
    torch.cuda.synchronize()
    for (src_dev, _), (_, dst_dev) in zip(out_pairs, in_pairs):
        if layers == 1:
            assert to_host(back_k[dst_dev], dtype).tobytes() == kc[src_dev].tobytes()
            assert to_host(back_v[dst_dev], dtype).tobytes() == vc[src_dev].tobytes()
        else:
            assert to_host(back_k[:, dst_dev], dtype).tobytes() == np.ascontiguousarray(kc[:, src_dev]).tobytes()
            assert to_host(back_v[:, dst_dev], dtype).tobytes() == np.ascontiguousarray(vc[:, src_dev]).tobytes()
    assert pa.pa_device_errors(clear=True) == 0


def test_non_pinned_host_memory_is_rejected(gpu):
    torch, pa = gpu
    dims = pa.make_dims(0, 2, 2, 64, 16, 8, 1, 0, "bf16")
    dkc = torch.zeros((8, 2, 16, 64), dtype=torch.bfloat16, device="cuda")
    pageable = np.zeros((4, 2, 16, 64), np.uint16)          # ordinary host memory
    pairs = torch.tensor([[0, 1]], dtype=torch.int64, device="cuda")
    import ctypes
    st = pa.lib.pa_swap_blocks(ctypes.byref(dims), dkc.data_ptr(), dkc.data_ptr(), pageable.ctypes.data,
                               pageable.ctypes.data, 4, 1, 0, 0, pairs.data_ptr(), 1, pa.PA_SWAP_OUT, None)
    assert st == pa.PA_ERR_INVALID


def test_preempted_sequence_decodes_identically_after_swap_in(gpu):
    """Preemption round trip on the 8B-shaped workload: decode, swap a sequence
    out, let another sequence reuse and overwrite its blocks, swap it back in
    (new blocks), decode again: the same output, bit for bit."""
    torch, pa = gpu
    st = workloads.build_step("gqa8b_b16", seed=3, binding=pa).first(16)
    dims = st.dims(pa)
    dt = st.dtype
    dkc, dvc = to_dev(torch, st.k_cache, dt), to_dev(torch, st.v_cache, dt)
    dq = to_dev(torch, st.q, dt)
    ws = torch.empty(pa.pa_decode_workspace_bytes(dims), dtype=torch.uint8, device="cuda")

    def decode(tables, lens):
        out = torch.full((st.num_seqs, st.num_q_heads, st.head_dim), float("nan"), device="cuda")
        pa.pa_decode(dims, dq, dkc, dvc, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                     st.scale, out, ws)
        torch.cuda.synchronize()
        return out.cpu()

    before = decode(st.tables, st.lens)
    # replay the allocator exactly as the workload builder did (every context
    # without its newest token, then one batched append of the newest tokens)
    full = workloads.build_step("gqa8b_b16", seed=3, values=False, binding=pa)
    dev = pa.Pool(st.num_blocks, st.block_size, st.free_order)
    host = pa.Pool(4096, st.block_size)
    ids = []
    for s in range(full.num_seqs):
        sid = pa.pa_seq_create(dev.handle)
        pa.pa_seq_append(dev.handle, sid, int(full.lens[s]) - 1)
        ids.append(sid)
    pa.pa_seq_append_batch(dev.handle, ids, 1)
    tables, lens = pa.pa_pool_export(dev.handle, ids[:16], st.max_blocks, -1)
    assert (tables == st.tables).all() and (lens == st.lens).all()
    victim = 5
    hid, pairs = pa.pa_seq_swap_out(dev.handle, host.handle, ids[victim])
    hk = torch.empty((4096, st.num_kv_heads, st.block_size, st.head_dim), dtype=torch.bfloat16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    pa.pa_swap_blocks(dims, dkc, dvc, hk, hv, torch.from_numpy(pairs).cuda(), pa.PA_SWAP_OUT)
    # the freed device blocks are reused by someone else: overwrite every slot
    old = pairs[:, 0]
    slots = (old[:, None] * st.block_size + np.arange(st.block_size)[None, :]).reshape(-1).astype(np.int64)
    junk = torch.full((len(slots), st.num_kv_heads, st.head_dim), 7.0, dtype=torch.bfloat16, device="cuda")
    pa.pa_write_kv(dims, junk, junk, torch.from_numpy(slots).cuda(), dkc, dvc)
    # swap back in (fresh blocks) and decode with the new table
    new_id, back = pa.pa_seq_swap_in(dev.handle, host.handle, hid)
    pa.pa_swap_blocks(dims, dkc, dvc, hk, hv, torch.from_numpy(back).cuda(), pa.PA_SWAP_IN)
    ids[victim] = new_id
    tables2, lens2 = pa.pa_pool_export(dev.handle, ids[:16], st.max_blocks, -1)
    n = -(-int(lens[victim]) // st.block_size)
    assert not set(tables2[victim, :n].tolist()) & set(old.tolist())
    after = decode(tables2, lens2)
    assert torch.equal(before[victim], after[victim])
    assert pa.pa_device_errors(clear=True) == 0
    dev.close()
    host.close()
