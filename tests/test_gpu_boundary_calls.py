"""Boundary calls added for serving loops: prepared calls (checked and
marshalled once, issued many times) must give exactly what the direct calls
give, and pa_copy_to_device / pa_copy_to_host must move bytes unchanged."""
import math

import numpy as np
import pytest

import oracle
from gpu_helpers import require_gpu, to_dev, to_host
from paged_helpers import assert_attention_close, random_case
from paged_kv_cache_127_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_prepared_calls_match_direct_calls_bitwise(dtype):
    torch, pa = require_gpu()
    rng = synth.make_rng(771)
    Hkv, G, D, B = 4, 4, 128, 16
    lens = [1, 33, 700, 1500, 64, 0, 2047]
    q, K, V, kc, vc, tables, lens = random_case(rng, dtype, len(lens), G * Hkv, Hkv, D, B, lens)
    S = len(lens)
    dims = pa.make_dims(S, G * Hkv, Hkv, D, B, kc.shape[0], tables.shape[1], 256, dtype)
    dq = to_dev(torch, q, dtype)
    dt, dl = torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda()
    ws = torch.empty(max(pa.pa_decode_workspace_bytes(dims), 16), dtype=torch.uint8, device="cuda")
    # the new tokens: one row per sequence into free slots past every context
    free = [b for b in range(kc.shape[0]) if b not in set(int(x) for x in tables[tables >= 0].ravel())]
    slots = torch.tensor([free[i % len(free)] * B + i // len(free) for i in range(S)], dtype=torch.int64,
                         device="cuda")
    kn = to_dev(torch, synth.normal(rng, (S, Hkv, D), 1.0, dtype), dtype)
    vn = to_dev(torch, synth.normal(rng, (S, Hkv, D), 1.0, dtype), dtype)
    outs, caches = [], []
    for prepared in (False, True):
        dkc, dvc = to_dev(torch, kc, dtype), to_dev(torch, vc, dtype)
        out = torch.full((S, G * Hkv, D), float("nan"), device="cuda")
        if prepared:
            write = pa.pa_write_kv(dims, kn, vn, slots, dkc, dvc, prepare=True)
            dec = pa.pa_decode(dims, dq, dkc, dvc, dt, dl, 1.0 / math.sqrt(D), out, ws, prepare=True)
            assert isinstance(write, pa.Prepared) and isinstance(dec, pa.Prepared)
            for _ in range(2):      # issued twice: the same result
                write()
                dec()
        else:
            pa.pa_write_kv(dims, kn, vn, slots, dkc, dvc)
            pa.pa_decode(dims, dq, dkc, dvc, dt, dl, 1.0 / math.sqrt(D), out, ws)
        torch.cuda.synchronize()
        outs.append(out.cpu().numpy())
        caches.append((to_host(dkc, dtype), to_host(dvc, dtype)))
    assert outs[0].tobytes() == outs[1].tobytes()
    assert caches[0][0].tobytes() == caches[1][0].tobytes() and caches[0][1].tobytes() == caches[1][1].tobytes()
    want = oracle.decode(q, kc, vc, tables, lens, 1.0 / math.sqrt(D), dtype)
    assert_attention_close(outs[1], want)
    assert pa.pa_device_errors(clear=True) == 0


def test_host_device_copies_round_trip():
    torch, pa = require_gpu()
    rng = np.random.default_rng(5)
    host = torch.from_numpy(rng.integers(0, 256, size=3 * (1 << 20) + 48, dtype=np.uint8)).pin_memory()
    dev = torch.empty(host.numel(), dtype=torch.uint8, device="cuda")
    back = torch.zeros(host.numel(), dtype=torch.uint8).pin_memory()
    side = torch.cuda.Stream()
    pa.pa_copy_to_device(dev, host, stream=side)
    pa.pa_copy_to_host(back, dev, stream=side)
    side.synchronize()
    assert torch.equal(back, host)
    # prepared copies, and a float tensor viewed through its bytes
    f = torch.from_numpy(rng.standard_normal((64, 33), dtype=np.float32)).pin_memory()
    fd = torch.empty((64, 33), dtype=torch.float32, device="cuda")
    fb = torch.empty((64, 33), dtype=torch.float32).pin_memory()
    h2d, d2h = pa.pa_copy_to_device(fd, f, prepare=True), pa.pa_copy_to_host(fb, fd, prepare=True)
    h2d()
    d2h()
    torch.cuda.synchronize()
    assert torch.equal(fb, f)
    with pytest.raises(ValueError):
        pa.pa_copy_to_device(fd, torch.empty(7, dtype=torch.float32))   # byte sizes differ
