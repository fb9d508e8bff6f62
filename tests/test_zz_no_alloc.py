"""pa_decode_noalloc: decode for callers that cannot allocate device memory.

Code that runs inside a memory pool or arena that forbids further device
allocations, or inside a host that owns every allocation, cannot hand
pa_decode a workspace.  pa_decode_noalloc takes its scratch from a fixed
buffer built into the library instead.  These tests call it through the C ABI
and compare it with pa_decode given a caller workspace, on two calls in a row
(the shared buffer still holds the first call's data when the second runs),
and check that a problem needing more scratch than the buffer holds is refused.
"""
import ctypes
import math

import numpy as np
import pytest

from gpu_helpers import require_gpu, to_dev
from paged_helpers import assert_attention_close, random_case
from paged_kv_cache_127_gb300 import synth

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_decode_on_two_calls():
    torch, pa = require_gpu()
    rng = synth.make_rng(4242)
    dtype, Hkv, G, D, B = "bf16", 4, 4, 128, 16
    lens = [1, 16, 17, 300, 1500, 2047, 0, 700]
    q1, K, V, kc, vc, tables, lens = random_case(rng, dtype, len(lens), G * Hkv, Hkv, D, B, lens)
    q2 = synth.normal(rng, q1.shape, 1.0, dtype)
    S = len(lens)
    # 256-token partitions: long sequences go through split-K, so the scratch is used
    dims = pa.make_dims(S, G * Hkv, Hkv, D, B, kc.shape[0], tables.shape[1], 256, dtype)
    need = pa.pa_decode_workspace_bytes(dims)
    assert 0 < need <= pa.PA_NOALLOC_SCRATCH_BYTES

    dkc, dvc = to_dev(torch, kc, dtype), to_dev(torch, vc, dtype)
    dt = torch.from_numpy(tables).cuda()
    dl = torch.from_numpy(lens).cuda()
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    pa.pa_device_errors(clear=True)
    for q in (q1, q2):                      # two calls in a row, different queries
        dq = to_dev(torch, q, dtype)
        ref = torch.full((S, G * Hkv, D), float("nan"), device="cuda")
        pa.pa_decode(dims, dq, dkc, dvc, dt, dl, 1.0 / math.sqrt(D), ref, ws)
        got = torch.full((S, G * Hkv, D), float("nan"), device="cuda")
        pa.pa_decode_noalloc(dims, dq, dkc, dvc, dt, dl, 1.0 / math.sqrt(D), got)
        torch.cuda.synchronize()
        assert_attention_close(got.cpu().numpy(), ref.cpu().numpy())
        np.testing.assert_array_equal(got[torch.from_numpy(lens == 0).cuda()].cpu().numpy(), 0.0)
    assert pa.pa_device_errors(clear=True) == 0


def test_noalloc_refuses_problems_beyond_its_buffer():
    torch, pa = require_gpu()
    # 1024 sequences x 64 heads x 64 partitions of split-K partials: far above 64 MiB
    dims = pa.make_dims(1024, 64, 8, 128, 16, 100000, 2048, 512, "bf16")
    assert pa.pa_decode_workspace_bytes(dims) > pa.PA_NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(0x10000)         # refused before any pointer is used
    st = pa.lib.pa_decode_noalloc(ctypes.byref(dims), fake, fake, fake, fake, fake, 1.0, fake, None)
    assert st == pa.PA_ERR_TOO_LARGE
