"""pa_decode_noalloc: decode for callers that cannot allocate device memory.

Code that runs inside a memory pool or arena that forbids further device
allocations, or inside a host that owns every allocation, cannot hand
pa_decode a workspace.  pa_decode_noalloc takes its scratch from a fixed
buffer built into the library instead.  These tests call it through the C ABI
and compare it with pa_decode given a caller workspace, on two calls in a row
(the shared buffer still holds the first call's data when the second runs),
in every cache dtype -- the f32 path runs a CUDA-core kernel and the merge on
that buffer, the 16-bit paths the tensor-core kernel -- on the default stream
and on a stream of the caller's, and against the fp64 oracle.  A problem
needing more scratch than the buffer holds must be refused.
"""
import ctypes
import math

import numpy as np
import pytest

import oracle
from gpu_helpers import require_gpu, to_dev
from paged_helpers import assert_attention_close, random_case
from paged_kv_cache_127_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", synth.DTYPES)
def test_noalloc_matches_workspace_decode_on_two_calls(dtype):
    torch, pa = require_gpu()
    rng = synth.make_rng(4242 + synth.DTYPES.index(dtype))
    Hkv, G, D, B = 4, 4, 128, 16
    lens = [1, 16, 17, 300, 1500, 2047, 0, 700]
    q1, K, V, kc, vc, tables, lens = random_case(rng, dtype, len(lens), G * Hkv, Hkv, D, B, lens)
    q2 = synth.normal(rng, q1.shape, 1.0, dtype)
    S = len(lens)
    scale = 1.0 / math.sqrt(D)
    # 256-token partitions: long sequences go through split-K, so the scratch is used
    dims = pa.make_dims(S, G * Hkv, Hkv, D, B, kc.shape[0], tables.shape[1], 256, dtype)
    need = pa.pa_decode_workspace_bytes(dims)
    assert 0 < need <= pa.PA_NOALLOC_SCRATCH_BYTES

    dkc, dvc = to_dev(torch, kc, dtype), to_dev(torch, vc, dtype)
    dt = torch.from_numpy(tables).cuda()
    dl = torch.from_numpy(lens).cuda()
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    pa.pa_device_errors(clear=True)
    # two calls in a row on the default stream, then one on the caller's own stream
    for q, stream in ((q1, None), (q2, None), (q1, side)):
        dq = to_dev(torch, q, dtype)
        torch.cuda.synchronize()
        ref = torch.full((S, G * Hkv, D), float("nan"), device="cuda")
        got = torch.full((S, G * Hkv, D), float("nan"), device="cuda")
        pa.pa_decode(dims, dq, dkc, dvc, dt, dl, scale, ref, ws, stream=stream)
        pa.pa_decode_noalloc(dims, dq, dkc, dvc, dt, dl, scale, got, stream=stream)
        torch.cuda.synchronize()
        got_h, ref_h = got.cpu().numpy(), ref.cpu().numpy()
        assert_attention_close(got_h, ref_h)
        np.testing.assert_array_equal(got_h[lens == 0], 0.0)
        want = oracle.decode(q, kc, vc, tables, lens, scale, dtype)
        assert_attention_close(got_h, want)
    assert pa.pa_device_errors(clear=True) == 0


def test_noalloc_refuses_problems_beyond_its_buffer():
    torch, pa = require_gpu()
    # 1024 sequences x 64 heads x 64 partitions of split-K partials: far above 64 MiB
    dims = pa.make_dims(1024, 64, 8, 128, 16, 100000, 2048, 512, "bf16")
    assert pa.pa_decode_workspace_bytes(dims) > pa.PA_NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(0x10000)         # refused before any pointer is used
    st = pa.lib.pa_decode_noalloc(ctypes.byref(dims), fake, fake, fake, fake, fake, 1.0, fake, None)
    assert st == pa.PA_ERR_TOO_LARGE
