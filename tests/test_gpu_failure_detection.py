"""Failure detection on the GPU without a fault: the kernels' bounded waits
give up, report it, and leave the context usable.

Every wait of the library's kernels on an mbarrier is bounded; on running out
it records PA_DEVERR_TIMEOUT and the kernel returns.  pa_selftest_bounded_wait
runs that wait on an mbarrier nothing ever arrives at (no fault, no hang: a
bounded number of polls, each bounded in time by the hardware).
"""
import math
import time

import pytest

import oracle
from gpu_helpers import require_gpu, run_decode
from paged_helpers import assert_attention_close, random_case
from paged_kv_cache_127_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gpu():
    return require_gpu()


def test_bounded_wait_gives_up_and_the_context_stays_usable(gpu):
    torch, pa = gpu
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    pa.pa_selftest_bounded_wait(1024, status)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 10.0
    assert status.item() == pa.PA_DEVERR_TIMEOUT
    # the library's kernels still run, and correctly, in the same context
    rng = synth.make_rng(77)
    q, _, _, kc, vc, tables, lens = random_case(rng, "bf16", 3, 8, 2, 128, 16, [5, 40, 300])
    scale = 1.0 / math.sqrt(128)
    ref = oracle.decode(q, kc, vc, tables, lens, scale, "bf16")
    got = run_decode(torch, pa, "bf16", q, kc, vc, tables, lens, scale)
    assert_attention_close(got, ref)
    assert pa.pa_device_errors(clear=True) == 0


def test_selftest_rejects_bad_arguments_on_the_host(gpu):
    torch, pa = gpu
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    for limit in (0, (1 << 20) + 1):
        with pytest.raises(pa.PaError):
            pa.pa_selftest_bounded_wait(limit, status)
    assert pa.lib.pa_selftest_bounded_wait(16, None, None) == pa.PA_ERR_INVALID
