"""The C-ABI library loads on a CPU-only host and exports what include/pa.h declares.

No call here reaches the GPU: only symbol lookup, the version string, the
workspace-size arithmetic and host-side argument validation.
"""
import ctypes
import os
import re
import subprocess

import pytest

from paged_kv_cache_127_gb300 import build as pa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")


@pytest.fixture(scope="module")
def pa():
    pa_build.build()
    from paged_kv_cache_127_gb300 import binding
    return binding


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^PA_API [^;]*?\b(pa_\w+)\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = _declared()
    for must in ("pa_decode", "pa_write_kv", "pa_copy_blocks", "pa_decode_workspace_bytes",
                 "pa_pool_create", "pa_seq_append", "pa_seq_fork", "pa_seq_free"):
        assert must in names


def test_library_exports_every_declared_symbol(pa):
    out = subprocess.run(["nm", "-D", "--defined-only", pa.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (pa_\w+)$", out, flags=re.M))
    declared = set(_declared())
    assert declared <= exported, f"missing: {sorted(declared - exported)}"
    assert exported <= declared, f"exported but undeclared: {sorted(exported - declared)}"
    for name in declared:
        assert getattr(pa.lib, name)


def test_binding_covers_every_symbol(pa):
    for name in _declared():
        assert name in pa._SIGNATURES
        assert hasattr(pa, name)


def test_version(pa):
    assert "sm_103a" in pa.pa_version()


def test_workspace_bytes(pa):
    def up(x):
        return (x + 255) // 256 * 256

    S, Hq, Hkv, D = 256, 32, 8, 128
    d = pa.make_dims(num_seqs=S, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=16,
                     num_blocks=1000, max_blocks_per_seq=256, partition_size=512, kv_dtype="bf16")
    P = (256 * 16 + 511) // 512
    expect = 256 + up(S * P * 16) + up(S * Hq * P * D * 4) + up(S * Hq * P * 2 * 4)
    assert pa.pa_decode_workspace_bytes(d) == expect
    d.max_blocks_per_seq = 32            # one partition covers every context: no partials
    assert pa.pa_decode_workspace_bytes(d) == 256 + up(S * 16)
    d.num_seqs = 0
    assert pa.pa_decode_workspace_bytes(d) == 0
    d.num_seqs = S
    d.num_q_heads = 30                   # Hq not a multiple of Hkv: invalid -> 0
    assert pa.pa_decode_workspace_bytes(d) == 0


def _decode_status(pa, **over):
    kw = dict(num_seqs=2, num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16, num_blocks=8,
              max_blocks_per_seq=4, partition_size=0, kv_dtype="bf16")
    kw.update(over)
    d = pa.make_dims(**kw)
    fake = ctypes.c_void_p(0x10000)      # never dereferenced: validation fails first
    return pa.lib.pa_decode(ctypes.byref(d), fake, fake, fake, fake, fake, 1.0, fake, None, 0, None)


def test_decode_rejects_bad_arguments_on_the_host(pa):
    assert _decode_status(pa, num_q_heads=7) == pa.PA_ERR_INVALID
    assert _decode_status(pa, head_dim=96) == pa.PA_ERR_UNSUPPORTED
    assert _decode_status(pa, block_size=8) == pa.PA_ERR_UNSUPPORTED
    assert _decode_status(pa, num_q_heads=32, num_kv_heads=2) == pa.PA_ERR_UNSUPPORTED   # G = 16
    assert _decode_status(pa, partition_size=24) == pa.PA_ERR_INVALID                   # not a multiple of B
    assert _decode_status(pa, kv_dtype=7) == pa.PA_ERR_INVALID
    assert _decode_status(pa, num_blocks=0) == pa.PA_ERR_INVALID
    # needs a workspace but none is given
    assert _decode_status(pa, partition_size=32) == pa.PA_ERR_INVALID
    assert _decode_status(pa) == pa.PA_ERR_INVALID
    assert _decode_status(pa, num_seqs=0) == pa.PA_OK             # nothing to do
    assert _decode_status(pa, num_seqs=-1) == pa.PA_ERR_INVALID
    d = pa.make_dims(num_seqs=1, num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                     num_blocks=8, max_blocks_per_seq=4)
    assert pa.lib.pa_decode(ctypes.byref(d), None, None, None, None, None, 1.0, None, None, 0,
                            None) == pa.PA_ERR_INVALID
    odd = ctypes.c_void_p(0x10004)       # not 16-byte aligned
    ok = ctypes.c_void_p(0x10000)
    assert pa.lib.pa_decode(ctypes.byref(d), odd, ok, ok, ok, ok, 1.0, ok, None, 0,
                            None) == pa.PA_ERR_INVALID


def test_write_and_copy_reject_bad_arguments_on_the_host(pa):
    d = pa.make_dims(num_kv_heads=2, head_dim=128, block_size=16, num_blocks=8, kv_dtype="f16")
    ok = ctypes.c_void_p(0x10000)
    assert pa.lib.pa_write_kv(ctypes.byref(d), ok, ok, ok, -1, ok, ok, None) == pa.PA_ERR_INVALID
    assert pa.lib.pa_write_kv(ctypes.byref(d), ok, ok, ok, 0, ok, ok, None) == pa.PA_OK   # no-op
    assert pa.lib.pa_write_kv(ctypes.byref(d), None, ok, ok, 3, ok, ok, None) == pa.PA_ERR_INVALID
    assert pa.lib.pa_copy_blocks(ctypes.byref(d), ok, ok, ok, -2, None) == pa.PA_ERR_INVALID
    assert pa.lib.pa_copy_blocks(ctypes.byref(d), ok, ok, ok, 0, None) == pa.PA_OK        # no-op
    bad = pa.make_dims(num_kv_heads=2, head_dim=4, block_size=16, num_blocks=8, kv_dtype="f16")
    assert pa.lib.pa_copy_blocks(ctypes.byref(bad), ok, ok, ok, 1, None) == pa.PA_ERR_UNSUPPORTED


def test_chunk_workspace_bytes(pa):
    def up(x):
        return (x + 255) // 256 * 256

    S, Hq, Hkv, D, T = 64, 32, 8, 128, 320
    d = pa.make_dims(num_seqs=S, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=16,
                     num_blocks=1000, max_blocks_per_seq=256, partition_size=512, kv_dtype="bf16")
    P = (256 * 16 + 511) // 512
    # five queries per sequence, G = 4: 20 rows -> two 16-row tiles, one row block of two
    R = 1
    expect = 256 + up(S * P * R * 16) + up(T * 4) + up(T * Hq * P * D * 4) + up(T * Hq * P * 2 * 4)
    assert pa.pa_chunk_workspace_bytes(d, T, 5) == expect
    # four queries: 16 rows, one tile per block; 64 queries: 256 rows in blocks of 32 -> 8 blocks
    assert pa.pa_chunk_workspace_bytes(d, T, 4) == 256 + up(S * P * 16) + up(T * 4) + \
        up(T * Hq * P * D * 4) + up(T * Hq * P * 2 * 4)
    # 64 queries x 4 heads >= 64 rows: the tcgen05 path, which keeps no split-K partials
    assert pa.pa_chunk_workspace_bytes(d, T, 64) == 256 + up(S * P * 8 * 16) + up(T * 4)
    assert pa.pa_chunk_workspace_bytes(d, T, 15) == 256 + up(S * P * 2 * 16) + up(T * 4) + \
        up(T * Hq * P * D * 4) + up(T * Hq * P * 2 * 4)
    assert pa.pa_chunk_workspace_bytes(d, T, 16) == 256 + up(S * P * 2 * 16) + up(T * 4)
    d.max_blocks_per_seq = 32            # one partition: no partials
    assert pa.pa_chunk_workspace_bytes(d, T, 5) == 256 + up(S * 16) + up(T * 4)
    assert pa.pa_chunk_workspace_bytes(d, T, 0) == 0          # max_query_len < 1
    assert pa.pa_chunk_workspace_bytes(d, -1, 5) == 0
    d.kv_dtype = pa.PA_F32                                      # tensor-core path only
    assert pa.pa_chunk_workspace_bytes(d, T, 5) == 0


def test_chunk_automatic_partition(pa):
    # partition_size 0: decode takes 512 tokens at W = S * Hkv / 4 >= 256 work
    # items per partition; chunk attention takes four times that, at most 2048
    def up(x):
        return (x + 255) // 256 * 256

    S, Hq, Hkv, D, T = 256, 32, 8, 128, 1280
    d = pa.make_dims(num_seqs=S, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=16,
                     num_blocks=1000, max_blocks_per_seq=256, partition_size=0, kv_dtype="bf16")
    P = (256 * 16 + 2047) // 2048
    assert pa.pa_chunk_workspace_bytes(d, T, 5) == 256 + up(S * P * 16) + up(T * 4) + \
        up(T * Hq * P * D * 4) + up(T * Hq * P * 2 * 4)
    d.num_seqs = 16                      # W = 32: decode 256, chunk 1024
    P = (256 * 16 + 1023) // 1024
    assert pa.pa_chunk_workspace_bytes(d, 80, 5) == 256 + up(16 * P * 16) + up(80 * 4) + \
        up(80 * Hq * P * D * 4) + up(80 * Hq * P * 2 * 4)


def test_chunk_rejects_bad_arguments_on_the_host(pa):
    def status(T=4, max_q=2, ws=None, ws_bytes=0, **over):
        kw = dict(num_seqs=2, num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16, num_blocks=8,
                  max_blocks_per_seq=4, partition_size=0, kv_dtype="bf16")
        kw.update(over)
        d = pa.make_dims(**kw)
        fake = ctypes.c_void_p(0x10000)
        return pa.lib.pa_chunk_attention(ctypes.byref(d), fake, fake, fake, fake, fake, fake, T, max_q, 1.0,
                                         fake, ws, ws_bytes, None)
    assert status(kv_dtype="f32") == pa.PA_ERR_UNSUPPORTED
    assert status(head_dim=96) == pa.PA_ERR_UNSUPPORTED
    assert status(num_q_heads=7) == pa.PA_ERR_INVALID
    assert status(max_q=0) == pa.PA_ERR_INVALID
    assert status(T=-3) == pa.PA_ERR_INVALID
    assert status() == pa.PA_ERR_INVALID                        # no workspace
    assert status(T=0) == pa.PA_OK                              # nothing to do
    assert status(num_seqs=0) == pa.PA_OK


def test_step_graph_refuses_overlapping_layers_on_the_host(pa):
    # with several layers every stride must cover one layer's tensor; these are
    # refused before any CUDA call
    S, Hq, Hkv, D, B, N, T = 4, 8, 2, 128, 16, 10, 4
    d = pa.make_dims(num_seqs=S, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=B, num_blocks=N,
                     max_blocks_per_seq=4, kv_dtype="bf16")
    pool, qb, kvb, ob = N * Hkv * B * D * 2, S * Hq * D * 2, T * Hkv * D * 2, S * Hq * D * 4
    fake = ctypes.c_void_p(0x10000)

    def status(cache=pool, q=qb, kv=kvb, out=ob, layers=2):
        st = ctypes.c_int32(-1)
        g = pa.lib.pa_step_graph_create(ctypes.byref(d), layers, fake, fake, cache, fake, q, fake, fake, kv, fake,
                                        T, fake, fake, 1.0, fake, out, fake, 1 << 20, ctypes.byref(st))
        assert g is None
        return st.value
    for over in (dict(cache=pool - 16), dict(q=qb - 2), dict(kv=kvb - 2), dict(out=ob - 16), dict(layers=0)):
        assert status(**over) == pa.PA_ERR_INVALID, over
    # strides of exactly one layer pass the check; without a GPU the call then fails
    # at its first CUDA call (with one it would capture a graph of these fake pointers)
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        assert status() == pa.PA_ERR_CUDA


def test_build_switch_of_the_cuda_core_comparison(monkeypatch):
    # PA_DECODE_CUDA_CORE=1 builds the 16-bit decode with CUDA-core arithmetic
    # (for comparing it with the tensor-core kernel); unset or 0 is the default build
    from paged_kv_cache_127_gb300 import build
    monkeypatch.delenv("PA_DECODE_CUDA_CORE", raising=False)
    assert build._switches() == []
    monkeypatch.setenv("PA_DECODE_CUDA_CORE", "0")
    assert build._switches() == []
    monkeypatch.setenv("PA_DECODE_CUDA_CORE", "1")
    assert build._switches() == ["-DPA_DECODE_CUDA_CORE=1"]


def test_host_device_copy_calls_refuse_bad_arguments(pa):
    # checked on the host before any copy: null pointers with bytes > 0, and
    # nothing to do for zero bytes
    fake = ctypes.c_void_p(0x10000)
    assert pa.lib.pa_copy_to_device(None, fake, 16, None) == pa.PA_ERR_INVALID
    assert pa.lib.pa_copy_to_host(fake, None, 16, None) == pa.PA_ERR_INVALID
    assert pa.lib.pa_copy_to_device(None, None, 0, None) == pa.PA_OK
    assert pa.lib.pa_copy_to_host(None, None, 0, None) == pa.PA_OK
    torch = pytest.importorskip("torch")
    with pytest.raises(ValueError):     # the binding wants one host and one CUDA tensor
        pa.pa_copy_to_device(torch.empty(4), torch.empty(4))


def test_layer_copies_refuse_more_layers_than_one_launch_covers(pa):
    # one launch moves K and V of every layer: its grid has 2 * num_layers rows,
    # at most 65535, so 32768 layers are refused on the host (not left to fail
    # at launch); refused before any pointer is used
    d = pa.make_dims(num_seqs=1, num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16, num_blocks=10,
                     max_blocks_per_seq=4, kv_dtype="bf16")
    fake = ctypes.c_void_p(0x10000)
    pool = 10 * 2 * 16 * 128 * 2
    for layers in (32768, 1 << 30):
        assert pa.lib.pa_copy_blocks_layers(ctypes.byref(d), fake, fake, layers, pool, fake, 1, None) == \
            pa.PA_ERR_INVALID
        assert pa.lib.pa_swap_blocks(ctypes.byref(d), fake, fake, fake, fake, 10, layers, pool, pool, fake, 1,
                                     pa.PA_SWAP_OUT, None) == pa.PA_ERR_INVALID
