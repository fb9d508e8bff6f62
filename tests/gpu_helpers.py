"""Helpers for the GPU parity tests: moving storage arrays to and from torch."""
from __future__ import annotations

import numpy as np
import pytest

from paged_kv_cache_127_gb300 import synth


def require_gpu():
    """The library and a CUDA device, or fail loudly (a GPU test never falls back)."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_127_gb300 import build
    build.build()
    from paged_kv_cache_127_gb300 import binding   # ImportError here is a failure, not a skip
    binding.pa_device_errors(clear=True)
    return torch, binding


def torch_dtype(torch, dtype: str):
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]


def to_dev(torch, arr: np.ndarray, dtype: str | None = None, device="cuda"):
    """Storage array -> CUDA tensor (bf16 arrays hold raw bits as uint16)."""
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(arr)).to(device)


def to_host(t, dtype: str) -> np.ndarray:
    """CUDA tensor -> storage array (bf16 as uint16 bits)."""
    torch = __import__("torch")
    t = t.detach().cpu().contiguous()
    if dtype == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def run_decode(torch, pa, dtype, q, kc, vc, tables, lens, scale, partition_size=0):
    """Upload, call pa_decode through the C ABI, return the fp32 output on the host."""
    S, Hq, D = q.shape
    N, Hkv, B, _ = kc.shape
    dims = pa.make_dims(S, Hq, Hkv, D, B, N, tables.shape[1], partition_size, dtype)
    dq, dk, dv = to_dev(torch, q, dtype), to_dev(torch, kc, dtype), to_dev(torch, vc, dtype)
    dt = torch.from_numpy(np.ascontiguousarray(tables, dtype=np.int32)).cuda()
    dl = torch.from_numpy(np.ascontiguousarray(lens, dtype=np.int32)).cuda()
    out = torch.full((S, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    nbytes = pa.pa_decode_workspace_bytes(dims)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda") if nbytes else None
    pa.pa_decode(dims, dq, dk, dv, dt, dl, scale, out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64)


def poison_unused(kc, vc, tables, lens, B, dtype):
    """NaN in every slot no sequence's context covers (padding tails and free blocks)."""
    keep = np.zeros(kc.shape[0] * B, dtype=bool)
    for s, n in enumerate(lens):
        for j in range(-(-int(n) // B)):
            b = int(tables[s][j])
            keep[b * B: b * B + min(B, int(n) - j * B)] = True
    mask = np.broadcast_to(~keep.reshape(kc.shape[0], 1, B, 1), kc.shape)
    nan = synth.nan_value(dtype)
    kc[mask] = nan
    vc[mask] = nan
