"""Thin ctypes binding over libpa.so, with the names of the C ABI (include/pa.h).

Argument marshalling only: every GPU step runs in the library's CUDA kernels.
The GPU calls take torch CUDA tensors (PyTorch supplies device memory and
streams) and check their shapes, dtypes, devices and contiguity against the
``pa_dims`` they are given, because the C ABI itself sees only pointers.
Importing this module fails with ImportError when the library has not been
built -- there is no fallback path.
"""
from __future__ import annotations

import contextlib
import ctypes
import os

import numpy as np

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libpa.so")

PA_OK, PA_ERR_INVALID, PA_ERR_UNSUPPORTED, PA_ERR_OOM, PA_ERR_BAD_INDEX, PA_ERR_CUDA, PA_ERR_TOO_LARGE = range(7)
PA_NOALLOC_SCRATCH_BYTES = 64 << 20
PA_F32, PA_F16, PA_BF16 = 0, 1, 2
DTYPE_CODES = {"f32": PA_F32, "f16": PA_F16, "bf16": PA_BF16}
STATUS_NAMES = {0: "PA_OK", 1: "PA_ERR_INVALID", 2: "PA_ERR_UNSUPPORTED", 3: "PA_ERR_OOM",
                4: "PA_ERR_BAD_INDEX", 5: "PA_ERR_CUDA", 6: "PA_ERR_TOO_LARGE"}
PA_SWAP_OUT, PA_SWAP_IN = 0, 1
PA_DEVERR_BAD_BLOCK, PA_DEVERR_BAD_LEN, PA_DEVERR_BAD_SLOT, PA_DEVERR_BAD_PAIR, PA_DEVERR_TIMEOUT = (
    1, 2, 4, 8, 16)


class PaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


class pa_dims(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("partition_size", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32)]


class pa_pool_stats(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("free_blocks", ctypes.c_int32), ("used_blocks", ctypes.c_int32),
                ("shared_blocks", ctypes.c_int32), ("live_seqs", ctypes.c_int32),
                ("cow_copies", ctypes.c_int64), ("tokens", ctypes.c_int64),
                ("table_slots", ctypes.c_int64), ("padded_slots", ctypes.c_int64)]


_vp, _i32, _i64, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
_SIGNATURES = {
    "pa_decode_workspace_bytes": (_sz, [_vp]),
    "pa_decode": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _sz, _vp]),
    "pa_decode_noalloc": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp]),
    "pa_chunk_workspace_bytes": (_sz, [_vp, _i32, _i32]),
    "pa_chunk_attention": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, ctypes.c_float, _vp, _vp, _sz,
                                  _vp]),
    "pa_write_kv": (_i32, [_vp, _vp, _vp, _vp, _i32, _vp, _vp, _vp]),
    "pa_copy_blocks": (_i32, [_vp, _vp, _vp, _vp, _i32, _vp]),
    "pa_copy_blocks_layers": (_i32, [_vp, _vp, _vp, _i32, _i64, _vp, _i32, _vp]),
    "pa_step_graph_create": (_vp, [_vp, _i32, _vp, _vp, _i64, _vp, _i64, _vp, _vp, _i64, _vp, _i32, _vp, _vp,
                                   ctypes.c_float, _vp, _i64, _vp, _sz, _vp]),
    "pa_step_graph_launch": (_i32, [_vp, _vp]),
    "pa_step_graph_destroy": (None, [_vp]),
    "pa_device_errors": (_i32, [_vp, _i32]),
    "pa_copy_to_device": (_i32, [_vp, _vp, _sz, _vp]),
    "pa_copy_to_host": (_i32, [_vp, _vp, _sz, _vp]),
    "pa_version": (ctypes.c_char_p, []),
    "pa_selftest_bounded_wait": (_i32, [ctypes.c_uint32, _vp, _vp]),
    "pa_pool_create": (_vp, [_i32, _i32, _vp]),
    "pa_pool_destroy": (None, [_vp]),
    "pa_seq_create": (_i32, [_vp]),
    "pa_seq_fork": (_i32, [_vp, _i32]),
    "pa_seq_append": (_i32, [_vp, _i32, _i32, _vp, _vp, _vp]),
    "pa_seq_append_batch": (_i32, [_vp, _vp, _i32, _i32, _vp, _vp, _vp]),
    "pa_seq_free": (_i32, [_vp, _i32]),
    "pa_seq_table": (_i32, [_vp, _i32, _vp, _i32]),
    "pa_seq_len": (_i32, [_vp, _i32]),
    "pa_pool_export": (_i32, [_vp, _vp, _i32, _i32, _i32, _vp, _vp]),
    "pa_pool_num_free": (_i32, [_vp]),
    "pa_block_refcount": (_i32, [_vp, _i32]),
    "pa_pool_get_stats": (_i32, [_vp, _vp]),
    "pa_pool_set_fail_after": (_i32, [_vp, _i32]),
    "pa_copy_pairs_check": (_i32, [_vp, _i32, _i32]),
    "pa_swap_blocks": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i64, _i64, _vp, _i32, _i32, _vp]),
    "pa_seq_swap_out": (_i32, [_vp, _vp, _i32, _vp, _vp, _vp]),
    "pa_seq_swap_in": (_i32, [_vp, _vp, _i32, _vp, _vp, _vp]),
    "pa_prefix_cache_create": (_vp, [_vp]),
    "pa_prefix_cache_destroy": (None, [_vp]),
    "pa_prefix_match": (_i32, [_vp, _vp, _i32, _vp, _i32]),
    "pa_prefix_insert": (_i32, [_vp, _vp, _i32, _vp, _i32]),
    "pa_prefix_evict": (_i32, [_vp, _i32]),
    "pa_prefix_cached_blocks": (_i32, [_vp]),
    "pa_seq_create_from_prefix": (_i32, [_vp, _vp, _i32]),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run `python -m paged_kv_cache_127_gb300.build` "
                          "(or __graft_entry__.build()) first -- there is no non-CUDA fallback")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def _check(status: int, what: str) -> None:
    if status != PA_OK:
        raise PaError(status, what)


def _np_ptr(a: np.ndarray) -> int:
    # the address as a plain int (c_void_p argument); the caller keeps `a` alive over the call
    return a.ctypes.data


def make_dims(num_seqs=0, num_q_heads=1, num_kv_heads=1, head_dim=128, block_size=16, num_blocks=1,
              max_blocks_per_seq=1, partition_size=0, kv_dtype="bf16") -> pa_dims:
    code = DTYPE_CODES[kv_dtype] if isinstance(kv_dtype, str) else int(kv_dtype)
    return pa_dims(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                   max_blocks_per_seq, partition_size, code)


# ------------------------------------------------------------------ GPU calls
def _torch():
    import torch
    return torch


def _torch_dtype(code: int):
    t = _torch()
    return {PA_F32: t.float32, PA_F16: t.float16, PA_BF16: t.bfloat16}[code]


def _expect(t, name, shape, dtype, device):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _on(device):
    """Make `device` current for one library call: the library keeps its
    per-device state (error word, fixed scratch, tensor-map cache) for the
    current device, and every pointer and the stream of a call must belong to it."""
    t = _torch()
    if t.cuda.current_device() == device.index:
        return contextlib.nullcontext()
    return t.cuda.device(device)


def _stream_ptr(stream, device):
    t = _torch()
    s = t.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


class Prepared:
    """One library call whose arguments were checked and marshalled once, issued
    again on every call(): for loops that repeat a call on the same buffers and
    stream (a serving step, a benchmark), where re-checking tensors each time
    would cost more host time than the kernel takes.  Holds references to the
    tensors it was prepared with; refresh their contents in place."""

    __slots__ = ("fn", "args", "what", "device", "keep")

    def __init__(self, fn, args, what, device, keep):
        self.fn, self.args, self.what, self.device, self.keep = fn, args, what, device, keep

    def __call__(self) -> None:
        with _on(self.device):
            st = self.fn(*self.args)
        _check(st, self.what)


def _issue(fn, args, what, device, prepare, keep):
    if prepare:
        return Prepared(fn, args, what, device, keep)
    with _on(device):
        st = fn(*args)
    _check(st, what)
    return None


def pa_decode_workspace_bytes(dims: pa_dims) -> int:
    return int(lib.pa_decode_workspace_bytes(ctypes.byref(dims)))


def pa_decode(dims: pa_dims, q, k_cache, v_cache, block_tables, context_lens, scale: float, out,
              workspace=None, stream=None, prepare: bool = False):
    """out[s, h] = softmax(scale * q[s, h] . K_s^T) . V_s over each sequence's paged context.
    With prepare=True nothing runs: the checked call is returned as a Prepared."""
    t = _torch()
    d, kv = dims, _torch_dtype(dims.kv_dtype)
    dev = q.device
    _expect(q, "q", (d.num_seqs, d.num_q_heads, d.head_dim), kv, dev)
    cache_shape = (d.num_blocks, d.num_kv_heads, d.block_size, d.head_dim)
    _expect(k_cache, "k_cache", cache_shape, kv, dev)
    _expect(v_cache, "v_cache", cache_shape, kv, dev)
    _expect(block_tables, "block_tables", (d.num_seqs, d.max_blocks_per_seq), t.int32, dev)
    _expect(context_lens, "context_lens", (d.num_seqs,), t.int32, dev)
    _expect(out, "out", (d.num_seqs, d.num_q_heads, d.head_dim), t.float32, dev)
    need = pa_decode_workspace_bytes(dims)
    ws_ptr, ws_bytes = None, 0
    if need:
        if workspace is None:
            raise ValueError(f"pa_decode needs a workspace of {need} bytes")
        if not workspace.is_cuda or not workspace.is_contiguous() or workspace.device != dev:
            raise ValueError("workspace must be a contiguous CUDA tensor on the same device")
        ws_bytes = workspace.numel() * workspace.element_size()
        ws_ptr = ctypes.c_void_p(workspace.data_ptr())
    args = (ctypes.byref(dims), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
            context_lens.data_ptr(), float(scale), out.data_ptr(), ws_ptr, ws_bytes, _stream_ptr(stream, dev))
    return _issue(lib.pa_decode, args, "pa_decode", dev, prepare,
                  (dims, q, k_cache, v_cache, block_tables, context_lens, out, workspace))


def pa_decode_noalloc(dims: pa_dims, q, k_cache, v_cache, block_tables, context_lens, scale: float, out,
                      stream=None) -> None:
    """pa_decode without a caller workspace, for callers that cannot allocate device memory.

    The scratch is a fixed PA_NOALLOC_SCRATCH_BYTES buffer inside the library,
    shared by every call: calls whose GPU work overlaps race on it, so keep them
    on one stream.  The first call on a device looks the buffer up; make it
    before any stream capture.  Raises PaError(PA_ERR_TOO_LARGE) when the
    problem needs more scratch than that buffer holds.
    """
    t = _torch()
    d, kv = dims, _torch_dtype(dims.kv_dtype)
    dev = q.device
    _expect(q, "q", (d.num_seqs, d.num_q_heads, d.head_dim), kv, dev)
    cache_shape = (d.num_blocks, d.num_kv_heads, d.block_size, d.head_dim)
    _expect(k_cache, "k_cache", cache_shape, kv, dev)
    _expect(v_cache, "v_cache", cache_shape, kv, dev)
    _expect(block_tables, "block_tables", (d.num_seqs, d.max_blocks_per_seq), t.int32, dev)
    _expect(context_lens, "context_lens", (d.num_seqs,), t.int32, dev)
    _expect(out, "out", (d.num_seqs, d.num_q_heads, d.head_dim), t.float32, dev)
    with _on(dev):
        st = lib.pa_decode_noalloc(ctypes.byref(dims), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                   block_tables.data_ptr(), context_lens.data_ptr(), float(scale), out.data_ptr(),
                                   _stream_ptr(stream, dev))
    _check(st, "pa_decode_noalloc")


def pa_chunk_workspace_bytes(dims: pa_dims, num_tokens: int, max_query_len: int) -> int:
    return int(lib.pa_chunk_workspace_bytes(ctypes.byref(dims), int(num_tokens), int(max_query_len)))


def pa_chunk_attention(dims: pa_dims, q, k_cache, v_cache, block_tables, context_lens, query_start, scale: float,
                       out, max_query_len: int, workspace=None, stream=None, prepare: bool = False):
    """Causal paged attention for the last n_s = query_start[s+1] - query_start[s]
    tokens of each sequence: the query at position pos sees keys 0..pos.
    With prepare=True nothing runs: the checked call is returned as a Prepared."""
    t = _torch()
    d, kv = dims, _torch_dtype(dims.kv_dtype)
    dev = q.device
    T = q.shape[0]
    _expect(q, "q", (T, d.num_q_heads, d.head_dim), kv, dev)
    cache_shape = (d.num_blocks, d.num_kv_heads, d.block_size, d.head_dim)
    _expect(k_cache, "k_cache", cache_shape, kv, dev)
    _expect(v_cache, "v_cache", cache_shape, kv, dev)
    _expect(block_tables, "block_tables", (d.num_seqs, d.max_blocks_per_seq), t.int32, dev)
    _expect(context_lens, "context_lens", (d.num_seqs,), t.int32, dev)
    _expect(query_start, "query_start", (d.num_seqs + 1,), t.int32, dev)
    _expect(out, "out", (T, d.num_q_heads, d.head_dim), t.float32, dev)
    need = pa_chunk_workspace_bytes(dims, T, max_query_len)
    ws_ptr, ws_bytes = None, 0
    if need:
        if workspace is None:
            raise ValueError(f"pa_chunk_attention needs a workspace of {need} bytes")
        if not workspace.is_cuda or not workspace.is_contiguous() or workspace.device != dev:
            raise ValueError("workspace must be a contiguous CUDA tensor on the same device")
        ws_bytes = workspace.numel() * workspace.element_size()
        ws_ptr = ctypes.c_void_p(workspace.data_ptr())
    args = (ctypes.byref(dims), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
            context_lens.data_ptr(), query_start.data_ptr(), T, int(max_query_len), float(scale), out.data_ptr(),
            ws_ptr, ws_bytes, _stream_ptr(stream, dev))
    return _issue(lib.pa_chunk_attention, args, "pa_chunk_attention", dev, prepare,
                  (dims, q, k_cache, v_cache, block_tables, context_lens, query_start, out, workspace))


def pa_write_kv(dims: pa_dims, k, v, slot_mapping, k_cache, v_cache, stream=None, prepare: bool = False):
    """k_cache[slot // B, h, slot % B] = k[t, h] (and v) for every slot >= 0.
    With prepare=True nothing runs: the checked call is returned as a Prepared."""
    t = _torch()
    d, kv = dims, _torch_dtype(dims.kv_dtype)
    dev = k.device
    T = int(slot_mapping.shape[0])
    _expect(k, "k", (T, d.num_kv_heads, d.head_dim), kv, dev)
    _expect(v, "v", (T, d.num_kv_heads, d.head_dim), kv, dev)
    _expect(slot_mapping, "slot_mapping", (T,), t.int64, dev)
    cache_shape = (d.num_blocks, d.num_kv_heads, d.block_size, d.head_dim)
    _expect(k_cache, "k_cache", cache_shape, kv, dev)
    _expect(v_cache, "v_cache", cache_shape, kv, dev)
    args = (ctypes.byref(dims), k.data_ptr(), v.data_ptr(), slot_mapping.data_ptr(), T, k_cache.data_ptr(),
            v_cache.data_ptr(), _stream_ptr(stream, dev))
    return _issue(lib.pa_write_kv, args, "pa_write_kv", dev, prepare, (dims, k, v, slot_mapping, k_cache, v_cache))


def pa_copy_blocks(dims: pa_dims, k_cache, v_cache, src_dst_pairs, stream=None, prepare: bool = False):
    """Copy whole blocks src -> dst in both caches for each row of src_dst_pairs [P, 2].
    With prepare=True nothing runs: the checked call is returned as a Prepared."""
    t = _torch()
    d, kv = dims, _torch_dtype(dims.kv_dtype)
    dev = k_cache.device
    P = int(src_dst_pairs.shape[0])
    cache_shape = (d.num_blocks, d.num_kv_heads, d.block_size, d.head_dim)
    _expect(k_cache, "k_cache", cache_shape, kv, dev)
    _expect(v_cache, "v_cache", cache_shape, kv, dev)
    _expect(src_dst_pairs, "src_dst_pairs", (P, 2), t.int64, dev)
    args = (ctypes.byref(dims), k_cache.data_ptr(), v_cache.data_ptr(), src_dst_pairs.data_ptr(), P,
            _stream_ptr(stream, dev))
    return _issue(lib.pa_copy_blocks, args, "pa_copy_blocks", dev, prepare, (dims, k_cache, v_cache, src_dst_pairs))


def pa_copy_blocks_layers(dims: pa_dims, k_caches, v_caches, src_dst_pairs, stream=None) -> None:
    """Copy whole blocks src -> dst in every layer of [L, N, Hkv, B, D] K and V pools."""
    t = _torch()
    d, kv = dims, _torch_dtype(dims.kv_dtype)
    dev = k_caches.device
    L = int(k_caches.shape[0])
    P = int(src_dst_pairs.shape[0])
    pool_shape = (L, d.num_blocks, d.num_kv_heads, d.block_size, d.head_dim)
    _expect(k_caches, "k_caches", pool_shape, kv, dev)
    _expect(v_caches, "v_caches", pool_shape, kv, dev)
    _expect(src_dst_pairs, "src_dst_pairs", (P, 2), t.int64, dev)
    stride = k_caches.stride(0) * k_caches.element_size()
    with _on(dev):
        st = lib.pa_copy_blocks_layers(ctypes.byref(dims), k_caches.data_ptr(), v_caches.data_ptr(), L, stride,
                                       src_dst_pairs.data_ptr(), P, _stream_ptr(stream, dev))
    _check(st, "pa_copy_blocks_layers")


class StepGraph:
    """pa_step_graph: one L-layer decode step (write_kv + decode per layer) as a CUDA graph.

    All tensors are kept referenced for the graph's lifetime; update their
    contents in place, then call launch().
      k_caches, v_caches  [L, N, Hkv, B, D]      q      [L, S, Hq, D]
      k_new, v_new        [L, T, Hkv, D]         out    [L, S, Hq, D] fp32
      slot_mapping int64 [T]; block_tables int32 [S, max_blocks]; context_lens int32 [S]
    """

    def __init__(self, dims: pa_dims, k_caches, v_caches, q, k_new, v_new, slot_mapping, block_tables,
                 context_lens, scale: float, out, workspace):
        t = _torch()
        d, kv = dims, _torch_dtype(dims.kv_dtype)
        dev = q.device
        L = int(q.shape[0])
        T = int(slot_mapping.shape[0])
        _expect(k_caches, "k_caches", (L, d.num_blocks, d.num_kv_heads, d.block_size, d.head_dim), kv, dev)
        _expect(v_caches, "v_caches", tuple(k_caches.shape), kv, dev)
        _expect(q, "q", (L, d.num_seqs, d.num_q_heads, d.head_dim), kv, dev)
        _expect(k_new, "k_new", (L, T, d.num_kv_heads, d.head_dim), kv, dev)
        _expect(v_new, "v_new", (L, T, d.num_kv_heads, d.head_dim), kv, dev)
        _expect(slot_mapping, "slot_mapping", (T,), t.int64, dev)
        _expect(block_tables, "block_tables", (d.num_seqs, d.max_blocks_per_seq), t.int32, dev)
        _expect(context_lens, "context_lens", (d.num_seqs,), t.int32, dev)
        _expect(out, "out", (L, d.num_seqs, d.num_q_heads, d.head_dim), t.float32, dev)
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor")
        self._keep = (dims, k_caches, v_caches, q, k_new, v_new, slot_mapping, block_tables, context_lens, out,
                      workspace)
        es = k_caches.element_size()
        status = ctypes.c_int32(0)
        with _on(dev):
            self.handle = lib.pa_step_graph_create(
                ctypes.byref(dims), L, k_caches.data_ptr(), v_caches.data_ptr(), k_caches.stride(0) * es,
                q.data_ptr(), q.stride(0) * es, k_new.data_ptr(), v_new.data_ptr(), k_new.stride(0) * es,
                slot_mapping.data_ptr(), T, block_tables.data_ptr(), context_lens.data_ptr(), float(scale),
                out.data_ptr(), out.stride(0) * 4, workspace.data_ptr(),
                workspace.numel() * workspace.element_size(), ctypes.byref(status))
        if not self.handle:
            raise PaError(status.value, "pa_step_graph_create")
        self.device = dev

    def launch(self, stream=None) -> None:
        with _on(self.device):
            _check(lib.pa_step_graph_launch(self.handle, _stream_ptr(stream, self.device)), "pa_step_graph_launch")

    def close(self) -> None:
        if self.handle:
            lib.pa_step_graph_destroy(self.handle)
            self.handle = None

    def __del__(self):
        self.close()


def pa_step_graph_create(dims: pa_dims, k_caches, v_caches, q, k_new, v_new, slot_mapping, block_tables,
                         context_lens, scale: float, out, workspace) -> "StepGraph":
    """Capture one L-layer decode step; returns the owning StepGraph."""
    return StepGraph(dims, k_caches, v_caches, q, k_new, v_new, slot_mapping, block_tables, context_lens,
                     scale, out, workspace)


def pa_step_graph_launch(graph: "StepGraph", stream=None) -> None:
    graph.launch(stream)


def pa_step_graph_destroy(graph: "StepGraph") -> None:
    graph.close()


def pa_swap_blocks(dims: pa_dims, k_cache, v_cache, host_k, host_v, pairs, direction: int, stream=None) -> None:
    """Move whole blocks device -> host (PA_SWAP_OUT) or host -> device (PA_SWAP_IN).

    Device caches [N, Hkv, B, D] or [L, N, Hkv, B, D]; host pools the same with
    their own block count, in pinned host memory (e.g. torch pin_memory=True)."""
    t = _torch()
    d, kv = dims, _torch_dtype(dims.kv_dtype)
    dev = k_cache.device
    layered = k_cache.dim() == 5
    L = int(k_cache.shape[0]) if layered else 1
    tail = (d.num_kv_heads, d.block_size, d.head_dim)
    _expect(k_cache, "k_cache", ((L,) if layered else ()) + (d.num_blocks,) + tail, kv, dev)
    _expect(v_cache, "v_cache", tuple(k_cache.shape), kv, dev)
    nh = int(host_k.shape[1] if layered else host_k.shape[0])
    for name, h in (("host_k", host_k), ("host_v", host_v)):
        if h.is_cuda or not h.is_pinned() or not h.is_contiguous() or h.dtype != kv:
            raise ValueError(f"{name} must be a contiguous pinned host tensor of the cache dtype")
        if tuple(h.shape) != ((L,) if layered else ()) + (nh,) + tail:
            raise ValueError(f"{name} has shape {tuple(h.shape)}")
    P = int(pairs.shape[0])
    _expect(pairs, "pairs", (P, 2), t.int64, dev)
    es = k_cache.element_size()
    dstride = k_cache.stride(0) * es if layered else 0
    hstride = host_k.stride(0) * es if layered else 0
    with _on(dev):
        _check(lib.pa_swap_blocks(ctypes.byref(dims), k_cache.data_ptr(), v_cache.data_ptr(), host_k.data_ptr(),
                                  host_v.data_ptr(), nh, L, dstride, hstride, pairs.data_ptr(), P, int(direction),
                                  _stream_ptr(stream, dev)), "pa_swap_blocks")


def _swap_seq(fn, dev_pool, host_pool, seq, name):
    # the sequence's table length bounds the pairs; ask the pool that owns it
    owner = dev_pool if name == "pa_seq_swap_out" else host_pool
    nb = lib.pa_seq_table(owner, seq, None, 0)
    if nb < 0:
        raise PaError(-nb, name)
    pairs = np.empty((max(nb, 1), 2), dtype=np.int64)
    out_id = ctypes.c_int32(0)
    npairs = ctypes.c_int32(0)
    _check(fn(dev_pool, host_pool, seq, ctypes.byref(out_id), _np_ptr(pairs), ctypes.byref(npairs)), name)
    return out_id.value, pairs[:npairs.value].copy()


def pa_seq_swap_out(dev_pool, host_pool, seq: int):
    """Returns (host sequence id, pairs int64 [n, 2] of (device block, host block))."""
    return _swap_seq(lib.pa_seq_swap_out, dev_pool, host_pool, seq, "pa_seq_swap_out")


def pa_seq_swap_in(dev_pool, host_pool, host_seq: int):
    """Returns (device sequence id, pairs int64 [n, 2] of (host block, device block))."""
    return _swap_seq(lib.pa_seq_swap_in, dev_pool, host_pool, host_seq, "pa_seq_swap_in")


def _host_device_pair(host, device, what):
    if host.is_cuda or not device.is_cuda:
        raise ValueError(f"{what}: expected one host tensor and one CUDA tensor")
    if not host.is_contiguous() or not device.is_contiguous():
        raise ValueError(f"{what}: tensors must be contiguous")
    nbytes = host.numel() * host.element_size()
    if device.numel() * device.element_size() != nbytes:
        raise ValueError(f"{what}: byte sizes differ")
    return nbytes


def pa_copy_to_device(dst, src, stream=None, prepare: bool = False):
    """Copy host tensor `src` into CUDA tensor `dst` (same byte size) on `stream`,
    asynchronously when `src` is pinned.  prepare=True returns a Prepared."""
    n = _host_device_pair(src, dst, "pa_copy_to_device")
    args = (dst.data_ptr(), src.data_ptr(), n, _stream_ptr(stream, dst.device))
    return _issue(lib.pa_copy_to_device, args, "pa_copy_to_device", dst.device, prepare, (dst, src))


def pa_copy_to_host(dst, src, stream=None, prepare: bool = False):
    """Copy CUDA tensor `src` into host tensor `dst` (same byte size) on `stream`,
    asynchronously when `dst` is pinned.  prepare=True returns a Prepared."""
    n = _host_device_pair(dst, src, "pa_copy_to_host")
    args = (dst.data_ptr(), src.data_ptr(), n, _stream_ptr(stream, src.device))
    return _issue(lib.pa_copy_to_host, args, "pa_copy_to_host", src.device, prepare, (dst, src))


def pa_device_errors(clear: bool = True) -> int:
    """The current device's sticky PA_DEVERR_* bits (see pa.h); `clear` resets them."""
    flags = ctypes.c_uint32(0)
    _check(lib.pa_device_errors(ctypes.byref(flags), 1 if clear else 0), "pa_device_errors")
    return int(flags.value)


def pa_version() -> str:
    return lib.pa_version().decode()


def pa_selftest_bounded_wait(limit, status, stream=None) -> None:
    """Run the kernels' bounded mbarrier wait on a barrier nothing arrives at;
    `status` (a one-element uint32/int32 CUDA tensor) receives PA_DEVERR_TIMEOUT
    when the wait gives up."""
    if status.numel() < 1 or status.element_size() != 4 or not status.is_cuda:
        raise ValueError("status must be a 4-byte CUDA tensor")
    with _on(status.device):
        rc = lib.pa_selftest_bounded_wait(int(limit), status.data_ptr(), _stream_ptr(stream, status.device))
    _check(rc, "pa_selftest_bounded_wait")


# ------------------------------------------------------------------ host allocator
def pa_pool_create(num_blocks: int, block_size: int, free_order=None) -> int:
    order = None
    if free_order is not None:
        order = np.ascontiguousarray(free_order, dtype=np.int32)
        if order.shape != (num_blocks,):
            raise ValueError("free_order must hold num_blocks ids")
    h = lib.pa_pool_create(num_blocks, block_size, None if order is None else _np_ptr(order))
    if not h:
        raise PaError(PA_ERR_INVALID, "pa_pool_create")
    return h


def pa_pool_destroy(pool) -> None:
    lib.pa_pool_destroy(pool)


def pa_seq_create(pool) -> int:
    r = lib.pa_seq_create(pool)
    if r < 0:
        raise PaError(-r, "pa_seq_create")
    return r


def pa_seq_fork(pool, parent: int) -> int:
    r = lib.pa_seq_fork(pool, parent)
    if r < 0:
        raise PaError(-r, "pa_seq_fork")
    return r


def pa_seq_append(pool, seq: int, n_tokens: int):
    """Returns (slots int64[n_tokens], cow_pairs int64[k, 2]) with k in {0, 1}."""
    slots = np.empty(max(n_tokens, 1), dtype=np.int64)
    pair = np.empty(2, dtype=np.int64)
    ncow = ctypes.c_int32(0)
    _check(lib.pa_seq_append(pool, seq, n_tokens, _np_ptr(slots), _np_ptr(pair), ctypes.byref(ncow)),
           "pa_seq_append")
    return slots[:n_tokens], pair.reshape(1, 2)[:ncow.value]


def pa_seq_append_batch(pool, seqs, tokens_each: int):
    """Returns (slots int64[n, tokens_each], cow_pairs int64[k, 2])."""
    seqs = np.ascontiguousarray(seqs, dtype=np.int32)
    n = seqs.shape[0]
    slots = np.empty((max(n, 1), max(tokens_each, 1)), dtype=np.int64)
    pairs = np.empty((max(n, 1), 2), dtype=np.int64)
    ncow = ctypes.c_int32(0)
    _check(lib.pa_seq_append_batch(pool, _np_ptr(seqs), n, tokens_each, _np_ptr(slots), _np_ptr(pairs),
                                   ctypes.byref(ncow)), "pa_seq_append_batch")
    return slots[:n, :tokens_each].copy(), pairs[:ncow.value].copy()


def pa_seq_free(pool, seq: int) -> None:
    _check(lib.pa_seq_free(pool, seq), "pa_seq_free")


def pa_seq_table(pool, seq: int) -> np.ndarray:
    n = lib.pa_seq_table(pool, seq, None, 0)
    if n < 0:
        raise PaError(-n, "pa_seq_table")
    out = np.empty(max(n, 1), dtype=np.int32)
    lib.pa_seq_table(pool, seq, _np_ptr(out), n)
    return out[:n]


def pa_seq_len(pool, seq: int) -> int:
    r = lib.pa_seq_len(pool, seq)
    if r < 0:
        raise PaError(-r, "pa_seq_len")
    return r


def pa_pool_export(pool, seqs, max_blocks: int, pad: int = -1):
    """Returns (tables int32[n, max_blocks], lens int32[n]) for the given sequences."""
    seqs = np.ascontiguousarray(seqs, dtype=np.int32)
    n = seqs.shape[0]
    tables = np.empty((max(n, 1), max_blocks), dtype=np.int32)
    lens = np.empty(max(n, 1), dtype=np.int32)
    _check(lib.pa_pool_export(pool, _np_ptr(seqs), n, max_blocks, pad, _np_ptr(tables), _np_ptr(lens)),
           "pa_pool_export")
    return tables[:n].copy(), lens[:n].copy()


def pa_pool_num_free(pool) -> int:
    return int(lib.pa_pool_num_free(pool))


def pa_block_refcount(pool, block: int) -> int:
    r = lib.pa_block_refcount(pool, block)
    if r < 0:
        raise PaError(-r, "pa_block_refcount")
    return r


def pa_pool_get_stats(pool) -> dict:
    st = pa_pool_stats()
    _check(lib.pa_pool_get_stats(pool, ctypes.byref(st)), "pa_pool_get_stats")
    return {name: getattr(st, name) for name, _ in pa_pool_stats._fields_}


def pa_pool_set_fail_after(pool, n) -> None:
    _check(lib.pa_pool_set_fail_after(pool, -1 if n is None else int(n)), "pa_pool_set_fail_after")


def pa_copy_pairs_check(pairs, num_blocks: int) -> None:
    """Raise PaError unless the host (src, dst) pairs are a valid copy-on-write list."""
    pairs = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
    _check(lib.pa_copy_pairs_check(_np_ptr(pairs) if pairs.size else None, pairs.shape[0], num_blocks),
           "pa_copy_pairs_check")


def _neg(r: int, what: str) -> int:
    if r < 0:
        raise PaError(-r, what)
    return r


def pa_prefix_cache_create(pool) -> int:
    h = lib.pa_prefix_cache_create(pool)
    if not h:
        raise PaError(PA_ERR_INVALID, "pa_prefix_cache_create")
    return h


def pa_prefix_cache_destroy(cache) -> None:
    lib.pa_prefix_cache_destroy(cache)


def pa_prefix_match(cache, tokens) -> np.ndarray:
    """Blocks (int32) of the longest cached block-aligned prefix of `tokens`."""
    t = np.ascontiguousarray(tokens, dtype=np.int32)
    cap = max(1, t.shape[0])
    out = np.empty(cap, dtype=np.int32)
    n = _neg(lib.pa_prefix_match(cache, _np_ptr(t), t.shape[0], _np_ptr(out), cap), "pa_prefix_match")
    return out[:n].copy()


def pa_prefix_insert(cache, tokens, blocks) -> int:
    t = np.ascontiguousarray(tokens, dtype=np.int32)
    b = np.ascontiguousarray(blocks, dtype=np.int32)
    return _neg(lib.pa_prefix_insert(cache, _np_ptr(t), t.shape[0], _np_ptr(b), b.shape[0]), "pa_prefix_insert")


def pa_prefix_evict(cache, n_blocks: int) -> int:
    return _neg(lib.pa_prefix_evict(cache, int(n_blocks)), "pa_prefix_evict")


def pa_prefix_cached_blocks(cache) -> int:
    return _neg(lib.pa_prefix_cached_blocks(cache), "pa_prefix_cached_blocks")


def pa_seq_create_from_prefix(pool, blocks) -> int:
    b = np.ascontiguousarray(blocks, dtype=np.int32)
    return _neg(lib.pa_seq_create_from_prefix(pool, _np_ptr(b), b.shape[0]), "pa_seq_create_from_prefix")


class Pool:
    """Owning wrapper: ``with Pool(n, B) as p: ...`` destroys the pool on exit."""

    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        self.handle = pa_pool_create(num_blocks, block_size, free_order)
        self.block_size = block_size
        self.num_blocks = num_blocks

    def close(self):
        if self.handle:
            pa_pool_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        self.close()
