"""CPU oracle for paged-KV decode attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library
(``paged_kv_cache_127_gb300``) shares no code with it and never calls it.

Contents
--------
* ``decode`` / ``decode_partitioned`` / ``chunk_attention`` / ``write_kv`` /
  ``copy_blocks`` / ``swap_blocks`` / ``slot_mapping``: ctypes wrappers over the
  fp64 C oracle in ``pa_oracle.c`` (plain definitions; see that file's header
  for the page citations).
* ``block_manager.BlockManager``: a plain Python model of the block manager
  (free list, reference counts, fork, growth, copy-on-write, swap).
* ``prefix_cache.PrefixCache``: a plain model of the block-level prefix cache.
* ``bookkeeping``: the pages' block-count and fragmentation arithmetic.

Array conventions: f32 data as ``np.float32``, f16 as ``np.float16``, bf16 as
``np.uint16`` holding the raw bfloat16 bits.  ``dtype`` is one of
``"f32"``, ``"f16"``, ``"bf16"``.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import build as _build

DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2}
_STORAGE = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}

_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(_build.build())
        i32, i64, dbl, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        lib.pa_oracle_decode.argtypes = [i32] * 8 + [vp] * 5 + [dbl, vp]
        lib.pa_oracle_decode_partitioned.argtypes = [i32] * 8 + [vp] * 5 + [dbl, i32, vp]
        lib.pa_oracle_write_kv.argtypes = [i32] * 6 + [vp] * 5
        lib.pa_oracle_copy_blocks.argtypes = [i32] * 5 + [vp] * 3 + [i32]
        lib.pa_oracle_slot_mapping.argtypes = [i32, vp, i32, i32, vp, vp, vp]
        lib.pa_oracle_slot.argtypes = [vp, i32, i32, ctypes.POINTER(i64)]
        lib.pa_oracle_swap_blocks.argtypes = [i32] * 4 + [vp, vp, i32, vp, vp, i32, vp, i32]
        lib.pa_oracle_chunk_attention.argtypes = [i32] * 8 + [vp] * 6 + [i32, dbl, vp]
        for f in (lib.pa_oracle_decode, lib.pa_oracle_decode_partitioned, lib.pa_oracle_write_kv,
                  lib.pa_oracle_copy_blocks, lib.pa_oracle_slot_mapping, lib.pa_oracle_slot,
                  lib.pa_oracle_swap_blocks, lib.pa_oracle_chunk_attention):
            f.restype = i32
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(arr: np.ndarray, dtype: str, name: str) -> np.ndarray:
    want = _STORAGE[dtype]
    if arr.dtype != want:
        raise TypeError(f"{name}: expected {np.dtype(want)} storage for {dtype}, got {arr.dtype}")
    return np.ascontiguousarray(arr)


def _decode_args(q, k_cache, v_cache, tables, lens, dtype):
    q = _check(q, dtype, "q")
    k_cache = _check(k_cache, dtype, "k_cache")
    v_cache = _check(v_cache, dtype, "v_cache")
    tables = np.ascontiguousarray(tables, dtype=np.int32)
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    S, Hq, D = q.shape
    N, Hkv, B, D2 = k_cache.shape
    if D2 != D or v_cache.shape != k_cache.shape or tables.shape[0] != S or lens.shape != (S,):
        raise ValueError("shape mismatch between q, caches, tables and lens")
    return q, k_cache, v_cache, tables, lens, (S, Hq, Hkv, D, B, N, tables.shape[1])


def decode(q, k_cache, v_cache, tables, lens, scale: float, dtype: str) -> np.ndarray:
    """fp64 softmax(scale * q K^T) V over each sequence's paged context; returns [S, Hq, D]."""
    q, k_cache, v_cache, tables, lens, (S, Hq, Hkv, D, B, N, mb) = _decode_args(
        q, k_cache, v_cache, tables, lens, dtype)
    out = np.zeros((S, Hq, D), dtype=np.float64)
    rc = _load().pa_oracle_decode(S, Hq, Hkv, D, B, N, mb, DTYPE_CODE[dtype], _ptr(q), _ptr(k_cache),
                                  _ptr(v_cache), _ptr(tables), _ptr(lens), float(scale), _ptr(out))
    if rc:
        raise ValueError(f"oracle decode rejected its inputs (rc={rc})")
    return out


def decode_partitioned(q, k_cache, v_cache, tables, lens, scale: float, dtype: str,
                       partition_size: int) -> np.ndarray:
    """Same result through per-partition (m_b, l_b, acc_b) and the log-sum-exp merge."""
    q, k_cache, v_cache, tables, lens, (S, Hq, Hkv, D, B, N, mb) = _decode_args(
        q, k_cache, v_cache, tables, lens, dtype)
    out = np.zeros((S, Hq, D), dtype=np.float64)
    rc = _load().pa_oracle_decode_partitioned(
        S, Hq, Hkv, D, B, N, mb, DTYPE_CODE[dtype], _ptr(q), _ptr(k_cache), _ptr(v_cache),
        _ptr(tables), _ptr(lens), float(scale), int(partition_size), _ptr(out))
    if rc:
        raise ValueError(f"oracle decode_partitioned rejected its inputs (rc={rc})")
    return out


def chunk_attention(q, k_cache, v_cache, tables, lens, query_start, scale: float, dtype: str) -> np.ndarray:
    """fp64 causal attention of each sequence's last n_s tokens over its paged
    context: q [T, Hq, D] with sequence s owning rows query_start[s]..query_start[s+1]-1;
    the query at position pos = lens[s] - n_s + t sees keys 0..pos.  Returns [T, Hq, D]."""
    q = _check(q, dtype, "q")
    k_cache = _check(k_cache, dtype, "k_cache")
    v_cache = _check(v_cache, dtype, "v_cache")
    tables = np.ascontiguousarray(tables, dtype=np.int32)
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    query_start = np.ascontiguousarray(query_start, dtype=np.int32)
    T, Hq, D = q.shape
    N, Hkv, B, D2 = k_cache.shape
    S = lens.shape[0]
    if D2 != D or v_cache.shape != k_cache.shape or tables.shape[0] != S or query_start.shape != (S + 1,):
        raise ValueError("shape mismatch between q, caches, tables, lens and query_start")
    out = np.zeros((T, Hq, D), dtype=np.float64)
    rc = _load().pa_oracle_chunk_attention(S, Hq, Hkv, D, B, N, tables.shape[1], DTYPE_CODE[dtype], _ptr(q),
                                           _ptr(k_cache), _ptr(v_cache), _ptr(tables), _ptr(lens),
                                           _ptr(query_start), T, float(scale), _ptr(out))
    if rc:
        raise ValueError(f"oracle chunk_attention rejected its inputs (rc={rc})")
    return out


def write_kv(k, v, slots, k_cache, v_cache, dtype: str) -> None:
    """In place: k_cache[slot // B, h, slot % B, :] = k[t, h, :] (and v); slot < 0 skipped."""
    k = _check(k, dtype, "k")
    v = _check(v, dtype, "v")
    for c in (k_cache, v_cache):
        if c.dtype != _STORAGE[dtype] or not c.flags.c_contiguous:
            raise TypeError("caches must be contiguous arrays of the storage dtype")
    slots = np.ascontiguousarray(slots, dtype=np.int64)
    T, Hkv, D = k.shape
    N, Hkv2, B, D2 = k_cache.shape
    if (Hkv2, D2) != (Hkv, D) or v.shape != k.shape or slots.shape != (T,):
        raise ValueError("shape mismatch")
    rc = _load().pa_oracle_write_kv(T, Hkv, D, B, N, DTYPE_CODE[dtype], _ptr(k), _ptr(v),
                                    _ptr(slots), _ptr(k_cache), _ptr(v_cache))
    if rc:
        raise ValueError("oracle write_kv: slot out of range")


def copy_blocks(k_cache, v_cache, pairs, dtype: str) -> None:
    """In place: for each (src, dst) pair copy the whole block src -> dst in both caches."""
    for c in (k_cache, v_cache):
        if c.dtype != _STORAGE[dtype] or not c.flags.c_contiguous:
            raise TypeError("caches must be contiguous arrays of the storage dtype")
    pairs = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
    N, Hkv, B, D = k_cache.shape
    rc = _load().pa_oracle_copy_blocks(Hkv, D, B, N, DTYPE_CODE[dtype], _ptr(k_cache),
                                       _ptr(v_cache), _ptr(pairs), pairs.shape[0])
    if rc:
        raise ValueError("oracle copy_blocks: block id out of range")


def swap_blocks(from_k, from_v, to_k, to_v, pairs, dtype: str) -> None:
    """In place: to[dst] = from[src] (whole blocks, K and V) for each (src, dst) pair."""
    for c in (from_k, from_v, to_k, to_v):
        if c.dtype != _STORAGE[dtype] or not c.flags.c_contiguous:
            raise TypeError("pools must be contiguous arrays of the storage dtype")
    pairs = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
    Nf, Hkv, B, D = from_k.shape
    Nt = to_k.shape[0]
    if to_k.shape[1:] != from_k.shape[1:] or from_v.shape != from_k.shape or to_v.shape != to_k.shape:
        raise ValueError("pool shapes differ")
    rc = _load().pa_oracle_swap_blocks(Hkv, D, B, DTYPE_CODE[dtype], _ptr(from_k), _ptr(from_v), Nf, _ptr(to_k),
                                       _ptr(to_v), Nt, _ptr(pairs), pairs.shape[0])
    if rc:
        raise ValueError("oracle swap_blocks: block id out of range")


def slot_mapping(tables, block_size: int, seq_of, positions) -> np.ndarray:
    """slot of (seq_of[t], positions[t]) through the block table; -1 where position < 0."""
    tables = np.ascontiguousarray(tables, dtype=np.int32)
    seq_of = np.ascontiguousarray(seq_of, dtype=np.int32)
    positions = np.ascontiguousarray(positions, dtype=np.int32)
    out = np.empty(positions.shape[0], dtype=np.int64)
    rc = _load().pa_oracle_slot_mapping(positions.shape[0], _ptr(tables), tables.shape[1],
                                        int(block_size), _ptr(seq_of), _ptr(positions), _ptr(out))
    if rc:
        raise ValueError("oracle slot_mapping: position beyond the table")
    return out


def slot(table_row, block_size: int, position: int) -> int:
    """slot (= physical block * B + offset) of one token position."""
    row = np.ascontiguousarray(table_row, dtype=np.int32)
    out = ctypes.c_int64()
    if _load().pa_oracle_slot(_ptr(row), int(block_size), int(position), ctypes.byref(out)):
        raise ValueError("bad position")
    return int(out.value)
