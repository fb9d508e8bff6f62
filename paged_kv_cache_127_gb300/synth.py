"""Seeded synthetic inputs for paged decode attention.

This module only draws random numbers and arranges them into the shapes the
workloads need: context lengths, random values in a storage dtype, random
placements of sequences' blocks in a pool, random slot sets and copy pairs.
It holds none of the attention arithmetic and none of the address translation,
so both the CUDA path and the CPU oracle can take their inputs from it.

Storage conventions (numpy): f32 -> ``float32``; f16 -> ``float16``;
bf16 -> ``uint16`` holding the raw bfloat16 bits (numpy has no bfloat16).

Workloads (shapes and distributions of the decode workloads the pages discuss:
a tiny worked example, a 7B-shaped multi-head layer, an 8B-shaped grouped-query
layer, a shared-prefix batch and a long-context 70B-shaped layer):

  tiny        Hq = Hkv = 4, D 64, f32, B 16, 64-block pool; lengths 25/47/12 with
              tables [3, 7], [0, 5, 9], [4]; q, K, V ~ N(0, 1); scale 1/8
  mha7b       Hq = Hkv = 32, D 128, f16, B 16; 64 sequences, lengths U{1..2048};
              pool 1.25x demand, placement a seeded permutation; N(0, 0.5^2);
              scale 1/sqrt(128)
  gqa8b_b16   Hq 32 over Hkv 8, D 128, bf16, B 16; 256 sequences, lognormal
  gqa8b_b32   lengths (median 600, sigma 0.8, clipped to [1, 4096]); shuffled
              placement in a 1.25x pool; N(0, 1) with q scaled by 1/sqrt(128) on
              the host and scale 1; fp32 output.  B 32 for the second sweep.
  prefix_cow  Hq 32 / Hkv 8, D 128, bf16, B 16; 128 sequences forked from one
              800-token prefix plus private suffixes U{1..512}; 32 pairs sharing
              a 24-token prefix whose next write forces a block copy; one new
              token per sequence per step
  verify8b    the gqa8b_b16 layer with 5 query tokens per sequence (4 drafted
              tokens + the last accepted one being verified): 256 sequences,
              cached context lognormal (median 600, sigma 0.8) + the 5 tokens
  prefill8b   the same layer, chunked prefill: 16 sequences each adding a
              512-token chunk to a cached context U{0..3584}
  long70b     Hq 64 / Hkv 8, D 128, bf16, B 16; 32 sequences, lengths
              U{8192..32768}; shuffled placement; partitions of 512 tokens;
              N(0, 1); scale 1/sqrt(128)
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

DTYPES = ("f32", "f16", "bf16")
STORAGE = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}


def make_rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


# ---------------------------------------------------------------- dtype helpers
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest even); return the bits.

    Works in 32-bit integers, a few million elements at a time: adding 0x7FFF
    plus the kept part's lowest bit can wrap around only for negative NaN
    payloads, and every NaN is replaced by the canonical quiet NaN afterwards."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    flat = x.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint16)
    step = 1 << 22
    for i in range(0, flat.size, step):
        part = flat[i:i + step]
        u = part.view(np.uint32)
        r = (u >> np.uint32(16)) & np.uint32(1)
        r += u
        r += np.uint32(0x7FFF)
        r >>= np.uint32(16)
        o = out[i:i + step]
        o[:] = r
        nan = np.isnan(part)
        if nan.any():
            o[nan] = 0x7FC0
    return out.reshape(x.shape)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def to_storage(x_f32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.ascontiguousarray(x_f32, dtype=np.float32)
    if dtype == "f16":
        return np.ascontiguousarray(x_f32.astype(np.float16))
    if dtype == "bf16":
        return f32_to_bf16_bits(x_f32)
    raise ValueError(dtype)


def storage_to_f32(a: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits_to_f32(a) if dtype == "bf16" else a.astype(np.float32)


def nan_value(dtype: str):
    """A NaN in the storage representation."""
    return {"f32": np.float32(np.nan), "f16": np.float16(np.nan), "bf16": np.uint16(0x7FC0)}[dtype]


def normal(rng: np.random.Generator, shape, std: float, dtype: str) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return to_storage(x, dtype)


# ---------------------------------------------------------------- lengths
def uniform_lengths(rng, n: int, lo: int, hi: int) -> np.ndarray:
    """n integers uniform in [lo, hi] inclusive."""
    return rng.integers(lo, hi + 1, size=n).astype(np.int32)


def lognormal_lengths(rng, n: int, median: float, sigma: float, lo: int, hi: int) -> np.ndarray:
    """round(median * exp(sigma * N(0, 1))) clipped to [lo, hi]."""
    x = np.rint(median * np.exp(sigma * rng.standard_normal(n)))
    return np.clip(x, lo, hi).astype(np.int32)


# ---------------------------------------------------------------- placements
def blocks_needed(lengths, block_size: int) -> np.ndarray:
    """Table length per sequence (input shape: ceil(len / B))."""
    lengths = np.asarray(lengths, dtype=np.int64)
    return ((lengths + block_size - 1) // block_size).astype(np.int32)


def pool_blocks(lengths, block_size: int, factor: float) -> int:
    return max(1, int(math.ceil(factor * int(blocks_needed(lengths, block_size).sum()))))


def scattered_tables(rng, lengths, block_size: int, num_blocks: int, shuffle: bool = True,
                     pad: int = -1, max_blocks: int | None = None):
    """Give each sequence distinct physical blocks drawn from a permutation of the pool.

    Returns (tables int32 [S, max_blocks] padded with `pad`, used-block mask).
    """
    nb = blocks_needed(lengths, block_size)
    total = int(nb.sum())
    if total > num_blocks:
        raise ValueError(f"pool of {num_blocks} blocks cannot hold {total}")
    ids = rng.permutation(num_blocks) if shuffle else np.arange(num_blocks)
    mb = int(max(1, nb.max() if len(nb) else 1)) if max_blocks is None else max_blocks
    tables = np.full((len(nb), mb), pad, dtype=np.int32)
    used = np.zeros(num_blocks, dtype=bool)
    cur = 0
    for s, n in enumerate(nb):
        tables[s, :n] = ids[cur:cur + n]
        used[ids[cur:cur + n]] = True
        cur += n
    return tables, used


def free_order(rng, num_blocks: int) -> np.ndarray:
    """A seeded permutation of block ids, for a pool's free list."""
    return rng.permutation(num_blocks).astype(np.int32)


def distinct_slots(rng, n: int, num_slots: int, frac_skip: float = 0.0) -> np.ndarray:
    """n distinct slot numbers in [0, num_slots); a fraction replaced by -1 (skip)."""
    s = rng.choice(num_slots, size=n, replace=False).astype(np.int64)
    if frac_skip > 0:
        s[rng.random(n) < frac_skip] = -1
    return s


def copy_pairs(rng, n: int, num_blocks: int) -> np.ndarray:
    """n (src, dst) block pairs; all dsts distinct and disjoint from all srcs."""
    ids = rng.permutation(num_blocks)
    if 2 * n > num_blocks:
        raise ValueError("pool too small for disjoint pairs")
    return np.stack([ids[:n], ids[n:2 * n]], axis=1).astype(np.int64)


def prefix_requests(rng, n: int, families: int = 8, family_median: float = 512, own_median: float = 90,
                    followup: float = 0.3, vocab: int = 32000, max_len: int = 8192) -> list:
    """n request token streams (int32 arrays) for prefix-cache workloads.

    Each request is one of `families` shared prompts (lengths lognormal around
    `family_median`; family i drawn with weight 1 / (i + 1)) followed by its
    own tokens (lognormal around `own_median`); a fraction `followup` instead
    continue one of the last 64 requests (its whole token list plus new own
    tokens), as a multi-turn conversation does.  Lengths are capped at max_len.
    """
    fam_len = lognormal_lengths(rng, families, family_median, 0.5, 16, max_len // 2)
    fams = [rng.integers(0, vocab, size=int(k), dtype=np.int32) for k in fam_len]
    w = 1.0 / np.arange(1, families + 1)
    w /= w.sum()
    out = []
    for _ in range(n):
        own = rng.integers(0, vocab, size=int(lognormal_lengths(rng, 1, own_median, 0.8, 1, 2048)[0]),
                           dtype=np.int32)
        if out and rng.random() < followup:
            base = out[-1 - int(rng.integers(0, min(64, len(out))))]
        else:
            base = fams[int(rng.choice(families, p=w))]
        out.append(np.concatenate([base, own])[:max_len])
    return out


# ---------------------------------------------------------------- workloads
@dataclass
class Workload:
    name: str
    dtype: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    partition_size: int
    scale: float
    std: float
    q_prescale: float = 1.0
    num_seqs: int = 0
    lengths: np.ndarray = field(default=None, repr=False)
    fixed_tables: list | None = field(default=None, repr=False)
    fixed_pool: int | None = None
    pool_factor: float = 1.25
    prefix_len: int = 0            # prefix_cow only
    prefix_group: int = 0
    pair_count: int = 0
    pair_prefix: int = 0
    query_len: int = 1             # query tokens per sequence per step (chunk workloads)


def workload(name: str, seed: int = 0) -> Workload:
    """Shapes and lengths of one named workload (values are drawn separately)."""
    rng = make_rng(seed)
    if name == "tiny":
        return Workload(name, "f32", 4, 4, 64, 16, 512, 1.0 / 8.0, 1.0, num_seqs=3,
                        lengths=np.array([25, 47, 12], dtype=np.int32),
                        fixed_tables=[[3, 7], [0, 5, 9], [4]], fixed_pool=64)
    if name == "mha7b":
        return Workload(name, "f16", 32, 32, 128, 16, 512, 1.0 / math.sqrt(128), 0.5,
                        num_seqs=64, lengths=uniform_lengths(rng, 64, 1, 2048))
    if name in ("gqa8b_b16", "gqa8b_b32"):
        B = 16 if name.endswith("16") else 32
        return Workload(name, "bf16", 32, 8, 128, B, 512, 1.0, 1.0,
                        q_prescale=1.0 / math.sqrt(128), num_seqs=256,
                        lengths=lognormal_lengths(rng, 256, 600, 0.8, 1, 4096))
    if name == "prefix_cow":
        suffix = uniform_lengths(rng, 128, 1, 512)
        return Workload(name, "bf16", 32, 8, 128, 16, 512, 1.0 / math.sqrt(128), 1.0,
                        num_seqs=128 + 64, lengths=suffix, prefix_len=800, prefix_group=128,
                        pair_count=32, pair_prefix=24)
    if name == "long70b":
        return Workload(name, "bf16", 64, 8, 128, 16, 512, 1.0 / math.sqrt(128), 1.0,
                        num_seqs=32, lengths=uniform_lengths(rng, 32, 8192, 32768))
    if name == "verify8b":
        ctx = lognormal_lengths(rng, 256, 600, 0.8, 1, 4096 - 5)
        # 2048-token partitions: what partition_size 0 picks for chunk attention at this batch
        return Workload(name, "bf16", 32, 8, 128, 16, 2048, 1.0, 1.0, q_prescale=1.0 / math.sqrt(128),
                        num_seqs=256, lengths=ctx + 5, query_len=5)
    if name == "prefill8b":
        ctx = uniform_lengths(rng, 16, 0, 4096 - 512)
        return Workload(name, "bf16", 32, 8, 128, 16, 512, 1.0, 1.0, q_prescale=1.0 / math.sqrt(128),
                        num_seqs=16, lengths=ctx + 512, query_len=512)
    raise KeyError(name)


WORKLOADS = ("tiny", "mha7b", "gqa8b_b16", "gqa8b_b32", "prefix_cow", "long70b")
CHUNK_WORKLOADS = ("verify8b", "prefill8b")
