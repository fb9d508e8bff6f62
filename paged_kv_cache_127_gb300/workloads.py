"""Assemble one decode step of a named workload (shapes and distributions in
``synth``), with the library's C++ allocator producing the block tables, the
new tokens' slots and the copy-on-write pairs.

A decode step is the whole hot path once:
  host:  append one token to every sequence (growth / copy-on-write decisions
         and slot mapping, in the allocator);
  GPU:   pa_copy_blocks(pairs) -> pa_write_kv(new K/V at the slots) ->
         pa_decode(q over every sequence's full context).
The step is idempotent (the same slots are rewritten with the same rows), so a
benchmark can repeat it.

Chunk workloads (``synth.CHUNK_WORKLOADS``) append query_len tokens to every
sequence instead of one; the GPU step is then pa_write_kv of all S * query_len
new rows followed by pa_chunk_attention over them (query_start = s * query_len).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import synth


@dataclass
class DecodeStep:
    name: str
    dtype: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    max_blocks: int
    partition_size: int
    scale: float
    free_order: np.ndarray     # the pool's initial free list
    tables: np.ndarray         # int32 [S, max_blocks] after the step's appends (pad -1)
    lens: np.ndarray           # int32 [S] context lengths including the new token(s)
    slots: np.ndarray          # int64 [S * query_len] slots of the new tokens, sequence-major
    pairs: np.ndarray          # int64 [P, 2] copy-on-write pairs of this step
    query_len: int = 1         # new (query) tokens per sequence
    q: np.ndarray | None = None
    k_new: np.ndarray | None = None
    v_new: np.ndarray | None = None
    k_cache: np.ndarray | None = None
    v_cache: np.ndarray | None = None

    @property
    def num_seqs(self) -> int:
        return int(self.lens.shape[0])

    def kv_bytes_per_token(self) -> int:
        """K and V bytes of one token of one layer: 2 * Hkv * D * sizeof(dtype)."""
        return 2 * self.num_kv_heads * self.head_dim * synth.ELEM_BYTES[self.dtype]

    def kv_bytes_logical(self) -> int:
        """KV bytes decode reads: every sequence's valid tokens (shared ones per sequence)."""
        return int(self.lens.astype(np.int64).sum()) * self.kv_bytes_per_token()

    def kv_bytes_unique(self) -> int:
        """KV bytes of distinct valid slots (a shared prefix counted once)."""
        seen = set()
        B = self.block_size
        total = 0
        for s in range(self.num_seqs):
            n = int(self.lens[s])
            for j in range(-(-n // B)):
                b = int(self.tables[s, j])
                if b not in seen:
                    seen.add(b)
                    total += min(B, n - j * B)
        return total * self.kv_bytes_per_token()

    @property
    def num_tokens(self) -> int:
        return self.num_seqs * self.query_len

    def query_start(self) -> np.ndarray:
        return (np.arange(self.num_seqs + 1) * self.query_len).astype(np.int32)

    def chunk_flops(self) -> int:
        """Attention FLOPs of a chunk step: 2 (q.k) + 2 (p.v) per head dimension,
        per query head, per visible key; the query at position pos sees pos + 1 keys."""
        n = self.query_len
        vis = (self.lens.astype(np.int64)[:, None] - n + np.arange(n)[None, :] + 1).sum()
        return int(4 * self.head_dim * self.num_q_heads * vis)

    def first(self, k: int) -> "DecodeStep":
        """The same step restricted to the first k sequences (pool unchanged)."""
        import copy
        sub = copy.copy(self)
        t = k * self.query_len
        sub.tables, sub.lens, sub.slots = self.tables[:k], self.lens[:k], self.slots[:t]
        if self.q is not None:
            sub.q, sub.k_new, sub.v_new = self.q[:t], self.k_new[:t], self.v_new[:t]
        return sub

    def dims(self, binding):
        return binding.make_dims(self.num_seqs, self.num_q_heads, self.num_kv_heads, self.head_dim,
                                 self.block_size, self.num_blocks, self.max_blocks, self.partition_size,
                                 self.dtype)


def _max_len(w: synth.Workload) -> int:
    if w.name == "tiny":
        return 64
    if w.name == "mha7b":
        return 2048
    if w.name.startswith("gqa8b") or w.name in synth.CHUNK_WORKLOADS:
        return 4096
    if w.name == "prefix_cow":
        return w.prefix_len + 512 + 16
    return 32768


def build_step(name: str, seed: int = 0, values: bool = True, binding=None) -> DecodeStep:
    """Run the allocator for one step of workload `name`; optionally draw the values."""
    if binding is None:
        from . import binding
    w = synth.workload(name, seed)
    rng = synth.make_rng(seed + 7919)
    B = w.block_size
    max_blocks = -(-_max_len(w) // B)

    if name == "prefix_cow":
        prefix_blocks = -(-w.prefix_len // B)
        need = prefix_blocks + int(synth.blocks_needed(w.lengths + 1, B).sum()) + 3 * w.pair_count
        N = int(np.ceil(w.pool_factor * need))
    elif w.fixed_pool:
        N = w.fixed_pool
    else:
        N = synth.pool_blocks(w.lengths, B, w.pool_factor)
    if w.fixed_tables:
        first = [b for t in w.fixed_tables for b in t]
        order = np.array(first + [b for b in range(N) if b not in first], dtype=np.int32)
    else:
        order = synth.free_order(rng, N)

    pool = binding.Pool(N, B, order)
    h = pool.handle
    seqs = []
    if name == "prefix_cow":
        root = binding.pa_seq_create(h)
        binding.pa_seq_append(h, root, w.prefix_len)
        for n in w.lengths:                       # 128 continuations of the 800-token prefix
            s = binding.pa_seq_fork(h, root)
            binding.pa_seq_append(h, s, int(n) - 1)
            seqs.append(s)
        binding.pa_seq_free(h, root)
        for _ in range(w.pair_count):             # pairs sharing one full + one 8-token block
            a = binding.pa_seq_create(h)
            binding.pa_seq_append(h, a, w.pair_prefix)
            seqs += [a, binding.pa_seq_fork(h, a)]
    else:
        for n in w.lengths:
            s = binding.pa_seq_create(h)
            binding.pa_seq_append(h, s, int(n) - w.query_len)   # the context already cached
            seqs.append(s)
    slots, pairs = binding.pa_seq_append_batch(h, seqs, w.query_len)   # this step's new tokens
    binding.pa_copy_pairs_check(pairs, N)   # pa_copy_blocks' precondition, on the host copy
    tables, lens = binding.pa_pool_export(h, seqs, max_blocks, -1)
    pool.close()

    step = DecodeStep(name=name, dtype=w.dtype, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                      head_dim=w.head_dim, block_size=B, num_blocks=N, max_blocks=max_blocks,
                      partition_size=w.partition_size, scale=w.scale, free_order=order, tables=tables,
                      lens=lens, slots=slots.reshape(-1).copy(), pairs=pairs, query_len=w.query_len)
    if values:
        T, Hq, Hkv, D = len(seqs) * w.query_len, w.num_q_heads, w.num_kv_heads, w.head_dim
        step.q = synth.normal(rng, (T, Hq, D), w.std * w.q_prescale, w.dtype)
        step.k_new = synth.normal(rng, (T, Hkv, D), w.std, w.dtype)
        step.v_new = synth.normal(rng, (T, Hkv, D), w.std, w.dtype)
        step.k_cache = synth.normal(rng, (N, Hkv, B, D), w.std, w.dtype)
        step.v_cache = synth.normal(rng, (N, Hkv, B, D), w.std, w.dtype)
    return step
