"""Prefix reuse feeding chunk prefill: requests that share a prompt reuse the
cached prompt blocks (radix-tree prefix cache) and only their own tokens are
written and attended as a prefill chunk; the chunk's outputs must equal the
oracle's over the whole context."""
import numpy as np
import pytest

import oracle
from gpu_helpers import require_gpu, to_dev
from paged_helpers import assert_attention_close
from paged_kv_cache_127_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gpu():
    return require_gpu()


def test_cached_prompt_blocks_serve_a_suffix_prefill(gpu):
    torch, pa = gpu
    dtype, Hq, Hkv, D, B, N = "bf16", 8, 2, 128, 16, 256
    rng = synth.make_rng(71)
    pool = pa.Pool(N, B, synth.free_order(rng, N))
    cache = pa.pa_prefix_cache_create(pool.handle)
    # the K/V a token position holds is a function of the token prefix, so the
    # cache is consistent: draw rows per (prompt id, position)
    prompt = rng.integers(0, 1000, size=200).astype(np.int32)           # 12 full blocks + 8 tokens
    kc = np.zeros((N, Hkv, B, D), np.uint16)
    vc = np.zeros((N, Hkv, B, D), np.uint16)
    dkc, dvc = to_dev(torch, kc, dtype), to_dev(torch, vc, dtype)

    def admit(tokens):
        """Reuse the cached prefix, store the rest; returns (seq, reused tokens, new slots)."""
        hit = pa.pa_prefix_match(cache, tokens)
        seq = pa.pa_seq_create_from_prefix(pool.handle, hit)
        slots, pairs = pa.pa_seq_append(pool.handle, seq, len(tokens) - len(hit) * B)
        assert pairs.shape[0] == 0                       # whole cached blocks: nothing to copy
        pa.pa_prefix_insert(cache, tokens, pa.pa_seq_table(pool.handle, seq))
        return seq, len(hit) * B, slots

    dims = pa.make_dims(1, Hq, Hkv, D, B, N, 32, 0, dtype)
    for r in range(3):
        own = rng.integers(0, 1000, size=int(rng.integers(20, 90))).astype(np.int32)
        tokens = np.concatenate([prompt, own])
        seq, reused, slots = admit(tokens)
        assert reused == (0 if r == 0 else 192)          # the first request fills the cache
        n = len(tokens) - reused                          # the prefill chunk
        k_new = synth.normal(rng, (n, Hkv, D), 1.0, dtype)
        v_new = synth.normal(rng, (n, Hkv, D), 1.0, dtype)
        if reused:
            # the reused positions 192..199 of the prompt are recomputed: same rows as the first request
            k_new[:200 - reused] = first_k[reused:200]
            v_new[:200 - reused] = first_v[reused:200]
        else:
            first_k, first_v = k_new.copy(), v_new.copy()
        pa.pa_write_kv(dims, to_dev(torch, k_new, dtype), to_dev(torch, v_new, dtype),
                       torch.from_numpy(slots).cuda(), dkc, dvc)
        table = np.full((1, 32), -1, np.int32)
        t = pa.pa_seq_table(pool.handle, seq)
        table[0, :len(t)] = t
        q = synth.normal(rng, (n, Hq, D), 1.0, dtype)
        qs = np.array([0, n], np.int32)
        lens = np.array([len(tokens)], np.int32)
        out = torch.full((n, Hq, D), float("nan"), device="cuda")
        ws = torch.empty(max(pa.pa_chunk_workspace_bytes(dims, n, n), 16), dtype=torch.uint8, device="cuda")
        pa.pa_chunk_attention(dims, to_dev(torch, q, dtype), dkc, dvc, torch.from_numpy(table).cuda(),
                              torch.from_numpy(lens).cuda(), torch.from_numpy(qs).cuda(), 1 / np.sqrt(D), out, n, ws)
        got = out.cpu().numpy().astype(np.float64)
        assert pa.pa_device_errors(clear=True) == 0
        k_host = dkc.cpu().view(torch.int16).numpy().view(np.uint16)
        v_host = dvc.cpu().view(torch.int16).numpy().view(np.uint16)
        ref = oracle.chunk_attention(q, k_host, v_host, table, lens, qs, 1 / np.sqrt(D), dtype)
        assert_attention_close(got, ref)
        # the shared prompt blocks hold the first request's rows, bit for bit
        for j in range(12):
            blk = t[j]
            for i in range(B):
                np.testing.assert_array_equal(k_host[blk, :, i], first_k[j * B + i])
        pa.pa_seq_free(pool.handle, seq)
    assert pa.pa_prefix_cached_blocks(cache) >= 12
    pa.pa_prefix_cache_destroy(cache)
    pool.close()
