"""Benchmark of the paged decode hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = the whole hot path once over one batch: copy-on-write block copies
(when the step has any), the KV write of one new token per sequence, and
PagedAttention decode of one query per sequence over its full paged context
(split-K partitions plus the merge).  Block tables, slots and copy pairs come
from the library's allocator when the workload is set up.  The default
workload is the 8B-shaped grouped-query layer: 256 sequences, 32 query heads
over 8 KV heads, head_dim 128, bf16, 16-token blocks, lognormal lengths
(median 600, clipped to [1, 4096]).

Printed: one JSON line (rank 0).  `value` is KV-read GB/s over the whole step
(KV bytes of every sequence's valid tokens / step time), inputs resident in
HBM; `e2e` is the same metric through the binding with host buffers (the
step's inputs packed in one pinned buffer copied host -> device, and the
output copied device -> host, inside the timed region); `roofline` is the decode launch alone
against the measured HBM copy bandwidth; `cpu_baseline` is the fp64 CPU
oracle on a bounded sample.  Under torchrun each rank runs its own workload
replica (different seed) -- the path has no cross-GPU exchange -- and the
timing is the max over ranks.

`--impl reference` times the CPU oracle (the only other implementation of
this path) on the host cores, on the same workload, metric and units.
"""
from __future__ import annotations

import argparse
import collections
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged-decode KV-read GB/s (% of GB300 HBM peak); decode query-tokens/s/layer"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 126 * 2**20
KERNEL_SOURCES = ("pa_decode_mma.cuh", "pa_plan.cu", "pa_cache_ops.cu", "pa_tmap.cu", "pa_api.cu",
                  "pa_device.cuh", "pa_internal.h", "pa_mma.cuh")
CHUNK_SOURCES = ("pa_chunk_mma.cuh", "pa_chunk_umma.cuh", "pa_tcgen05.cuh", "pa_chunk.cu", "pa_merge.cuh", "pa_tmap.cu",
                 "pa_api.cu", "pa_device.cuh", "pa_internal.h", "pa_mma.cuh")


# --------------------------------------------------------------------------- distributed helpers
def dist_env():
    """(rank, local_rank, world_size) from the torchrun environment (1-process default)."""
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def dist_init(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def reduce_scalar(dist, value: float, op: str, device=None) -> float:
    """max / sum of a scalar over all ranks (identity with one process)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if (device is not None and dist.get_backend() == "nccl") else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


# --------------------------------------------------------------------------- peaks, clocks, profiles
def measured_hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(sources=KERNEL_SOURCES) -> str:
    h = hashlib.sha256()
    for name in sources:
        with open(os.path.join(ROOT, "paged_kv_cache_127_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kind: str = "decode", sources=KERNEL_SOURCES):
    """ncu DRAM bytes per call, if the summary matches the current kernel sources."""
    path = os.path.join(ROOT, "profiles", f"{kind}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)\s+sources:\s*([0-9a-f]+)", text)
    if not m or m.group(2) != kernel_source_hash(sources):
        return None
    return int(m.group(1))


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while it runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"pa_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- oracle timing
def host_cores() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the baseline's record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for key in ("Model name", "CPU part"):
            m = re.search(rf"^{key}:\s*(.+)$", out, flags=re.M)
            if m:
                arch = re.search(r"^Architecture:\s*(.+)$", out, flags=re.M)
                return f"{m.group(1).strip()} ({arch.group(1).strip() if arch else os.uname().machine})"
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip() + f" ({os.uname().machine})"
    except OSError:
        pass
    return os.uname().machine


def time_oracle(step, seq_ids, kc=None, vc=None):
    """Run the fp64 CPU oracle (KV write then decode) for the given sequences; return seconds."""
    import oracle
    kc = step.k_cache if kc is None else kc
    vc = step.v_cache if vc is None else vc
    t0 = time.perf_counter()
    oracle.write_kv(step.k_new[seq_ids], step.v_new[seq_ids], step.slots[seq_ids], kc, vc, step.dtype)
    oracle.decode(step.q[seq_ids], kc, vc, step.tables[seq_ids], step.lens[seq_ids], step.scale, step.dtype)
    return time.perf_counter() - t0


def cpu_baseline(step, budget_s: float = 15.0):
    """The oracle as it stands, single-threaded, on a bounded sample of sequences."""
    rng = np.random.default_rng(12345)
    order = rng.permutation(step.num_seqs)
    done, secs, nbytes = [], 0.0, 0
    per_tok = step.kv_bytes_per_token()
    for s in order:
        secs += time_oracle(step, np.array([s]))
        done.append(int(s))
        nbytes += int(step.lens[s]) * per_tok
        if secs >= budget_s:
            break
    tokens = int(step.lens[done].sum())
    return {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{len(done)} of {step.num_seqs} sequences ({tokens} context tokens), KV write + fp64 "
                      f"decode, single thread, {secs:.1f} s",
            "seconds": secs}


# The all-core baseline runs the unchanged oracle in a pool of spawned worker
# processes, one per host core; each worker maps the step's arrays from files
# (copy-on-write, so each KV write stays private) and takes sequences from a
# shared task list.
_POOL_STEP = None
_STEP_FIELDS = ("q", "k_new", "v_new", "slots", "tables", "lens", "k_cache", "v_cache")


def _pool_init(folder, dtype, scale):
    global _POOL_STEP
    import types
    import oracle
    oracle._load()
    arrs = {f: np.load(os.path.join(folder, f + ".npy"), mmap_mode="c") for f in _STEP_FIELDS}
    _POOL_STEP = types.SimpleNamespace(dtype=dtype, scale=scale, **arrs)


def _pool_task(ids):
    ids = np.asarray(ids)
    return time_oracle(_POOL_STEP, ids), int(_POOL_STEP.lens[ids].sum())


def _pool_ready(_):
    return _POOL_STEP is not None


class OraclePool:
    """A spawn-started process pool running the oracle over sequences of one step."""

    def __init__(self, step, cores=None):
        import multiprocessing as mp
        import tempfile
        import oracle
        oracle._load()                       # built once here, not by every worker
        self.cores = cores or host_cores()
        self.step = step
        self.folder = tempfile.mkdtemp(prefix="pa_oracle_pool_")
        for f in _STEP_FIELDS:
            np.save(os.path.join(self.folder, f + ".npy"), np.ascontiguousarray(getattr(step, f)))
        self.pool = mp.get_context("spawn").Pool(self.cores, initializer=_pool_init,
                                                 initargs=(self.folder, step.dtype, step.scale))
        assert all(self.pool.map(_pool_ready, range(4 * self.cores), chunksize=1))

    def run(self, tasks):
        """Run the tasks (arrays of sequence ids); returns (wall seconds, context tokens)."""
        t0 = time.perf_counter()
        res = self.pool.map(_pool_task, tasks, chunksize=1)
        return time.perf_counter() - t0, sum(r[1] for r in res)

    def close(self):
        import shutil
        self.pool.close()
        self.pool.join()
        shutil.rmtree(self.folder, ignore_errors=True)


def oracle_tasks(step, passes: int, per_task: int = 2, seed: int = 99):
    rng = np.random.default_rng(seed)
    tasks = []
    for _ in range(passes):
        order = rng.permutation(step.num_seqs)
        tasks += [order[i:i + per_task] for i in range(0, len(order), per_task)]
    return tasks


def cpu_baseline_all_cores(step, single_gbs: float, target_s: float = 8.0):
    """The unchanged oracle on every host core: whole passes over the step's
    sequences, as many as fit about target_s seconds at the expected speed-up."""
    pool = OraclePool(step)
    try:
        per_pass_s = step.kv_bytes_logical() / (single_gbs * 1e9) / pool.cores
        passes = int(max(1, min(200, round(target_s / max(per_pass_s, 1e-6)))))
        secs, tokens = pool.run(oracle_tasks(step, passes))
    finally:
        pool.close()
    nbytes = tokens * step.kv_bytes_per_token()
    return {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": pool.cores, "kind": "oracle",
            "sample": f"{passes} pass(es) over all {step.num_seqs} sequences ({tokens} context tokens), "
                      f"KV write + fp64 decode, {pool.cores} worker processes, {secs:.1f} s"}


# --------------------------------------------------------------------------- GPU timing helpers
def time_per_call(torch, fn, stream, reps: int, flush=None):
    """Per-call CUDA-event times (ms) of `fn`, one event pair per call; with
    `flush`, a buffer larger than L2 is overwritten before each call (outside
    the pair), so the call starts with cold caches.  Returns (median, min, all)."""
    pairs = []
    for _ in range(reps):
        if flush is not None:
            flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        pairs.append((e0, e1))
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in pairs]
    return float(np.median(ms)), float(np.min(ms)), ms


def time_back_to_back(torch, fn, stream, n: int):
    """Mean time (ms) of `fn` over n calls issued back to back between one event pair."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(n):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


def decode_launches(step, partition_size=None) -> int:
    """Kernels one pa_decode call launches: plan + tensor-core decode (+ merge when
    a sequence can span partitions) for 16-bit caches; CUDA-core decode (+ merge) for f32."""
    pt = partition_size or step.partition_size
    split = step.max_blocks * step.block_size > pt
    return (1 if step.dtype == "f32" else 2) + (1 if split else 0)


def decode_config(step, workload: str, world: int) -> dict:
    """The workload's description, shared by both arms' JSON lines."""
    kv_bytes = step.kv_bytes_logical()
    return {
        "workload": workload,
        "num_seqs": step.num_seqs, "num_q_heads": step.num_q_heads, "num_kv_heads": step.num_kv_heads,
        "head_dim": step.head_dim, "block_size": step.block_size, "partition_size": step.partition_size,
        "num_blocks": step.num_blocks, "context_tokens": int(step.lens.sum()),
        "max_context": int(step.lens.max()), "cow_pairs": int(step.pairs.shape[0]),
        "kv_bytes_per_step": kv_bytes, "kv_bytes_unique_per_step": step.kv_bytes_unique(),
        "l2": f"inputs larger than L2 ({kv_bytes / 2**20:.0f} MiB of KV read per step vs "
              f"{L2_BYTES / 2**20:.0f} MiB L2); no flush between steps",
        "parallelism": f"replicas x{world} (one workload per GPU, no collective on the data path)",
    }


# --------------------------------------------------------------------------- our arm
SWEEP_WORKLOADS = ("gqa8b_b32", "mha7b", "prefix_cow", "long70b", "tiny")
COMPONENT_REPS = 25          # per-call event pairs, each after an L2 flush
BACK_TO_BACK_CALLS = 200     # pa_decode calls between one event pair
SWEEP_STEPS = 50


class DecodeBuffers:
    """One decode step's device tensors and its prepared library calls
    (copy_blocks when the step has pairs, write_kv, decode) on `stream`."""

    def __init__(self, torch, pa, step, device, stream, q, k_new, v_new, slots, tables, lens, pairs, k_cache,
                 v_cache, extra_pairs=None):
        self.step, self.dims = step, step.dims(pa)
        S, Hq, D = step.num_seqs, step.num_q_heads, step.head_dim
        self.k_cache, self.v_cache = k_cache, v_cache
        self.out = torch.empty((S, Hq, D), dtype=torch.float32, device=device)
        ws_bytes = pa.pa_decode_workspace_bytes(self.dims)
        self.ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=device)
        self.npairs = int(pairs.shape[0])
        self.copy = (pa.pa_copy_blocks(self.dims, k_cache, v_cache, pairs, stream, prepare=True)
                     if self.npairs else None)
        self.write = pa.pa_write_kv(self.dims, k_new, v_new, slots, k_cache, v_cache, stream, prepare=True)
        self.decode = pa.pa_decode(self.dims, q, k_cache, v_cache, tables, lens, step.scale, self.out, self.ws,
                                   stream, prepare=True)
        # copy_blocks timed alone: the step's own pairs, else pairs into blocks no table uses
        self.copy_alone = self.copy
        if self.copy is None and extra_pairs is not None and len(extra_pairs):
            xp = torch.from_numpy(np.ascontiguousarray(extra_pairs, dtype=np.int64)).to(device)
            self.copy_alone = pa.pa_copy_blocks(self.dims, k_cache, v_cache, xp, stream, prepare=True)
        self.copy_alone_pairs = self.npairs or (0 if extra_pairs is None else len(extra_pairs))
        self.launches_per_step = (1 if self.npairs else 0) + 1 + decode_launches(step)

    def step_calls(self):
        if self.copy is not None:
            self.copy()
        self.write()
        self.decode()


def spare_pairs(step, n: int = 32) -> np.ndarray:
    """n copy pairs from blocks the step's tables use into blocks none uses
    (destinations distinct and never a source), for timing copy_blocks alone."""
    B = step.block_size
    used = set()
    for s in range(step.num_seqs):
        nb = -(-int(step.lens[s]) // B)
        used.update(int(b) for b in step.tables[s, :nb])
    free = [b for b in range(step.num_blocks) if b not in used]
    src = sorted(used)[:n]
    k = min(n, len(free), len(src))
    return np.array([[src[i], free[i]] for i in range(k)], dtype=np.int64).reshape(-1, 2)


def measure_components(torch, bufs: DecodeBuffers, stream, flush):
    """Fixed-length timings of the step's kernels, independent of --steps."""
    for _ in range(5):
        bufs.decode()
    b2b = time_back_to_back(torch, bufs.decode, stream, BACK_TO_BACK_CALLS)
    d_med, d_min, _ = time_per_call(torch, bufs.decode, stream, COMPONENT_REPS, flush)
    w_med, w_min, _ = time_per_call(torch, bufs.write, stream, COMPONENT_REPS, flush)
    out = {"decode_ms": {"back_to_back": round(b2b, 5), "median": round(d_med, 5), "min": round(d_min, 5),
                         "calls_back_to_back": BACK_TO_BACK_CALLS, "reps": COMPONENT_REPS},
           "write_kv_us": {"median": round(w_med * 1e3, 2), "min": round(w_min * 1e3, 2),
                           "tokens": int(bufs.step.slots.shape[0]), "reps": COMPONENT_REPS}}
    if bufs.copy_alone is not None:
        c_med, c_min, _ = time_per_call(torch, bufs.copy_alone, stream, COMPONENT_REPS, flush)
        out["copy_blocks_us"] = {"median": round(c_med * 1e3, 2), "min": round(c_min * 1e3, 2),
                                 "pairs": bufs.copy_alone_pairs, "reps": COMPONENT_REPS,
                                 "pairs_from": "the step's copy-on-write pairs" if bufs.npairs else
                                               "blocks in use copied into unused blocks"}
    return out


def roofline_of(step, comp, peak, peak_kind, workload):
    """The decode call against the HBM roofline: distinct KV bytes per call over
    its back-to-back mean time (and over the median of single calls after an L2 flush)."""
    kv_unique = step.kv_bytes_unique()
    dm = comp["decode_ms"]
    achieved = kv_unique / (dm["back_to_back"] / 1e3) / 1e9
    return {
        "bound": "hbm",
        "kernel": "pa_decode call (plan + tensor-core decode + split-K merge kernels)",
        "achieved": round(achieved, 1),
        "achieved_single_call_median": round(kv_unique / (dm["median"] / 1e3) / 1e9, 1),
        "achieved_logical": round(step.kv_bytes_logical() / (dm["back_to_back"] / 1e3) / 1e9, 1),
        "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
        "frac": round(achieved / peak, 4),
        "pct_of_nominal_8tbs": round(100 * achieved / NOMINAL_HBM_GBS, 2),
        "traffic": profiled_traffic(workload),
        "bytes": "distinct KV slots read per pa_decode call (2 * Hkv * D * sizeof per token)",
        "timing": f"mean of {dm['calls_back_to_back']} back-to-back calls between one CUDA event pair on the "
                  f"launch stream; single-call median/min over {dm['reps']} event pairs, L2 flushed before each",
    }


def timed_steps(torch, fn, stream, n):
    """Device time (ms) of n steps between one event pair, synchronised on both sides."""
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(n):
        fn()
    t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1)


def sweep_entry(torch, pa, name, rank, device, stream, flush, peak, peak_kind):
    """Another workload's decode step, with cache, query and new-row values drawn
    on the device (N(0, std) as the workload states); tables, slots and pairs
    from the allocator as for the headline."""
    from paged_kv_cache_127_gb300 import synth, workloads
    st = workloads.build_step(name, seed=rank, values=False, binding=pa)
    w = synth.workload(name, rank)
    kvt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[st.dtype]
    gen = torch.Generator(device=device)
    gen.manual_seed(7000 + 31 * rank + SWEEP_WORKLOADS.index(name))
    S, Hq, Hkv, D, B, N = (st.num_seqs, st.num_q_heads, st.num_kv_heads, st.head_dim, st.block_size,
                           st.num_blocks)
    T = int(st.slots.shape[0])

    def rnd(shape, std):
        t = torch.randn(shape, generator=gen, device=device, dtype=kvt)
        return t.mul_(std) if std != 1.0 else t

    kc, vc = rnd((N, Hkv, B, D), w.std), rnd((N, Hkv, B, D), w.std)
    q = rnd((S, Hq, D), w.std * w.q_prescale)
    kn, vn = rnd((T, Hkv, D), w.std), rnd((T, Hkv, D), w.std)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    bufs = DecodeBuffers(torch, pa, st, device, stream, q, kn, vn, dev(st.slots), dev(st.tables), dev(st.lens),
                         dev(st.pairs), kc, vc, extra_pairs=spare_pairs(st))
    for _ in range(5):
        bufs.step_calls()
    ms = timed_steps(torch, bufs.step_calls, stream, SWEEP_STEPS) / SWEEP_STEPS
    comp = measure_components(torch, bufs, stream, flush)
    torch.cuda.synchronize()
    assert torch.isfinite(bufs.out).all().item(), f"{name}: non-finite output"
    entry = {
        "value": round(st.kv_bytes_logical() / (ms / 1e3) / 1e9, 1), "unit": "GB/s",
        "ms_per_step": round(ms, 5), "steps": SWEEP_STEPS,
        "q_tok_per_s_per_layer": round(S / (ms / 1e3), 1),
        "dtype": st.dtype,
        **comp,
        "roofline": roofline_of(st, comp, peak, peak_kind, name),
        "config": decode_config(st, name, 1),
        "data": "synthetic: tables, slots and pairs from the allocator; values drawn on the device",
    }
    del bufs, kc, vc, q, kn, vn
    torch.cuda.empty_cache()
    return entry


def run_ours(args):
    import torch

    from paged_kv_cache_127_gb300 import binding as pa
    from paged_kv_cache_127_gb300 import workloads

    rank, local_rank, world = dist_env()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    dist = dist_init(world, "nccl")

    step = workloads.build_step(args.workload, seed=rank, binding=pa)
    if args.partition_size:
        step.partition_size = args.partition_size
    S, Hq, D = step.num_seqs, step.num_q_heads, step.head_dim
    kvt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[step.dtype]
    stream = torch.cuda.current_stream(device)

    # The step's inputs, packed in one pinned host buffer (for the end-to-end leg,
    # one host-to-device copy per step) and two device mirrors of it; the device
    # tensors are views into the mirrors.
    def as_bytes(x):
        return np.ascontiguousarray(x).view(np.uint8).reshape(-1)

    parts = [("q", step.q), ("k", step.k_new), ("v", step.v_new), ("slots", step.slots),
             ("tables", step.tables), ("lens", step.lens), ("pairs", np.ascontiguousarray(step.pairs))]
    tdt = {"q": kvt, "k": kvt, "v": kvt, "slots": torch.int64, "tables": torch.int32, "lens": torch.int32,
           "pairs": torch.int64}
    offs, total = {}, 0
    for name, arr in parts:
        offs[name] = total
        total += (as_bytes(arr).size + 255) // 256 * 256
    h_in = torch.empty(total, dtype=torch.uint8).pin_memory()
    for name, arr in parts:
        b = as_bytes(arr)
        h_in[offs[name]:offs[name] + b.size] = torch.from_numpy(b)
    d_ins = [torch.empty(total, dtype=torch.uint8, device=device) for _ in range(2)]
    for d in d_ins:
        pa.pa_copy_to_device(d, h_in, stream)

    def host_cache(x):
        t = torch.from_numpy(np.ascontiguousarray(x))
        return t.view(torch.int16).view(torch.bfloat16) if step.dtype == "bf16" else t

    d_kc, d_vc = host_cache(step.k_cache).to(device), host_cache(step.v_cache).to(device)

    def views(d_in):
        return {name: d_in[offs[name]:offs[name] + np.ascontiguousarray(arr).nbytes].view(tdt[name])
                .view(np.ascontiguousarray(arr).shape) for name, arr in parts}

    vws = [views(d) for d in d_ins]
    bufs = [DecodeBuffers(torch, pa, step, device, stream, v["q"], v["k"], v["v"], v["slots"], v["tables"],
                          v["lens"], v["pairs"], d_kc, d_vc, extra_pairs=spare_pairs(step)) for v in vws]
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)
    peak, peak_kind = measured_hbm_peak()

    pa.pa_device_errors(clear=True)
    sampler = ClockSampler(device.index).start() if rank == 0 else None
    for _ in range(args.warmup):
        bufs[0].step_calls()
    torch.cuda.synchronize(device)
    assert pa.pa_device_errors(clear=True) == 0, "device error flags set during warm-up"

    # ---- the timed steps: exactly K steps between one event pair, inputs resident in HBM
    barrier(dist, device)
    ms_local = timed_steps(torch, bufs[0].step_calls, stream, args.steps)
    barrier(dist, device)
    ms_total = reduce_scalar(dist, ms_local, "max", device)

    # ---- fixed-length component timings (roofline), independent of --steps
    comp = measure_components(torch, bufs[0], stream, flush)

    # ---- end to end through the library with host buffers.  Every step copies
    # all of its inputs host -> device (one packed pa_copy_to_device) and its
    # output device -> host (pa_copy_to_host); steps are double-buffered over
    # three streams, so step i's copies overlap the compute of steps i - 1 and
    # i + 1.  The host orders the buffers: it waits for step i's inputs to land
    # before it enqueues step i's kernels (the GPU is still busy with step
    # i - 1 then), and collects step i - 1's result before it reuses that
    # step's buffers for step i + 1.  So the compute stream carries no
    # cross-stream waits, and consecutive steps' kernels keep their
    # programmatic-launch overlap.
    e2e_steps = max(1, args.e2e_steps)
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    h_outs = [torch.empty((S, Hq, D), dtype=torch.float32).pin_memory() for _ in range(2)]
    h2d = [pa.pa_copy_to_device(d_ins[b], h_in, s_in, prepare=True) for b in range(2)]
    d2h = [pa.pa_copy_to_host(h_outs[b], bufs[b].out, s_out, prepare=True) for b in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_loop(n):
        for i in range(n):
            b = i & 1
            h2d[b]()                            # buffer b's last user, step i - 2, is complete
            ev_in[b].record(s_in)
            ev_in[b].synchronize()              # step i's inputs are on the device
            bufs[b].step_calls()
            ev_cmp[b].record(stream)
            s_out.wait_event(ev_cmp[b])
            d2h[b]()
            ev_out[b].record(s_out)
            if i >= 1:
                ev_out[b ^ 1].synchronize()     # the host has step i - 1's result
        torch.cuda.synchronize(device)

    e2e_loop(3)
    barrier(dist, device)
    torch.cuda.synchronize(device)
    w0 = time.perf_counter()
    e2e_loop(e2e_steps)
    e2e_s = time.perf_counter() - w0
    barrier(dist, device)
    e2e_s = reduce_scalar(dist, e2e_s, "max", device)
    assert pa.pa_device_errors(clear=True) == 0, "device error flags set during the timed steps"
    assert torch.isfinite(bufs[0].out).all().item()

    sweeps = {}
    if rank == 0 and world == 1 and not args.no_sweeps and args.workload == "gqa8b_b16" \
            and not args.partition_size:
        del bufs, vws, d_ins, d_kc, d_vc
        torch.cuda.empty_cache()
        for name in SWEEP_WORKLOADS:
            sweeps[name] = sweep_entry(torch, pa, name, rank, device, stream, flush, peak, peak_kind)
        assert pa.pa_device_errors(clear=True) == 0, "device error flags set during the sweeps"
    clocks = sampler.stop() if sampler else None

    kv_bytes = step.kv_bytes_logical()
    kv_all = reduce_scalar(dist, kv_bytes, "sum", device)
    seqs_all = reduce_scalar(dist, S, "sum", device)
    step_s = ms_total / 1e3 / args.steps
    if rank != 0:
        return None
    value = kv_all / step_s / 1e9
    launches_per_step = (1 if step.pairs.shape[0] else 0) + 1 + decode_launches(step)
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_total / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": step.dtype,
        "data": "synthetic (seeded; shapes and length distributions of the workload)",
        "config": decode_config(step, args.workload, world),
        "q_tok_per_s_per_layer": round(seqs_all / step_s, 1),
        "pct_of_nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        **comp,
        "roofline": roofline_of(step, comp, peak, peak_kind, args.workload),
        "e2e": {"value": round(kv_all * e2e_steps / e2e_s / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": h_in.numel(),
                "d2h_bytes_per_step": h_outs[0].numel() * h_outs[0].element_size(),
                "ms_per_step": round(e2e_s * 1e3 / e2e_steps, 5), "steps": e2e_steps,
                "copies": "pa_copy_to_device / pa_copy_to_host (cudaMemcpyAsync in the library), pinned host "
                          "buffers, double-buffered over copy-in / compute / copy-out streams"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if sweeps:
        line["sweeps"] = sweeps
    if world == 1 and not args.no_cpu_baseline:
        single = {k: v for k, v in cpu_baseline(step).items() if k != "seconds"}
        try:
            base = cpu_baseline_all_cores(step, single["value"])
        except Exception as e:   # the single-thread figure then stands alone
            base = dict(single, all_cores_unavailable=f"{type(e).__name__}: {e}")
        base["single_thread"] = single
        base["cpu_model"] = cpu_model()
        line["cpu_baseline"] = base
    return line


# --------------------------------------------------------------------------- chunk attention
def measured_bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (cuBLAS bf16 GEMM, burst)"
    except Exception:
        return 1900.0, "fallback"


def run_chunk(args):
    """Chunk attention (several query tokens per sequence): one step is the KV
    write of every new token followed by pa_chunk_attention over them."""
    import torch

    from paged_kv_cache_127_gb300 import binding as pa
    from paged_kv_cache_127_gb300 import workloads

    rank, local_rank, world = dist_env()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    dist = dist_init(world, "nccl")
    step = workloads.build_step(args.workload, seed=rank, binding=pa)
    if args.partition_size:
        step.partition_size = args.partition_size
    dims = step.dims(pa)
    T, Hq, D, n = step.num_tokens, step.num_q_heads, step.head_dim, step.query_len
    kvt = torch.bfloat16 if step.dtype == "bf16" else torch.float16

    def dev(x, dt=None):
        if dt is None:
            return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(kvt).to(device)
        return torch.from_numpy(np.ascontiguousarray(x)).to(device)

    d_q, d_k, d_v = dev(step.q), dev(step.k_new), dev(step.v_new)
    d_kc, d_vc = dev(step.k_cache), dev(step.v_cache)
    d_slots, d_tables = dev(step.slots, 1), dev(step.tables, 1)
    d_lens, d_qs = dev(step.lens, 1), dev(step.query_start(), 1)
    d_out = torch.empty((T, Hq, D), dtype=torch.float32, device=device)
    ws = torch.empty(max(pa.pa_chunk_workspace_bytes(dims, T, n), 16), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    G = Hq // step.num_kv_heads
    umma = n * G >= 64                                # long chunks: the tcgen05 kernel, no split-K merge
    split = step.max_blocks * step.block_size > step.partition_size and not umma
    launches_per_step = 1 + 2 + (1 if split else 0)   # write_kv, plan, chunk kernel, merge
    write = pa.pa_write_kv(dims, d_k, d_v, d_slots, d_kc, d_vc, stream, prepare=True)
    attend = pa.pa_chunk_attention(dims, d_q, d_kc, d_vc, d_tables, d_lens, d_qs, step.scale, d_out, n, ws, stream,
                                   prepare=True)

    def device_step():
        write()
        attend()

    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)
    pa.pa_device_errors(clear=True)
    sampler = ClockSampler(device.index).start() if rank == 0 else None
    for _ in range(args.warmup):
        device_step()
    torch.cuda.synchronize(device)
    barrier(dist, device)
    ms = reduce_scalar(dist, timed_steps(torch, device_step, stream, args.steps), "max", device) / args.steps
    barrier(dist, device)
    call_ms = time_back_to_back(torch, attend, stream, BACK_TO_BACK_CALLS // 4)
    c_med, c_min, _ = time_per_call(torch, attend, stream, COMPONENT_REPS, flush)
    clocks = sampler.stop() if sampler else None
    assert pa.pa_device_errors(clear=True) == 0, "device error flags set during the timed steps"
    assert torch.isfinite(d_out).all().item()
    kv = step.kv_bytes_unique()      # every visible KV slot once (the last query sees the whole context)
    flops = step.chunk_flops()
    if rank != 0:
        return None
    hbm_peak, hbm_kind = measured_hbm_peak()
    tc_peak, tc_kind = measured_bf16_peak()
    gbs = kv / (call_ms / 1e3) / 1e9
    tfs = flops / (call_ms / 1e3) / 1e12
    hbm_bound = kv / (hbm_peak * 1e9) > flops / (tc_peak * 1e12)
    roof = ({"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak, "peak_kind": hbm_kind, "unit": "GB/s",
             "frac": round(gbs / hbm_peak, 4)} if hbm_bound else
            {"bound": "tensor", "achieved": round(tfs, 2), "peak": tc_peak, "peak_kind": tc_kind, "unit": "TFLOP/s",
             "frac": round(tfs / tc_peak, 4)})
    roof.update({"traffic": profiled_traffic(args.workload, "chunk", CHUNK_SOURCES),
                 "kernel": ("pa_chunk_attention (plan + tcgen05 chunk kernel)" if umma else
                            "pa_chunk_attention (plan + mma.sync chunk kernel + split-K merge)"),
                 "call_ms": round(call_ms, 5),
                 "call_ms_single_median": round(c_med, 5), "call_ms_single_min": round(c_min, 5),
                 "timing": f"mean of {BACK_TO_BACK_CALLS // 4} back-to-back calls between one CUDA event pair; "
                           f"single-call median/min over {COMPONENT_REPS} event pairs, L2 flushed before each",
                 "bytes": "distinct visible KV slots per call", "flops": "4 * D * Hq per (query, visible key)"})
    line = {
        "metric": "paged chunk-attention query-tokens/s (KV write + causal attention of every new token)",
        "value": round(T * world / (ms / 1e3), 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": step.dtype, "data": "synthetic (seeded)",
        "config": {"workload": args.workload, "num_seqs": step.num_seqs, "query_len": n, "num_q_heads": Hq,
                   "num_kv_heads": step.num_kv_heads, "head_dim": D, "block_size": step.block_size,
                   "partition_size": step.partition_size,
                   "context_tokens": int(step.lens.sum()), "kv_bytes_unique_per_step": kv,
                   "flops_per_step": flops,
                   "l2": f"{kv / 2**20:.0f} MiB of KV per step vs {L2_BYTES / 2**20:.0f} MiB L2; no flush"},
        "kv_gbs": round(gbs, 1), "tflops": round(tfs, 2),
        "roofline": roof, "gpu_launches": launches_per_step * args.steps, "clocks": clocks,
    }
    if world == 1 and not args.no_cpu_baseline:
        import oracle  # the CPU-baseline leg only

        rng = np.random.default_rng(7)
        order = rng.permutation(step.num_seqs)
        kc, vc = step.k_cache, step.v_cache
        oracle.write_kv(step.k_new, step.v_new, step.slots, kc, vc, step.dtype)
        secs, done, toks = 0.0, 0, 0
        # a sample of query rows: rows a..b-1 of a chunk are the last b - a queries of
        # the context cut after row b - 1, so a long chunk is sampled a few rows at a time
        r = min(n, 8)
        for s_ in order:
            a0 = int(rng.integers(0, n - r + 1))
            cut = int(step.lens[s_]) - n + a0 + r
            c0 = time.perf_counter()
            oracle.chunk_attention(step.q[s_ * n + a0:s_ * n + a0 + r], kc, vc, step.tables[s_:s_ + 1],
                                   np.array([cut], np.int32), np.array([0, r], np.int32), step.scale, step.dtype)
            secs += time.perf_counter() - c0
            done += 1
            toks += r
            if secs > 15.0:
                break
        line["cpu_baseline"] = {"value": round(toks / secs, 2), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                "sample": f"{toks} query tokens ({r} consecutive rows from each of {done} sequences), "
                                          f"fp64 chunk attention, single thread, {secs:.1f} s"}
    return line


# --------------------------------------------------------------------------- multi-layer step
def run_layers(args):
    """One decode step over L layers of a multi-layer pool: a captured step graph
    (write_kv + decode per layer) against the same launches issued one by one."""
    import torch

    from paged_kv_cache_127_gb300 import binding as pa
    from paged_kv_cache_127_gb300 import workloads

    rank, local_rank, world = dist_env()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    dist = dist_init(world, "nccl")
    L = args.layers
    step = workloads.build_step(args.workload, seed=rank, binding=pa)
    if args.num_seqs:
        step = step.first(args.num_seqs)
    if args.partition_size:
        step.partition_size = args.partition_size
    dims = step.dims(pa)
    S, Hq, Hkv, D, B, N = (step.num_seqs, step.num_q_heads, step.num_kv_heads, step.head_dim,
                           step.block_size, step.num_blocks)
    kvt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[step.dtype]

    def host(x):
        if step.dtype == "bf16":
            return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(x))

    gen = torch.Generator(device=device)
    gen.manual_seed(1234 + rank)

    def layered(first, shape, std):
        t = torch.empty((L,) + tuple(shape), dtype=kvt, device=device)
        t[0].copy_(host(first))
        for layer in range(1, L):
            t[layer].copy_(torch.randn(shape, generator=gen, device=device) * std)
        return t

    w_std = 1.0
    kc = layered(step.k_cache, step.k_cache.shape, w_std)
    vc = layered(step.v_cache, step.v_cache.shape, w_std)
    q = layered(step.q, step.q.shape, w_std * (1.0 / math.sqrt(D) if step.name.startswith("gqa8b") else 1.0))
    kn = layered(step.k_new, step.k_new.shape, w_std)
    vn = layered(step.v_new, step.v_new.shape, w_std)
    slots = torch.from_numpy(step.slots).to(device)
    tables = torch.from_numpy(step.tables).to(device)
    lens = torch.from_numpy(step.lens).to(device)
    out = torch.empty((L, S, Hq, D), dtype=torch.float32, device=device)
    ws = torch.empty(max(pa.pa_decode_workspace_bytes(dims), 256), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    graph = pa.pa_step_graph_create(dims, kc, vc, q, kn, vn, slots, tables, lens, step.scale, out, ws)

    def eager():
        for layer in range(L):
            pa.pa_write_kv(dims, kn[layer], vn[layer], slots, kc[layer], vc[layer], stream)
            pa.pa_decode(dims, q[layer], kc[layer], vc[layer], tables, lens, step.scale, out[layer], ws, stream)

    def timed(fn, n):
        barrier(dist, device)
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(device)
        return reduce_scalar(dist, e0.elapsed_time(e1) / n, "max", device)

    pa.pa_device_errors(clear=True)
    sampler = ClockSampler(device.index).start() if rank == 0 else None
    for _ in range(args.warmup):
        graph.launch(stream)
        eager()
    graph_ms = timed(graph.launch, args.steps)
    eager_ms = timed(eager, max(1, args.steps // 2))
    clocks = sampler.stop() if sampler else None
    assert pa.pa_device_errors(clear=True) == 0
    graph.close()
    kv_bytes = step.kv_bytes_logical() * L
    kv_all = reduce_scalar(dist, kv_bytes, "sum", device)
    if rank != 0:
        return None
    return {
        "metric": METRIC + f" -- one decode step over {L} layers",
        "value": round(kv_all / (graph_ms / 1e3) / 1e9, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(graph_ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": step.dtype,
        "data": "synthetic (layer 0 from the workload generator, layers 1.. from a seeded device generator)",
        "config": {"workload": args.workload, "layers": L, "num_seqs": S, "num_q_heads": Hq,
                   "num_kv_heads": Hkv, "head_dim": D, "block_size": B, "num_blocks_per_layer": N,
                   "kv_bytes_per_step": kv_bytes},
        "graph_ms_per_step": round(graph_ms, 4), "eager_ms_per_step": round(eager_ms, 4),
        "eager_over_graph": round(eager_ms / graph_ms, 3),
        "gpu_launches": L * (2 + (2 if step.max_blocks * B > step.partition_size else 1)) * args.steps,
        "clocks": clocks,
    }


# --------------------------------------------------------------------------- block swap
def run_swap(args):
    """Swap-out / swap-in bandwidth: N whole blocks (all KV heads, K and V)
    between the device pool and pinned host memory, one pa_swap_blocks call per
    direction per step."""
    import torch

    from paged_kv_cache_127_gb300 import binding as pa
    from paged_kv_cache_127_gb300 import synth

    rank, local_rank, world = dist_env()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    w = synth.workload(args.workload)
    nb = args.swap_blocks
    N = 2 * nb
    dims = pa.make_dims(0, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, N, 1, 0, w.dtype)
    kvt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[w.dtype]
    shape = (N, w.num_kv_heads, w.block_size, w.head_dim)
    gen = torch.Generator(device=device)
    gen.manual_seed(99 + rank)
    kc = torch.randn(shape, generator=gen, device=device).to(kvt)
    vc = torch.randn(shape, generator=gen, device=device).to(kvt)
    hk = torch.empty((nb,) + shape[1:], dtype=kvt).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    rng = np.random.default_rng(5 + rank)
    dev_ids = rng.permutation(N)[:nb]
    out_pairs = torch.from_numpy(np.stack([dev_ids, rng.permutation(nb)], 1).astype(np.int64)).to(device)
    in_pairs = torch.from_numpy(np.stack([out_pairs[:, 1].cpu().numpy(), rng.permutation(N)[:nb]], 1)
                                .astype(np.int64)).to(device)
    stream = torch.cuda.current_stream(device)
    block_bytes = 2 * w.num_kv_heads * w.block_size * w.head_dim * synth.ELEM_BYTES[w.dtype]

    def timed(direction, pairs, n):
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            pa.pa_swap_blocks(dims, kc, vc, hk, hv, pairs, direction, stream)
        e1.record(stream)
        torch.cuda.synchronize(device)
        return e0.elapsed_time(e1) / n

    for _ in range(args.warmup):
        pa.pa_swap_blocks(dims, kc, vc, hk, hv, out_pairs, pa.PA_SWAP_OUT, stream)
        pa.pa_swap_blocks(dims, kc, vc, hk, hv, in_pairs, pa.PA_SWAP_IN, stream)
    out_ms = timed(pa.PA_SWAP_OUT, out_pairs, args.steps)
    in_ms = timed(pa.PA_SWAP_IN, in_pairs, args.steps)
    assert pa.pa_device_errors(clear=True) == 0
    if rank != 0:
        return None
    total = nb * block_bytes
    return {"metric": "block swap GB/s (device pool <-> pinned host memory)", "unit": "GB/s",
            "value": round(total / (out_ms / 1e3) / 1e9, 1), "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True,
            "config": {"workload": args.workload, "blocks": nb, "bytes_per_block": block_bytes,
                       "bytes_per_call": total},
            "swap_out_gbs": round(total / (out_ms / 1e3) / 1e9, 1), "swap_out_ms": round(out_ms, 4),
            "swap_in_gbs": round(total / (in_ms / 1e3) / 1e9, 1), "swap_in_ms": round(in_ms, 4),
            "gpu_launches": 2 * args.steps}


# --------------------------------------------------------------------------- prefix cache
class _ProductPrefix:
    """The C-ABI pool + radix-tree cache behind the calls the serving loop makes."""

    def __init__(self, pa, num_blocks, B, order):
        self.pa, self.pool = pa, pa.Pool(num_blocks, B, order)
        self.cache = pa.pa_prefix_cache_create(self.pool.handle)

    def match(self, toks):
        return self.pa.pa_prefix_match(self.cache, toks)

    def create(self, blocks):
        return self.pa.pa_seq_create_from_prefix(self.pool.handle, blocks)

    def append(self, sid, n):
        self.pa.pa_seq_append(self.pool.handle, sid, n)

    def insert(self, toks, sid):
        return self.pa.pa_prefix_insert(self.cache, toks, self.pa.pa_seq_table(self.pool.handle, sid))

    def evict(self, n):
        return self.pa.pa_prefix_evict(self.cache, n)

    def free(self, sid):
        self.pa.pa_seq_free(self.pool.handle, sid)

    def num_free(self):
        return self.pa.pa_pool_num_free(self.pool.handle)

    def cached(self):
        return self.pa.pa_prefix_cached_blocks(self.cache)

    def close(self):
        self.pa.pa_prefix_cache_destroy(self.cache)
        self.pool.close()


class _OraclePrefix:
    """The same calls on the oracle's block-manager and prefix-cache models."""

    def __init__(self, num_blocks, B, order):
        from oracle.block_manager import BlockManager
        from oracle.prefix_cache import PrefixCache, create_from_prefix
        self.bm = BlockManager(num_blocks, B, list(order))
        self.pc, self._create = PrefixCache(self.bm), create_from_prefix

    def match(self, toks):
        return self.pc.match(toks.tolist())

    def create(self, blocks):
        return self._create(self.bm, blocks)

    def append(self, sid, n):
        self.bm.append(sid, n)

    def insert(self, toks, sid):
        return self.pc.insert(toks.tolist(), self.bm.table(sid))

    def evict(self, n):
        return self.pc.evict(n)

    def free(self, sid):
        self.bm.free_seq(sid)

    def num_free(self):
        return self.bm.num_free()

    def cached(self):
        return self.pc.cached_blocks()

    def close(self):
        pass


def serve_prefix_stream(ops, reqs, B, live_cap, budget_s=None):
    """Admit requests in order: reuse the longest cached prefix, evict cached
    blocks (then finish the oldest running request) when the pool is short,
    store the rest of the prompt, cache it; at most live_cap requests run.
    Returns (requests done, seconds, per-request hit blocks)."""
    live, hits = collections.deque(), []
    t0 = time.perf_counter()
    for i, toks in enumerate(reqs):
        if budget_s is not None and i and time.perf_counter() - t0 > budget_s:
            break
        hit = ops.match(toks)
        sid = ops.create(hit)
        need = -(-len(toks) // B) - len(hit)
        while ops.num_free() < need:
            if ops.evict(need - ops.num_free()) == 0:
                if not live:
                    raise RuntimeError("request larger than the pool")
                ops.free(live.popleft())
        ops.append(sid, len(toks) - len(hit) * B)
        ops.insert(toks, sid)
        hits.append(len(hit))
        live.append(sid)
        if len(live) > live_cap:
            ops.free(live.popleft())
    return len(hits), time.perf_counter() - t0, hits


def run_prefix(args):
    """Host throughput of prefix-cache admission and the blocks it saves, on a
    stream of requests sharing a few system prompts and multi-turn histories."""
    rank, _, world = dist_env()
    if rank != 0:
        return None
    from paged_kv_cache_127_gb300 import binding as pa
    from paged_kv_cache_127_gb300 import synth

    B = synth.workload(args.workload).block_size
    rng = synth.make_rng(31)
    reqs = synth.prefix_requests(rng, args.prefix_requests)
    live_cap = 256
    blocks = np.array([-(-len(t) // B) for t in reqs])
    num_blocks = int(1.25 * live_cap * blocks.mean()) + int(blocks.max())
    order = synth.free_order(rng, num_blocks)
    for _ in range(min(args.warmup, 5)):
        ops = _ProductPrefix(pa, num_blocks, B, order)
        serve_prefix_stream(ops, reqs[:200], B, live_cap)
        ops.close()
    runs = []
    # each repetition serves the whole stream (about a second): at most 5, the median reported
    for _ in range(max(1, min(args.steps, 5))):
        ops = _ProductPrefix(pa, num_blocks, B, order)
        done, secs, hits = serve_prefix_stream(ops, reqs, B, live_cap)
        cached_end = ops.cached()
        ops.close()
        runs.append(secs)
    secs = float(np.median(runs))
    line = {
        "metric": "prefix-cache admissions/s (host: match + create + append + insert, evict on demand)",
        "value": round(done / secs, 1), "unit": "requests/s", "n_gpus": world, "steps": len(runs),
        "warmup": args.warmup, "ms_per_step": round(secs * 1e3, 3), "higher_is_better": True,
        "dtype": "int32", "data": "synthetic (seeded request stream)",
        "config": {"workload": f"prefix stream: {len(reqs)} requests, 8 shared prompts (median 512 tokens), "
                               f"30% multi-turn follow-ups, B={B}, {live_cap} running, pool {num_blocks} blocks",
                   "block_size": B, "requests": len(reqs), "pool_blocks": num_blocks, "running": live_cap},
        "hit_blocks_fraction": round(float(np.sum(hits)) / float(blocks.sum()), 4),
        "blocks_allocated": int(blocks.sum() - np.sum(hits)), "blocks_without_cache": int(blocks.sum()),
        "cached_blocks_at_end": int(cached_end), "gpu_launches": 0,
    }
    if not args.no_cpu_baseline:
        ref = _OraclePrefix(num_blocks, B, order)
        k, rsecs, rhits = serve_prefix_stream(ref, reqs, B, live_cap, budget_s=15.0)
        line["cpu_baseline"] = {"value": round(k / rsecs, 1), "unit": "requests/s", "cores": 1, "kind": "oracle",
                                "sample": f"first {k} requests of the same stream, single thread"}
        line["agrees_with_oracle"] = rhits == hits[:k]
    return line


# --------------------------------------------------------------------------- reference arm
class _OracleAllocator:
    """The allocator calls a workload's set-up makes, served by the oracle's
    block-manager model (the pages' bookkeeping rules in plain Python), so the
    reference arm builds the same tables, slots and pairs without loading the
    product library."""

    class Pool:
        def __init__(self, num_blocks, block_size, order):
            from oracle.block_manager import BlockManager
            self.handle = BlockManager(num_blocks, block_size, [int(b) for b in order])

        def close(self):
            pass

    @staticmethod
    def pa_seq_create(bm):
        return bm.create()

    @staticmethod
    def pa_seq_fork(bm, parent):
        return bm.fork(parent)

    @staticmethod
    def pa_seq_append(bm, seq, n):
        return bm.append(seq, int(n))

    @staticmethod
    def pa_seq_free(bm, seq):
        bm.free_seq(seq)

    @staticmethod
    def pa_seq_append_batch(bm, seqs, n):
        slots, pairs = [], []
        for s_ in seqs:
            sl, pr = bm.append(s_, int(n))
            slots += sl
            pairs += pr
        return (np.array(slots, dtype=np.int64).reshape(len(seqs), int(n)),
                np.array(pairs, dtype=np.int64).reshape(-1, 2))

    @staticmethod
    def pa_copy_pairs_check(pairs, num_blocks):
        dst = [int(d) for d in pairs[:, 1]]
        if len(set(dst)) != len(dst) or set(dst) & {int(x) for x in pairs[:, 0]} or \
                any(not 0 <= int(b) < num_blocks for b in pairs.reshape(-1)):
            raise ValueError("copy pairs violate the copy precondition")

    @staticmethod
    def pa_pool_export(bm, seqs, max_blocks, pad=-1):
        tables = np.full((len(seqs), max_blocks), pad, dtype=np.int32)
        lens = np.zeros(len(seqs), dtype=np.int32)
        for i, s_ in enumerate(seqs):
            t = bm.table(s_)
            tables[i, :len(t)] = t
            lens[i] = bm.length(s_)
        return tables, lens


def run_reference(args):
    """Time the CPU oracle on every host core: each step is one bounded sample
    of the workload (the whole batch when it fits), run by a spawned process
    pool, with tables, slots and pairs from the oracle's own block manager."""
    rank, _, world = dist_env()
    if rank != 0:
        return None
    from paged_kv_cache_127_gb300 import workloads

    step = workloads.build_step(args.workload, seed=0, binding=_OracleAllocator)
    if args.partition_size:
        step.partition_size = args.partition_size
    rng = np.random.default_rng(7)
    order = rng.permutation(step.num_seqs)
    per_seq = max(time_oracle(step, order[:2]) / 2, 1e-4)       # one thread, seconds per sequence
    pool = OraclePool(step)
    try:
        # size each step so that the whole run stays within ~2 minutes
        budget = 100.0 / max(1, args.steps + args.warmup)
        k = int(max(1, min(step.num_seqs, budget * pool.cores / per_seq)))
        per_tok = step.kv_bytes_per_token()
        pos = 0

        def one():
            nonlocal pos
            ids = np.array([order[(pos + i) % step.num_seqs] for i in range(k)])
            pos += k
            return pool.run([ids[i:i + 2] for i in range(0, k, 2)])

        for _ in range(args.warmup):
            one()
        secs, tokens = 0.0, 0
        for _ in range(args.steps):
            s_, t_ = one()
            secs += s_
            tokens += t_
    finally:
        pool.close()
    value = tokens * per_tok / secs / 1e9
    config = decode_config(step, args.workload, world)
    config["sequences_per_step"] = k
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; same workload as the GPU arm)",
        "config": config,
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": pool.cores, "kind": "oracle",
                         "cpu_model": cpu_model(),
                         "sample": f"{k} of {step.num_seqs} sequence(s) per step, KV write + fp64 decode, "
                                   f"{pool.cores} worker processes"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description="paged decode benchmark")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", default="gqa8b_b16")
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--e2e-steps", type=int, default=200,
                    help="steps of the end-to-end leg (a fixed count, independent of --steps)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweeps", action="store_true",
                    help="skip the other decode workloads in the default gqa8b_b16 run")
    ap.add_argument("--num-seqs", type=int, default=0,
                    help="with --layers: use only the first K sequences of the workload")
    ap.add_argument("--swap-blocks", type=int, default=0,
                    help="measure block swap bandwidth for this many blocks instead")
    ap.add_argument("--layers", type=int, default=1,
                    help="time one step over this many layers through the captured step graph")
    ap.add_argument("--prefix-requests", type=int, default=0,
                    help="measure prefix-cache admission on a stream of this many requests instead")
    ap.add_argument("--partition-size", type=int, default=0,
                    help="context tokens per split-K partition (default: the workload's, 512)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        line = run_reference(args)
    elif args.prefix_requests > 0:
        line = run_prefix(args)
    elif args.workload in ("verify8b", "prefill8b"):
        line = run_chunk(args)
    elif args.swap_blocks > 0:
        line = run_swap(args)
    elif args.layers > 1:
        line = run_layers(args)
    else:
        line = run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)
    if dist_env()[2] > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
