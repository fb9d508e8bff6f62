"""Host-side pieces of bench.py: the multi-rank timing reduction over gloo
(world size 2, CPU only), the CPU-oracle reference arm on the tiny workload
(all host cores, its own allocator model, no product library loaded)."""
import io
import json
import os
import socket
import subprocess
import sys
from contextlib import redirect_stdout

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    r, lr, w = bench.dist_env()
    dist = bench.dist_init(w, "gloo")
    bench.barrier(dist)
    # each rank times its own replica; the job is as slow as its slowest rank and
    # its throughput counts every rank's bytes
    mx = bench.reduce_scalar(dist, 10.0 + rank, "max")
    sm = bench.reduce_scalar(dist, 100 * (rank + 1), "sum")
    bench.barrier(dist)
    dist.destroy_process_group()
    q.put((r, lr, w, mx, sm))


def test_two_rank_timing_reduction_over_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 0, 2, 11.0, 300.0), (1, 1, 2, 11.0, 300.0)]


def test_single_process_helpers_are_identity(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 0, 1)
    assert bench.dist_init(1, "gloo") is None
    assert bench.reduce_scalar(None, 3.5, "max") == 3.5


def test_reference_arm_runs_the_oracle_on_cpu(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        monkeypatch.delenv(k, raising=False)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "3"])
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["metric"] == bench.METRIC
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == bench.host_cores()
    assert line["cpu_baseline"]["cpu_model"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    # the same workload description as the GPU arm prints
    for key in ("num_q_heads", "num_kv_heads", "head_dim", "block_size", "num_blocks", "context_tokens",
                "kv_bytes_per_step", "partition_size"):
        assert key in line["config"]


def test_reference_arm_loads_no_product_library():
    code = ("import sys, io, contextlib; sys.path.insert(0, %r); import bench\n"
            "with contextlib.redirect_stdout(io.StringIO()):\n"
            "    bench.main(['--impl', 'reference', '--workload', 'tiny', '--steps', '3', '--warmup', '3'])\n"
            "maps = open('/proc/self/maps').read()\n"
            "print('libpa.so' in maps, 'paged_kv_cache_127_gb300.binding' in sys.modules)\n" % ROOT)
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "LOCAL_RANK", "WORLD_SIZE")}
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=600)
    assert out.returncode == 0, out.stderr
    assert out.stdout.split() == ["False", "False"]


@pytest.mark.parametrize("name", ["tiny", "mha7b", "gqa8b_b16", "gqa8b_b32", "prefix_cow", "long70b",
                                  "verify8b", "prefill8b"])
def test_reference_allocator_builds_the_product_allocator_step(name):
    # the reference arm's inputs come from the oracle's block manager; they must
    # be the very tables, lengths, slots and pairs the product allocator makes
    sys.path.insert(0, ROOT)
    import bench
    from paged_kv_cache_127_gb300 import binding as pa
    from paged_kv_cache_127_gb300 import workloads
    a = workloads.build_step(name, seed=0, values=False, binding=pa)
    b = workloads.build_step(name, seed=0, values=False, binding=bench._OracleAllocator)
    for f in ("tables", "lens", "slots", "pairs", "free_order"):
        np.testing.assert_array_equal(getattr(a, f), getattr(b, f), err_msg=f)
    assert a.num_blocks == b.num_blocks and a.max_blocks == b.max_blocks


def test_prefix_cache_mode_bounds_its_repetitions(monkeypatch):
    # host-only mode: the default --steps (sized for the decode bench) must not
    # repeat the whole request stream thousands of times
    sys.path.insert(0, ROOT)
    import bench
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        monkeypatch.delenv(k, raising=False)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--prefix-requests", "300", "--steps", "5000", "--warmup", "50", "--no-cpu-baseline"])
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["steps"] == 5 and line["unit"] == "requests/s" and line["value"] > 0
    assert line["gpu_launches"] == 0



def test_profiled_traffic_follows_the_kernel_sources(tmp_path, monkeypatch):
    # roofline.traffic comes from an ncu summary only while the kernel sources hash
    # to the value recorded in it; any edit to them makes it null
    sys.path.insert(0, ROOT)
    import bench
    fake = tmp_path / "repo"
    (fake / "profiles").mkdir(parents=True)
    (fake / "paged_kv_cache_127_gb300" / "csrc").mkdir(parents=True)
    for name in set(bench.KERNEL_SOURCES):
        data = open(os.path.join(ROOT, "paged_kv_cache_127_gb300", "csrc", name), "rb").read()
        (fake / "paged_kv_cache_127_gb300" / "csrc" / name).write_bytes(data)
    monkeypatch.setattr(bench, "ROOT", str(fake))
    (fake / "profiles" / "decode_w.md").write_text(
        f"# decode, workload w\n\ntraffic_bytes_per_launch: 123456 sources: {bench.kernel_source_hash()}\n")
    assert bench.profiled_traffic("w") == 123456
    assert bench.profiled_traffic("w", "chunk") is None            # no chunk summary for w
    assert bench.profiled_traffic("no_such_workload") is None
    edited = fake / "paged_kv_cache_127_gb300" / "csrc" / bench.KERNEL_SOURCES[0]
    edited.write_bytes(edited.read_bytes() + b"\n// edited\n")
    assert bench.profiled_traffic("w") is None


def test_clock_sampler_reports_median_clock_and_throttle_reasons(tmp_path, monkeypatch):
    # a stand-in nvidia-smi prints three samples in the queried column order
    # (index, sm, max sm, power, active mask, hw, hw thermal, sw thermal, sw power cap)
    fake = tmp_path / "nvidia-smi"
    fake.write_text("#!/bin/bash\n"
                    "printf '0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active\\n'\n"
                    "printf '0, 1965, 2070, 1390.5, 0x4, Not Active, Not Active, Not Active, Active\\n'\n"
                    "printf '0, 1800, 2070, 1400.0, 0x8, Active, Not Active, Not Active, Active\\n'\n"
                    "printf '[N/A], [N/A]\\n'\n"
                    "exec sleep 30\n")
    fake.chmod(0o755)
    monkeypatch.setenv("PATH", f"{tmp_path}:{os.environ['PATH']}")
    sys.path.insert(0, ROOT)
    import time

    import bench
    s = bench.ClockSampler(0).start()
    for _ in range(100):                      # until the three samples are written
        time.sleep(0.05)
        if os.path.exists(s.path) and open(s.path).read().count("\n") >= 4:
            break
    got = s.stop()
    assert got == {"sm_mhz": 1965.0, "sm_max_mhz": 2070.0, "reasons": ["hw_slowdown", "sw_power_cap"], "samples": 3}
    assert not os.path.exists(s.path)


def test_roofline_peaks_come_from_the_measured_file_else_the_fallback(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_hbm_peak() == (6800.0, "fallback")
    assert bench.measured_bf16_peak() == (1900.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6698.2, "bf16_tflops": 1883.0}))
    assert bench.measured_hbm_peak() == (6698.2, "measured")
    assert bench.measured_bf16_peak()[0] == 1883.0
