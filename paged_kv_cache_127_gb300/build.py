"""Build libpa.so (CUDA kernels for sm_103a + C-ABI + host allocator) in-tree.

    python -m paged_kv_cache_127_gb300.build [--force] [--verbose]

Each translation unit is compiled by its own nvcc process, in parallel, with a
single ``-gencode arch=compute_103a,code=sm_103a``; the objects are linked into
``paged_kv_cache_127_gb300/_build/libpa.so`` with the CUDA runtime linked
statically, so the library has no dependency on a particular libcudart.
Rebuilds only what is older than its sources or headers.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIBRARY = os.path.join(BUILD, "libpa.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", f"-I{INCLUDE}"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpa")


def _headers():
    return (glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout.strip() or r.stderr.strip()):
        print(r.stdout + r.stderr, flush=True)
    return r


def _switches():
    """Build-time kernel switches taken from the environment: PA_DECODE_CUDA_CORE=1
    builds the 16-bit decode with q.k and p.v on the CUDA cores instead of the
    tensor cores (an alternative for comparing the two; the default is off)."""
    flags = []
    if os.environ.get("PA_DECODE_CUDA_CORE", "0") not in ("", "0"):
        flags.append("-DPA_DECODE_CUDA_CORE=1")
    return flags


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile and link libpa.so; return its path."""
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    extra_flags = [*extra_flags, *_switches()]
    # a change of switches rebuilds everything
    stamp = os.path.join(BUILD, "switches.txt")
    want = " ".join(_switches())
    have = open(stamp).read() if os.path.exists(stamp) else None
    if have != want:
        force = True
    headers = _headers()
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    jobs = []
    objects = []
    for src in sources:
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        objects.append(obj)
        if force or _stale(obj, [src, __file__] + headers):
            if src.endswith(".cu"):
                cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
            else:
                cmd = [nvcc, "-O2", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
                       f"-I{INCLUDE}", "-x", "c++", "-c", src, "-o", obj]
            jobs.append(cmd)
    if jobs:
        workers = min(len(jobs), max(1, os.cpu_count() or 1))
        with cf.ThreadPoolExecutor(workers) as ex:
            for f in [ex.submit(_run, cmd, verbose) for cmd in jobs]:
                f.result()
    if force or jobs or _stale(LIBRARY, objects):
        tmp = LIBRARY + f".tmp{os.getpid()}"
        _run([nvcc, *ARCH, "-shared", "-cudart", "static", *objects, "-o", tmp], verbose)
        os.replace(tmp, LIBRARY)
    with open(stamp, "w") as f:
        f.write(want)
    return LIBRARY


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true", help="print register / smem usage (-Xptxas -v)")
    args = ap.parse_args()
    extra = ["-Xptxas", "-v"] if args.ptxas_info else []
    print(build(force=args.force or args.ptxas_info, verbose=args.verbose or args.ptxas_info, extra_flags=extra))


if __name__ == "__main__":
    main()
