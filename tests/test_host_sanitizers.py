"""Host code under AddressSanitizer and UndefinedBehaviorSanitizer.

Two drivers in tests/native are built with -fsanitize=address,undefined and
run on seeded random inputs (no GPU involved):

- host_stress.cpp drives the block allocator, copy-on-write, batched appends,
  fault injection, swap pools and the prefix cache (the allocator's C++
  sources linked directly), checking after every operation that refcounts
  equal the blocks the live tables and the cache hold and that the free count
  equals the blocks at refcount 0;
- oracle_stress.c drives every entry point of the CPU oracle, checking the
  partitioned decode against the plain one, the last query of a chunk against
  a decode, the cache operations' effects, and that bad inputs are refused.

A memory error or undefined behaviour aborts the driver (-fno-sanitize-recover).
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
NATIVE = os.path.join(ROOT, "tests", "native")
CSRC = os.path.join(ROOT, "paged_kv_cache_127_gb300", "csrc")
SAN = ["-O1", "-g", "-fsanitize=address,undefined", "-fno-sanitize-recover=all", "-fno-omit-frame-pointer"]


def _build(tmp_path, compiler, args, name):
    exe = shutil.which(compiler)
    if not exe:
        pytest.skip(f"{compiler} not found")
    probe = tmp_path / "probe.c"
    probe.write_text("int main(void) { return 0; }\n")
    if subprocess.run([exe, *SAN, "-x", "c", str(probe), "-o", str(tmp_path / "probe")],
                      capture_output=True).returncode != 0:
        pytest.skip("sanitizer runtime not available")
    out = tmp_path / name
    r = subprocess.run([exe, *SAN, *args, "-o", str(out)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    return str(out)


def _run(exe, *args):
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1:abort_on_error=0", UBSAN_OPTIONS="print_stacktrace=1")
    r = subprocess.run([exe, *map(str, args)], capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, (r.stdout + r.stderr)[-4000:]
    return r.stdout


@pytest.fixture(scope="module")
def host_stress(tmp_path_factory):
    d = tmp_path_factory.mktemp("host_stress")
    return _build(d, "g++", ["-std=c++17", f"-I{os.path.join(ROOT, 'include')}",
                             os.path.join(NATIVE, "host_stress.cpp"), os.path.join(CSRC, "pa_alloc.cpp"),
                             os.path.join(CSRC, "pa_prefix.cpp")], "host_stress")


@pytest.fixture(scope="module")
def oracle_stress(tmp_path_factory):
    d = tmp_path_factory.mktemp("oracle_stress")
    return _build(d, "gcc", ["-std=c11", "-ffp-contract=off", os.path.join(ROOT, "oracle", "pa_oracle.c"),
                             os.path.join(NATIVE, "oracle_stress.c"), "-lm"], "oracle_stress")


@pytest.mark.parametrize("seed", [1, 2, 3, 4, 6, 12])
def test_allocator_and_prefix_cache_under_sanitizers(host_stress, seed):
    # seeds cover block sizes 1, 2, 4 and 16 (copy-on-write needs B > 1)
    out = _run(host_stress, seed, 20000)
    assert "0 failures" in out


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_oracle_under_sanitizers(oracle_stress, seed):
    out = _run(oracle_stress, seed, 200)
    assert "0 failures" in out
