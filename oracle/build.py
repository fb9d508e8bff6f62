"""Compile the C oracle (test infrastructure) into oracle/_build/liboracle.so.

Plain gcc, no fused multiply-add contraction, so the fp64 results are the same
on x86-64 and Arm hosts.  Building the checker is not using it: the product
build step may call this, but only tests, the smoke check and the benchmark's
CPU-baseline leg may load the result.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "pa_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIBRARY = os.path.join(BUILD_DIR, "liboracle.so")


def build(force: bool = False) -> str:
    """Build liboracle.so if missing or older than its source; return its path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(LIBRARY)
            and os.path.getmtime(LIBRARY) >= os.path.getmtime(SOURCE)):
        return LIBRARY
    tmp = LIBRARY + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
           "-Wall", "-Wextra", SOURCE, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force=True))
