"""Compile the C oracle into ``oracle/libls_oracle.so``.

The oracle is test infrastructure; building it is part of the repository's
build step so that the checker exists on every machine the tests run on.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ls_oracle.c")
LIB = os.path.join(HERE, "libls_oracle.so")


def build_oracle(force: bool = False, verbose: bool = False) -> str:
    """Build the oracle shared library if it is missing or stale; return its path."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    # -ffp-contract=off: no fused multiply-add contraction, so that x86 and
    # aarch64 hosts produce the same double results.  No -ffast-math: the FP32
    # quantization decision relies on IEEE division and rintf.
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wextra",
           SRC, "-o", tmp, "-lm"]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force=True, verbose=True))
