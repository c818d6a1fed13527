"""Compile the C oracle into ``oracle/libnf4oracle.so``.

Test infrastructure only: the tests, the package smoke check and the
benchmark's CPU-baseline leg load the result.  Plain ``gcc`` with
``-ffp-contract=off`` so that no multiply-add is fused on either x86-64 or
aarch64 hosts.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "nf4_oracle.c")
HDR = os.path.join(HERE, "nf4_oracle.h")
LIB = os.path.join(HERE, "libnf4oracle.so")

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
          "-fPIC", "-shared", "-Wall", "-Wextra"]


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in (SRC, HDR, __file__))


def build_oracle(force: bool = False) -> str:
    """Build the shared library if it is missing or older than its sources."""
    if force or is_stale():
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", *CFLAGS, "-o", tmp, SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force="--force" in sys.argv))
