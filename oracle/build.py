"""Builds the oracle's shared library (test infrastructure only).

The oracle is a plain single-threaded C++ evaluator used by the tests, by
``__graft_entry__.smoke()`` and by the CPU-baseline leg of ``bench.py``; the
CUDA library never links it. Built with the FP environment that the
canonical-reduce page states for its cross-platform witness: no floating-point
contraction and no fast-math.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "cro.cpp")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libcro.so")

CXXFLAGS = [
    "-O2", "-std=c++17", "-fPIC", "-shared",
    "-ffp-contract=off", "-fno-fast-math", "-fexcess-precision=standard",
]


def build(force: bool = False) -> str:
    """Compile ``cro.cpp`` into ``_build/libcro.so`` if it is missing or stale."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["g++", *CXXFLAGS, SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
