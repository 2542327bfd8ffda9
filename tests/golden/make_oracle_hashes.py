"""Writes oracle_hashes.txt: SHA-256 of oracle outputs on fixed inputs.

Mirrors the cross-platform witness on "Canonical Parallel Reduction and Scan"
(P4229R0 Key results, Appendix F: bit-identical scan output hashes across
x86-64, AArch64 and CUDA under a matched FP environment). The file is written
on one platform and re-checked on the others by tests/test_oracle_xplat.py.
Calls only the oracle and the input generators (bit-built inputs, no libm).

Usage: python tests/golden/make_oracle_hashes.py
"""
import hashlib
import os
import platform
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import workloads as W  # noqa: E402

N = (1 << 16) + 37


def cases():
    """(name, bytes) of every witnessed oracle output."""
    x64 = W.family2(N, np.float64)
    x32 = W.family2(N, np.float32)
    for L in (1, 16, 128, 1024):
        yield "reduce f64 L=%d" % L, oracle.reduce(x64, L, 0.0).tobytes()
        yield "reduce f32 L=%d" % L, oracle.reduce(x32, L, np.float32(0.0)).tobytes()
    x3 = W.family3(N)
    for policy, B in (("left_fold", 1), ("pairwise", 1), ("iterated_pairwise", 1),
                      ("block_dyadic", 16), ("block_dyadic", 256)):
        yield "scan f64 %s B=%d" % (policy, B), oracle.scan(x3, policy, B).tobytes()
        yield "scan f32 %s B=%d" % (policy, B), \
            oracle.scan(x3.astype(np.float32), policy, B).tobytes()
    rows, cols = 64, 4096 + 5
    xb = W.family2(rows * cols, np.float32)
    yield "reduce_batched f32 L=128", oracle.reduce_batched(xb, rows, cols, 1, cols, 128,
                                                            np.float32(0.0)).tobytes()
    xc = W.family2(90 * 1001, np.float64)
    yield "scan_batched f64 block_dyadic B=16", \
        oracle.scan_batched(xc, 1001, 90, 1001, 1, "block_dyadic", 16).tobytes()


def digest_lines():
    return ["%s : %s" % (name, hashlib.sha256(b).hexdigest()) for name, b in cases()]


if __name__ == "__main__":
    out = os.path.join(HERE, "oracle_hashes.txt")
    with open(out, "w") as f:
        f.write("# SHA-256 of oracle outputs; written on %s by make_oracle_hashes.py\n"
                % platform.machine())
        for line in digest_lines():
            f.write(line + "\n")
    print(out)
