"""Cross-platform witness of the oracle: the same SHA-256 of its outputs on
every platform (the method of the cross-platform witness on "Canonical
Parallel Reduction and Scan", P4229R0 Key results / Appendix F). The stored
hashes were written by tests/golden/make_oracle_hashes.py; the gpu-marked
twin repeats the check where the GPU tests run (the aarch64 host of the
GB300), so both instruction sets are covered."""
import os
import platform

import pytest

from tests.golden import make_oracle_hashes as M

HERE = os.path.join(os.path.dirname(__file__), "golden", "oracle_hashes.txt")


def _check():
    with open(HERE) as f:
        want = [l.rstrip("\n") for l in f if l.strip() and not l.startswith("#")]
    got = M.digest_lines()
    assert got == want, "oracle output differs on %s" % platform.machine()


def test_oracle_hashes_match_stored():
    _check()


@pytest.mark.gpu
def test_oracle_hashes_match_stored_on_gpu_host():
    _check()
