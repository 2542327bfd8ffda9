"""The carry chain's folded rise (csrc/cr_chain_map.h, built here for the host
with g++; CPU only): a rise by d binades folded into a map 2^j M + b[p]
equals the rise applied after the map, for every d <= j <= 7 and both
parities of M. The expected value is computed with exact integers: the
chain's sum in the old unit is A + f (A an integer, f = 0 or 0 < f < 1), and
the rise rounds (A + f) / 2^d to the nearest integer, ties to even."""
import ctypes
import os
import random
import subprocess

import pytest

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "scan_canonical_reduce_gb300", "csrc")
SHIM = r"""
#include "cr_chain_map.h"
extern "C" int fold_apply(uint64_t a, uint64_t b0, uint64_t b1, int d, int64_t q, int fpos,
                          uint64_t M, uint64_t* out) {
  const cr::Map g{a, b0, b1};
  if (!cr::rise_foldable(g, d)) return 0;
  *out = cr::apply(cr::fold_rise(g, d, q, fpos != 0), M);
  return 1;
}
"""
U64 = (1 << 64) - 1


@pytest.fixture(scope="module")
def lib(tmp_path_factory):
    tmp = tmp_path_factory.mktemp("fold")
    src, so = os.path.join(tmp, "shim.cpp"), os.path.join(tmp, "shim.so")
    with open(src, "w") as f:
        f.write(SHIM)
    subprocess.run(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-I", CSRC, src, "-o", so],
                   check=True)
    L = ctypes.CDLL(so)
    L.fold_apply.restype = ctypes.c_int
    L.fold_apply.argtypes = [ctypes.c_uint64] * 3 + [ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                                     ctypes.c_uint64,
                                                     ctypes.POINTER(ctypes.c_uint64)]
    return L


def signed(v):
    v &= U64
    return v - (1 << 64) if v >> 63 else v


def rise(A, fpos, d):
    """Round (A + f) / 2^d to nearest, ties to even; f = 0 unless fpos, when
    0 < f < 1 (so (A + f) / 2^d is never a tie)."""
    Q, r = A >> d, A & ((1 << d) - 1)
    half = 1 << (d - 1)
    up = r >= half if fpos else (r > half or (r == half and Q & 1))
    return Q + (1 if up else 0)


def call(lib, a, b0, b1, d, q, fpos, M):
    out = ctypes.c_uint64(0)
    ok = lib.fold_apply(a & U64, b0 & U64, b1 & U64, d, q, int(fpos), M & U64, ctypes.byref(out))
    return ok, signed(out.value)


def test_fold_equals_rise_after_map(lib):
    rng = random.Random(20260)
    n = 0
    for _ in range(20000):
        j = rng.randint(1, 7)
        d = rng.randint(1, j)
        sign = lambda: rng.choice((-1, 1))  # noqa: E731
        m_in = sign() * ((1 << 52) | rng.getrandbits(52))   # entry M of a valid chain
        m_prev = sign() * ((1 << 52) | rng.getrandbits(52))  # M after the map
        b = m_prev - (m_in << j)  # the map's true offset for that entry
        bo = b + rng.randint(-2, 2)  # the other parity's offset (ties seen differently)
        b0, b1 = (bo, b) if m_in & 1 else (b, bo)
        q = sign() * rng.getrandbits(52 + d)  # T in the old unit: A stays below 2^(53+d)
        fpos = rng.random() < 0.5
        for M in (m_in, m_in + 1):  # both parities
            bp = b1 if M & 1 else b0
            want = rise((M << j) + bp + q, fpos, d)
            ok, got = call(lib, 1 << j, b0, b1, d, q, fpos, M)
            assert ok
            assert got == want, (j, d, q, fpos, M, got, want)
            n += 1
    assert n == 40000


def test_ties_at_the_rounding_point(lib):
    """A exactly halfway between two multiples of 2^d: ties go to even."""
    for j in range(1, 8):
        for d in range(1, j + 1):
            for M in (5, 6, -5, -6, (1 << 52) + 3):
                for k in range(-4, 5):
                    A_target = ((M << (j - d)) + k) * (1 << d) + (1 << (d - 1))  # a tie
                    b = A_target - (M << j)
                    want = rise(A_target, False, d)
                    ok, got = call(lib, 1 << j, b, b, d, 0, False, M)
                    assert ok and got == want, (j, d, M, k, got, want)
                    assert got % 2 == 0  # to even


@pytest.mark.parametrize("j", range(0, 11))
def test_foldable_limits(lib, j):
    for d in range(1, 9):
        ok, _ = call(lib, 1 << j, 0, 0, d, 0, False, 0)
        assert ok == (d <= j <= 7), (j, d)
    assert call(lib, 0, 0, 0, 1, 0, False, 0)[0] == 0       # a multiplier 2^64 = 0
    assert call(lib, 12, 0, 0, 1, 0, False, 0)[0] == 0      # not a power of two
