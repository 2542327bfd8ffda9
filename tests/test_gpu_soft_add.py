"""libcr's integer-pipe binary64 add (a measured alternative to the FP64
pipe, exposed through cr_add_pairs_int; the kernels do not use it):
bit-for-bit equal to IEEE-754 round-to-nearest-even addition (numpy on the
host), NaNs compared as a class."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def scr():
    import scan_canonical_reduce_gb300 as m
    return m


def check(scr, a, b):
    got = scr.add_pairs_int(torch.from_numpy(a).to(DEV), torch.from_numpy(b).to(DEV)).cpu().numpy()
    with np.errstate(all="ignore"):
        want = a + b
    gn, wn = np.isnan(got), np.isnan(want)
    bad = ((got.view(np.uint64) != want.view(np.uint64)) & ~(gn & wn)) | (gn != wn)
    idx = np.nonzero(bad)[0]
    assert idx.size == 0, "%d mismatches, first a=%r b=%r got=%r want=%r" % (
        idx.size, a[idx[0]], b[idx[0]], got[idx[0]], want[idx[0]])


def bits(n, seed):
    return W.splitmix64(seed, 0, n)


def test_random_bit_patterns(scr):
    n = 1 << 22
    check(scr, bits(n, 1).view(np.float64), bits(n, 2).view(np.float64))


@pytest.mark.parametrize("gap", list(range(0, 71)))
def test_exponent_gaps_and_signs(scr, gap):
    n = 1 << 16
    u = bits(n, 100 + gap)
    v = bits(n, 200 + gap)
    ea = (u >> np.uint64(53)) % np.uint64(1800) + np.uint64(120)      # normal exponents
    eb = ea - np.uint64(gap)
    a = ((u & np.uint64(1 << 63)) | (ea << np.uint64(52)) | (u & np.uint64((1 << 52) - 1)))
    b = ((v & np.uint64(1 << 63)) | (eb << np.uint64(52)) | (v & np.uint64((1 << 52) - 1)))
    check(scr, a.view(np.float64), b.view(np.float64))
    check(scr, b.view(np.float64), a.view(np.float64))


def test_near_cancellation_and_ties(scr):
    n = 1 << 18
    a = W.signed_pow2(n, 7, np.float64, -300, 300)
    k = (bits(n, 8) % np.uint64(64)).astype(np.int64) - 32
    b = -(a.view(np.int64) + k).view(np.float64)          # |b| within 32 ulps of |a|
    check(scr, a, b)
    # exact ties: b = half an ulp of a (times an odd factor below a's ulp)
    ulp = np.spacing(np.abs(a))
    check(scr, a, ulp / 2)
    check(scr, a, -ulp / 2)
    check(scr, a, ulp * 1.5)
    check(scr, a, ulp / 2 + ulp / 2 ** 30)
    check(scr, np.full(8, 1.0), np.array([2.0 ** -53, -2.0 ** -54, 2.0 ** -53 * 3, 1.0,
                                          -1.0, 2.0 ** 53, -2.0 ** 52, 0.5]))


def test_special_values(scr):
    big, tiny = np.finfo(np.float64).max, np.finfo(np.float64).tiny
    vals = np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, np.nan, big, -big, tiny, -tiny,
                     tiny / 3, -tiny / 7, 5e-324, -5e-324, 1.5 * tiny, 2.0 ** 1023, 1e308,
                     -1e308, 3.0], dtype=np.float64)
    a = np.repeat(vals, vals.size)
    b = np.tile(vals, vals.size)
    check(scr, a, b)
    # results just below the normal range
    x = tiny * (1 + np.arange(1, 1000) / 1e3)
    check(scr, x, -tiny * np.ones_like(x))
    # overflow
    check(scr, np.full(5, big), np.array([big, big / 2, big * 2 ** -52, 1e292, -big]))


def test_int_add_rate(scr):
    rate = scr.measure_int_add_rate(DEV)
    hw, _ = scr.measure_add_peak(torch.float64, DEV)
    print("integer-pipe fp64 adds/s %.3e, hardware %.3e" % (rate, hw))
    assert rate > 0
