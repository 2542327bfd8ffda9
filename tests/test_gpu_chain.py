"""The exact parallel left fold (block_dyadic carries, 1-D left_fold) against
the oracle's serial fold, 0 ULP, on inputs chosen to stress it: frequent
zero crossings, ties at the chain's unit, binade jumps of many orders,
cancellation to exact zeros, signed zeros, subnormals, non-finite values,
monotone growth through every power of two; in place; and inputs whose
breaks overflow the segment buffer (device-side serial fallback)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def scr():
    import scan_canonical_reduce_gb300 as m
    return m


def same_bits_nan_as_class(got, want):
    """Raw-bit equality, except that NaNs compare as a class (payloads differ
    between x86 and the GPU's canonical NaN)."""
    iv = np.uint64 if got.dtype == np.float64 else np.uint32
    gn, wn = np.isnan(got), np.isnan(want)
    diff = (got.view(iv) != want.view(iv)) & ~(gn & wn)
    return np.nonzero(diff | (gn != wn))[0]


def check_fold(scr, x, inplace=False):
    t = torch.from_numpy(x).to(DEV)
    got = (scr.inclusive_scan(t, "left_fold", out=t) if inplace
           else scr.inclusive_scan(t, "left_fold")).cpu().numpy()
    want = oracle.scan(x, "left_fold")
    d = same_bits_nan_as_class(got, want)
    if d.size:
        raise AssertionError("first diff at %d of %d (%d diffs): got %r want %r" %
                             (d[0], x.size, d.size, got[d[0]], want[d[0]]))


def u(n, seed):
    return W.uniform_pm1(n, seed)


CASES = {
    "uniform_pm1": lambda n, dt: u(n, 11).astype(dt),
    "uniform_pm1_small": lambda n, dt: (u(n, 12) * 1e-3).astype(dt),
    "positive_growth": lambda n, dt: (np.abs(u(n, 13)) + 0.5).astype(dt),
    "wide_exponents": lambda n, dt: W.signed_pow2(n, 14, dt, -40, 40),
    "drift_and_cross": lambda n, dt: (u(n, 15) + 0.001 * np.sin(np.arange(n) / 5000.0)).astype(dt),
    "constant_tenth": lambda n, dt: np.full(n, 0.1, dtype=dt),
    "halves_ties": lambda n, dt: (np.round(u(n, 16) * 64) / 128 + 2.0 ** 20 * (np.arange(n) == 0)
                                  ).astype(dt),
    "cancel_to_zero": lambda n, dt: np.where(np.arange(n) % 2 == 0, 1.0, -1.0).astype(dt)
    * (np.arange(n) // 2 % 7 + 1),
    "big_small_mix": lambda n, dt: np.where(np.arange(n) % 97 == 0, 1e12, 1.0).astype(dt)
    * u(n, 17).astype(dt),
    # one large first value, then small steps that never change its binade:
    # long runs of tiles without any break
    "big_then_small": lambda n, dt: np.where(np.arange(n) == 0, 2.0 ** 30,
                                             np.abs(u(n, 18)) * 1e-3).astype(dt),
}


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("case", sorted(CASES))
def test_left_fold_adversarial(scr, dtype, case):
    for n in (1000, 5000, 2048 * 9 + 3, 300007):
        x = np.ascontiguousarray(CASES[case](n, dtype))
        check_fold(scr, x)


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_left_fold_special_values(scr, dtype):
    n = 20000
    x = u(n, 21).astype(dtype)
    x[5000] = np.inf
    check_fold(scr, x)
    x = u(n, 22).astype(dtype)
    x[7000] = np.nan
    check_fold(scr, x)
    z = np.full(n, -0.0, dtype=dtype)
    check_fold(scr, z)
    tiny = (u(n, 23) * (1e-310 if dtype == np.float64 else 1e-40)).astype(dtype)
    check_fold(scr, tiny)
    huge = (u(n, 24) * (1e307 if dtype == np.float64 else 1e37)).astype(dtype)
    check_fold(scr, huge)


def test_left_fold_in_place_and_large(scr):
    x = u((1 << 22) + 17, 31)
    check_fold(scr, x, inplace=True)
    check_fold(scr, W.family3(1 << 24))


@pytest.mark.parametrize("B", [2, 16, 256])
def test_block_dyadic_carries_adversarial(scr, B):
    for case in ("wide_exponents", "drift_and_cross", "cancel_to_zero", "big_small_mix"):
        x = np.ascontiguousarray(CASES[case](B * 3001 + 5, np.float64))
        got = scr.inclusive_scan(torch.from_numpy(x).to(DEV), "block_dyadic", B).cpu().numpy()
        want = oracle.scan(x, "block_dyadic", B)
        assert got.tobytes() == want.tobytes(), (case, B)
