"""All-(-0.0) inputs through every call: an add gives -0.0 only from two -0.0
operands, so every result must be -0.0 (or init op -0.0). A padding value
of +0.0 that reached an add anywhere on a kept path (a ragged tile, block or
lane, a chain's last group) would show as a +0.0. Against the oracle, raw
bits."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SIZES = [1, 2, 3, 17, 2048 * 3 + 5, 16 * 70000 + 3]
POLICIES = [("left_fold", 1), ("iterated_pairwise", 1), ("pairwise", 1), ("block_dyadic", 2),
            ("block_dyadic", 16), ("block_dyadic", 256), ("block_dyadic", 4096)]


@pytest.fixture(scope="module")
def scr():
    import scan_canonical_reduce_gb300 as m
    return m


def same(got, want):
    return np.asarray(got).tobytes() == np.asarray(want).tobytes()


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("n", SIZES)
def test_reduce_minus_zero(scr, dtype, n):
    x = np.full(n, -0.0, dtype=dtype)
    t = torch.from_numpy(x).to(DEV)
    for L in (1, 16, 128, 1024):
        for init in (-0.0, 0.0):
            got = scr.reduce(t, L, init).cpu().numpy()[0]
            want = oracle.reduce(x, L, dtype(init))
            assert same(np.array([got]), np.array([want])), (n, L, init, got, want)


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("policy,B", POLICIES)
@pytest.mark.parametrize("n", SIZES)
def test_scans_minus_zero(scr, dtype, policy, B, n):
    x = np.full(n, -0.0, dtype=dtype)
    t = torch.from_numpy(x).to(DEV)
    got = scr.inclusive_scan(t, policy, B).cpu().numpy()
    assert same(got, oracle.scan(x, policy, B)), (n, policy, B)
    r = scr.reduce_policy(t, policy, B).cpu().numpy()[0]
    assert same(np.array([r]), np.array([oracle.reduce_policy(x, policy, B)])), (n, policy, B)
    for mode, f in (("exclusive", scr.exclusive_scan), ("include_initial", scr.scan_include_initial)):
        got = f(t, policy, B, -0.0).cpu().numpy()
        assert same(got, oracle.scan_ex(x, policy, B, dtype(-0.0), mode)), (n, policy, B, mode)
