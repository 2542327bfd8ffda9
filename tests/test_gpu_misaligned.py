"""Inputs and outputs that start one element into an allocation (aligned to
the element, not to 16 bytes: the kernels' vector accesses fall back to
scalar ones there). Every scan policy and kernel path, the shifted forms,
reduce<E>, against the oracle at 0 ULP."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

POLICIES = [("iterated_pairwise", 1), ("pairwise", 1), ("left_fold", 1), ("block_dyadic", 2),
            ("block_dyadic", 16), ("block_dyadic", 256), ("block_dyadic", 4096)]


@pytest.fixture(scope="module")
def scr():
    import scan_canonical_reduce_gb300 as m
    return m


def bits(a):
    return np.asarray(a).tobytes()


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("policy,B", POLICIES)
def test_misaligned_scan(scr, dtype, policy, B):
    tdt = torch.float64 if dtype == np.float64 else torch.float32
    for n in (2048 * 5 + 3, 16 * 20000 + 7):
        x = W.signed_pow2(n, W.seed_for(35, n % 89), dtype, -20, 20)
        xb = torch.zeros(n + 1, dtype=tdt, device=DEV)
        xb[1:] = torch.from_numpy(x).to(DEV)
        ob = torch.full((n + 2,), float("nan"), dtype=tdt, device=DEV)
        xs, os_ = xb[1:], ob[1:n + 1]
        assert xs.data_ptr() % 16 != 0 and os_.data_ptr() % 16 != 0
        scr.inclusive_scan(xs, policy, B, out=os_)
        got = ob.cpu().numpy()
        assert bits(got[1:n + 1]) == bits(oracle.scan(x, policy, B)), (n, policy, B)
        assert np.isnan(got[0]) and np.isnan(got[n + 1])  # nothing written outside


@pytest.mark.parametrize("mode", ["exclusive", "include_initial"])
@pytest.mark.parametrize("policy,B", [("iterated_pairwise", 1), ("block_dyadic", 16),
                                      ("left_fold", 1)])
def test_misaligned_shifted(scr, mode, policy, B):
    n = 2048 * 7 + 5
    x = W.family3(n)
    xb = torch.zeros(n + 1, dtype=torch.float64, device=DEV)
    xb[1:] = torch.from_numpy(x).to(DEV)
    m = n + 1 if mode == "include_initial" else n
    ob = torch.zeros(m + 1, dtype=torch.float64, device=DEV)
    f = scr.exclusive_scan if mode == "exclusive" else scr.scan_include_initial
    f(xb[1:], policy, B, 0.5, out=ob[1:])
    assert bits(ob[1:].cpu().numpy()) == bits(oracle.scan_ex(x, policy, B, 0.5, mode))


@pytest.mark.parametrize("policy,B", [("left_fold", 1), ("block_dyadic", 16), ("pairwise", 1)])
def test_misaligned_reduce_policy(scr, policy, B):
    n = 16 * 5000 + 3
    x = W.family3(n)
    xb = torch.zeros(n + 1, dtype=torch.float64, device=DEV)
    xb[1:] = torch.from_numpy(x).to(DEV)
    got = scr.reduce_policy(xb[1:], policy, B).cpu().numpy()[0]
    assert bits(np.array([got])) == bits(np.array([oracle.reduce_policy(x, policy, B)]))
