"""Long binary32 carry chains through the exact parallel evaluation: the
1-D left fold and the block_dyadic carries, classified against the
estimated chain with a statistical margin, every step still checked exactly
(a failed check sends the chain to the serial fold). 0 ULP against the
oracle at the benchmark size and on value families whose rounding is
unbiased (the estimate holds) or biased (the checks fail and the serial
fold takes over), and a check that the benchmark family needs no recovery."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
RECOVERY = ("chain_fallback_kernel", "scan_local_again_kernel", "fixup_again_kernel")


@pytest.fixture(scope="module")
def scr():
    import scan_canonical_reduce_gb300 as m
    return m


def first_diff(a, b):
    idx = np.nonzero(a.view(np.uint32) != b.view(np.uint32))[0]
    return None if idx.size == 0 else (int(idx[0]), int(idx.size))


def f32(x):
    return np.ascontiguousarray(x.astype(np.float32))


FAMILIES = {
    "uniform_pm1": lambda n: f32(W.uniform_pm1(n, W.seed_for(36, 1))),
    "normal": lambda n: f32(W.standard_normal(n, W.seed_for(36, 2))),
    "signed_pow2": lambda n: W.signed_pow2(n, W.seed_for(36, 3), np.float32, -20, 20),
    "uniform01": lambda n: f32(W.uniform01(n, W.seed_for(36, 4))),
    "lognormal": lambda n: f32(W.lognormal(n, W.seed_for(36, 5))),
    "one_plus_tiny": lambda n: f32(1.0 + W.uniform01(n, W.seed_for(36, 6)) * 2.0 ** -7),
}


@pytest.mark.parametrize("family", sorted(FAMILIES))
@pytest.mark.parametrize("policy,B", [("left_fold", 1), ("block_dyadic", 16)])
def test_families(scr, family, policy, B):
    """2^22 + 3 elements (left fold: 2^22 steps; block_dyadic<16>: 2^18 carries)."""
    x = FAMILIES[family]((1 << 22) + 3)
    got = scr.inclusive_scan(torch.from_numpy(x).to(DEV), policy, B).cpu().numpy()
    want = oracle.scan(x, policy, B)
    assert first_diff(got, want) is None, (family, policy, first_diff(got, want))


@pytest.mark.parametrize("policy,B", [("block_dyadic", 16), ("block_dyadic", 256),
                                      ("left_fold", 1)])
def test_full_size(scr, policy, B):
    """The benchmark's 1-D scan input rounded to binary32, n = 2^28: every
    element against the oracle."""
    x = f32(W.family3(1 << 28))
    got = scr.inclusive_scan(torch.from_numpy(x).to(DEV), policy, B).cpu().numpy()
    want = oracle.scan(x, policy, B)
    assert first_diff(got, want) is None, (policy, B, first_diff(got, want))


@pytest.mark.parametrize("policy,B,n", [("block_dyadic", 16, 1 << 28),
                                        ("block_dyadic", 256, 1 << 28),
                                        ("left_fold", 1, 1 << 28)])
def test_needs_no_recovery(scr, policy, B, n):
    """On the benchmark family every binary32 step validates: the recovery
    kernels read the chain's flag and return at once."""
    x = torch.from_numpy(f32(W.family3(n))).to(DEV)
    y = torch.empty_like(x)
    scr.inclusive_scan(x, policy, B, out=y)
    torch.cuda.synchronize()
    scr.profile_enable(True)
    scr.inclusive_scan(x, policy, B, out=y)
    torch.cuda.synchronize()
    scr.profile_enable(False)
    prof = scr.profile_collect()
    rec = [(k, ms) for k, ms in prof if k in RECOVERY]
    assert rec, prof
    assert all(ms < 0.5 for _, ms in rec), rec


@pytest.mark.parametrize("policy,B", [("left_fold", 1), ("block_dyadic", 16),
                                      ("block_dyadic", 4)])
def test_reduce_policy_and_shifted_forms(scr, policy, B):
    """reduce<E> (the chain's last value, no prefix written) and the
    exclusive / include_initial scans of the binary32 chains."""
    x = f32(W.family3((1 << 24) + 7))
    xd = torch.from_numpy(x).to(DEV)
    got = scr.reduce_policy(xd, policy, B).cpu().numpy()[0]
    assert got.tobytes() == np.asarray(oracle.reduce_policy(x, policy, B)).tobytes()
    for form, fn in (("exclusive", scr.exclusive_scan),
                     ("include_initial", scr.scan_include_initial)):
        got = fn(xd, policy, B, 0.375).cpu().numpy()
        want = oracle.scan_ex(x, policy, B, np.float32(0.375), form)
        assert first_diff(got, want) is None, (form, first_diff(got, want))


def test_in_place_and_host(scr):
    """In place (the chain reads a copy of its input) and from host buffers
    (carries folded chunk by chunk)."""
    x = f32(W.family3((1 << 23) + 11))
    want = oracle.scan(x, "left_fold", 1)
    t = torch.from_numpy(x.copy()).to(DEV)
    scr.inclusive_scan(t, "left_fold", 1, out=t)
    assert first_diff(t.cpu().numpy(), want) is None
    for B in (16, 256):
        got = scr.inclusive_scan(torch.from_numpy(x).pin_memory(), "block_dyadic", B).numpy()
        assert first_diff(got, oracle.scan(x, "block_dyadic", B)) is None, B
