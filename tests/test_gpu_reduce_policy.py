"""GPU reduce<E> (the root of each named scan expression) against the
oracle's reduce<E>, which evaluates the root from its own definition, 0 ULP;
and GPU against GPU: for the consistent policies the inclusive scan's last
element equals reduce<E> (two different kernel paths)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

POLICIES = [("left_fold", 1), ("iterated_pairwise", 1), ("pairwise", 1), ("block_dyadic", 1),
            ("block_dyadic", 2), ("block_dyadic", 16), ("block_dyadic", 256),
            ("block_dyadic", 4096), ("block_dyadic", 1 << 20)]
SIZES = [1, 2, 3, 15, 16, 17, 255, 1000, 4097, 100003, (1 << 20) + 7]


@pytest.fixture(scope="module")
def scr():
    import scan_canonical_reduce_gb300 as m
    return m


def bits(a):
    return np.asarray(a).tobytes()


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("policy,B", POLICIES)
def test_reduce_policy_sizes(scr, dtype, policy, B):
    for n in SIZES:
        x = W.signed_pow2(n, W.seed_for(3, 11 + n % 89), dtype, -20, 20)
        got = scr.reduce_policy(torch.from_numpy(x).to(DEV), policy, B).cpu().numpy()[0]
        want = oracle.reduce_policy(x, policy, B)
        assert bits(got) == bits(want), (n, got, want)


@pytest.mark.parametrize("policy,B", [("left_fold", 1), ("iterated_pairwise", 1),
                                      ("block_dyadic", 16), ("block_dyadic", 256)])
def test_scan_back_equals_reduce_on_gpu(scr, policy, B):
    """Consistency (P4229R0): inclusive_scan<E>(x)[n-1] == reduce<E>(x), both
    computed on the GPU by different kernels, at the benchmark's size."""
    x = W.family3((1 << 28) if policy != "left_fold" else (1 << 24))
    xd = torch.from_numpy(x).to(DEV)
    y = scr.inclusive_scan(xd, policy, B)
    r = scr.reduce_policy(xd, policy, B)
    assert bits(y[-1:].cpu().numpy()) == bits(r.cpu().numpy())
    want = oracle.reduce_policy(x, policy, B)
    assert bits(r.cpu().numpy()[0]) == bits(want)


def test_pairwise_root_is_the_tree(scr):
    """reduce<pairwise> is the tree of all x (the root of the one tree), which
    the canonical reduction with one lane and init -0.0 also computes."""
    x = W.family2((1 << 22) + 5)
    xd = torch.from_numpy(x).to(DEV)
    a = scr.reduce_policy(xd, "pairwise").cpu().numpy()
    b = scr.reduce(xd, 1, -0.0).cpu().numpy()
    assert bits(a) == bits(b)


def test_reduce_policy_rejects_empty(scr):
    with pytest.raises(ValueError):
        scr.reduce_policy(torch.empty(0, dtype=torch.float64, device=DEV), "left_fold")


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("policy,B", [("left_fold", 1), ("block_dyadic", 2)])
@pytest.mark.parametrize("n", [2, 5, 64, 65, 1000, 1023])
def test_reduce_policy_ends_at_minus_zero(scr, dtype, policy, B, n):
    """Chains short enough for the serial kernel whose value ends at -0.0 (an
    add gives -0.0 only from two -0.0 operands, so every operand is -0.0):
    the root keeps its sign, so the kernel's padding past the last step must
    be the identity -0.0, not +0.0."""
    x = np.full(n, -0.0, dtype=dtype)
    want = oracle.reduce_policy(x, policy, B)
    assert np.signbit(want)
    got = scr.reduce_policy(torch.from_numpy(x).to(DEV), policy, B).cpu().numpy()[0]
    assert bits(np.array([got])) == bits(np.array([want])), (got, want)
