"""GPU parity of the exclusive scan and the include_initial form against the
oracle, 0 ULP (raw bits): out[0] = init, out[k] = init + inclusive[k - 1]
(n or n + 1 outputs). Every policy and kernel path (one-pass tiles, pairwise
up/down, block_dyadic local + fix-up and up/down, the left-fold chain, the
per-sequence batched kernel), ragged sizes, in place, empty inputs, columns
of a level-major array written to n + 1 interface levels, and the benchmark
size."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

POLICIES = [("iterated_pairwise", 1), ("pairwise", 1), ("left_fold", 1), ("block_dyadic", 1),
            ("block_dyadic", 2), ("block_dyadic", 4), ("block_dyadic", 16),
            ("block_dyadic", 256), ("block_dyadic", 2048), ("block_dyadic", 4096),
            ("block_dyadic", 1 << 16)]
SIZES = [1, 2, 3, 7, 8, 9, 16, 17, 255, 256, 257, 2047, 2048, 2049, 4096, 4097,
         2048 * 3 + 5, 2048 * 7, 100003, (1 << 20) + 37]


@pytest.fixture(scope="module")
def scr():
    import scan_canonical_reduce_gb300 as m
    return m


def bits(a):
    return np.asarray(a).tobytes()


def first_diff(a, b):
    a = np.asarray(a)
    b = np.asarray(b)
    u = np.uint64 if a.dtype.itemsize == 8 else np.uint32
    idx = np.nonzero(a.view(u) != b.view(u))[0]
    return (int(idx[0]), len(idx)) if len(idx) else None


def run(scr, x, policy, B, init, mode):
    xd = torch.from_numpy(x).to(DEV)
    f = scr.exclusive_scan if mode == "exclusive" else scr.scan_include_initial
    return f(xd, policy, B, init).cpu().numpy()


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("mode", ["exclusive", "include_initial"])
@pytest.mark.parametrize("policy,B", POLICIES)
def test_sizes(scr, dtype, mode, policy, B):
    init = dtype(0.75)
    for n in SIZES:
        x = W.signed_pow2(n, W.seed_for(3, 7 + n % 97), dtype, -20, 20)
        got = run(scr, x, policy, B, init, mode)
        want = oracle.scan_ex(x, policy, B, init, mode)
        assert got.size == want.size
        assert bits(got) == bits(want), (n, first_diff(got, want))


@pytest.mark.parametrize("mode", ["exclusive", "include_initial"])
def test_empty(scr, mode):
    x = torch.empty(0, dtype=torch.float64, device=DEV)
    for policy, B in POLICIES:
        f = scr.exclusive_scan if mode == "exclusive" else scr.scan_include_initial
        y = f(x, policy, B, 2.5).cpu().numpy()
        assert y.tolist() == ([] if mode == "exclusive" else [2.5])


@pytest.mark.parametrize("policy,B", POLICIES)
def test_in_place(scr, policy, B):
    """out == x: exclusive on the n-element buffer; include_initial on a
    buffer of n + 1 whose first n elements are the input."""
    n = 2048 * 5 + 77
    x = W.family3(n)
    t = torch.from_numpy(x).to(DEV)
    scr.exclusive_scan(t, policy, B, -1.25, out=t)
    assert bits(t.cpu().numpy()) == bits(oracle.scan_ex(x, policy, B, -1.25, "exclusive"))
    buf = torch.zeros(n + 1, dtype=torch.float64, device=DEV)
    buf[:n] = torch.from_numpy(x).to(DEV)
    scr.scan_include_initial(buf[:n], policy, B, -1.25, out=buf)
    assert bits(buf.cpu().numpy()) == bits(oracle.scan_ex(x, policy, B, -1.25,
                                                          "include_initial"))


@pytest.mark.parametrize("policy,B", [("iterated_pairwise", 1), ("pairwise", 1),
                                      ("block_dyadic", 16), ("block_dyadic", 4096),
                                      ("left_fold", 1)])
def test_minus_zero_init_is_the_shifted_inclusive_scan(scr, policy, B):
    """GPU against GPU: with init = -0.0 the exclusive scan is the inclusive
    scan moved one place right (different kernels or epilogues)."""
    x = W.family3((1 << 20) + 3)
    xd = torch.from_numpy(x).to(DEV)
    inc = scr.inclusive_scan(xd, policy, B).cpu().numpy()
    ex = scr.exclusive_scan(xd, policy, B, -0.0).cpu().numpy()
    ii = scr.scan_include_initial(xd, policy, B, -0.0).cpu().numpy()
    assert bits(ex[1:]) == bits(inc[:-1]) and bits(ex[:1]) == bits(np.array([-0.0]))
    assert bits(ii[1:]) == bits(inc)


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("mode", ["exclusive", "include_initial"])
@pytest.mark.parametrize("policy,B", [("left_fold", 1), ("block_dyadic", 16),
                                      ("block_dyadic", 8), ("block_dyadic", 4),
                                      ("block_dyadic", 2), ("block_dyadic", 64),
                                      ("iterated_pairwise", 1), ("pairwise", 1)])
def test_batched(scr, dtype, mode, policy, B):
    """Columns of a level-major (levels x cols) array, written to a
    (levels + extra) x cols array; rows of a (cols x levels) array."""
    levels, cols = 90, 1001
    extra = 1 if mode == "include_initial" else 0
    buf = W.signed_pow2(levels * cols, W.seed_for(5, 4), dtype)
    init = dtype(3.0)
    f = scr.exclusive_scan_batched if mode == "exclusive" else scr.scan_include_initial_batched
    t = torch.from_numpy(buf).to(DEV).view(levels, cols)
    got = f(t, policy, B, init, dim=0).cpu().numpy().reshape(-1)
    want = np.full((levels + extra) * cols, np.nan, dtype=dtype)
    oracle.scan_ex_batched(buf, cols, levels, cols, 1, policy, B, init, mode, want, cols, 1)
    assert bits(got) == bits(want)
    t2 = torch.from_numpy(buf).to(DEV).view(cols, levels)
    got2 = f(t2, policy, B, init, dim=1).cpu().numpy().reshape(-1)
    want2 = np.full(cols * (levels + extra), np.nan, dtype=dtype)
    oracle.scan_ex_batched(buf, cols, levels, 1, levels, policy, B, init, mode, want2, 1,
                           levels + extra)
    assert bits(got2) == bits(want2)


def test_batched_empty_sequences(scr):
    t = torch.empty(0, 5, dtype=torch.float64, device=DEV)
    y = scr.scan_include_initial_batched(t, "left_fold", 1, 4.0, dim=0).cpu().numpy()
    assert y.shape == (1, 5) and (y == 4.0).all()
    assert scr.exclusive_scan_batched(t, "left_fold", 1, 4.0, dim=0).numel() == 0


def test_column_interfaces_full_size(scr):
    """The weather-column shape: 90 levels x 200,000 columns, level-major,
    lognormal values, to 91 interface levels with the boundary value first."""
    levels, cols = 90, 200000
    buf = W.family5(levels, cols)
    t = torch.from_numpy(buf).to(DEV).view(levels, cols)
    for policy, B in (("block_dyadic", 16), ("left_fold", 1)):
        got = scr.scan_include_initial_batched(t, policy, B, 0.5, dim=0).cpu().numpy()
        want = np.empty((levels + 1) * cols)
        oracle.scan_ex_batched(buf, cols, levels, cols, 1, policy, B, 0.5, "include_initial",
                               want, cols, 1)
        assert bits(got.reshape(-1)) == bits(want), first_diff(got.reshape(-1), want)


@pytest.mark.parametrize("policy,B", [("iterated_pairwise", 1), ("pairwise", 1),
                                      ("block_dyadic", 16), ("block_dyadic", 256)])
def test_full_size(scr, policy, B):
    """n = 2^28, U[-1, 1): every element of both forms against the oracle."""
    n = 1 << 28
    x = W.family3(n)
    xd = torch.from_numpy(x).to(DEV)
    for mode in ("exclusive", "include_initial"):
        f = scr.exclusive_scan if mode == "exclusive" else scr.scan_include_initial
        got = f(xd, policy, B, 0.125).cpu().numpy()
        want = oracle.scan_ex(x, policy, B, 0.125, mode)
        assert bits(got) == bits(want), (mode, first_diff(got, want))
        del got, want


def test_left_fold_chain_size(scr):
    """The parallel exact chain with a shifted output, n = 2^24."""
    x = W.family3(1 << 24)
    xd = torch.from_numpy(x).to(DEV)
    for mode in ("exclusive", "include_initial"):
        f = scr.exclusive_scan if mode == "exclusive" else scr.scan_include_initial
        got = f(xd, "left_fold", 1, 0.125).cpu().numpy()
        assert bits(got) == bits(oracle.scan_ex(x, "left_fold", 1, 0.125, mode)), mode


@pytest.mark.parametrize("policy,B", [("left_fold", 1), ("block_dyadic", 16),
                                      ("block_dyadic", 4), ("iterated_pairwise", 1)])
def test_batched_exclusive_in_place(scr, policy, B):
    """out == x with the same strides: every element is read before the
    store one level further down overwrites it."""
    levels, cols = 90, 777
    buf = W.signed_pow2(levels * cols, W.seed_for(5, 9))
    t = torch.from_numpy(buf).to(DEV).view(levels, cols)
    scr.exclusive_scan_batched(t, policy, B, 0.5, dim=0, out=t)
    want = np.empty(levels * cols)
    oracle.scan_ex_batched(buf, cols, levels, cols, 1, policy, B, 0.5, "exclusive", want, cols,
                           1)
    assert bits(t.cpu().numpy().reshape(-1)) == bits(want)
