"""Randomised parity: seeded draws of sizes (biased toward tile, block and
chunk edges), policies, block sizes, element types, value families and
output forms, every result against the oracle at 0 ULP (NaN compared as a
class). Reproducible: the draws come from fixed seeds."""
import random

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


def same(got, want):
    got, want = np.asarray(got), np.asarray(want)
    assert got.shape == want.shape, (got.shape, want.shape)
    u = np.uint64 if got.dtype.itemsize == 8 else np.uint32
    gn, wn = np.isnan(got), np.isnan(want)
    diff = ((got.view(u) != want.view(u)) & ~(gn & wn)) | (gn != wn)
    idx = np.nonzero(diff.reshape(-1))[0]
    return None if idx.size == 0 else (int(idx[0]), int(idx.size))


def draw_n(rng):
    edges = [2048, 4096, 16, 256, 1 << 20]
    kind = rng.random()
    if kind < 0.3:  # just around a tile / block / chunk edge
        e = rng.choice(edges) * rng.randint(1, 40)
        return max(1, e + rng.randint(-3, 3))
    if kind < 0.5:
        return rng.randint(1, 300)
    return rng.randint(1, 3_000_000)


def draw_values(rng, n, dtype, seed):
    fam = rng.randrange(5)
    if fam == 0:
        return W.signed_pow2(n, seed, dtype, -30, 30)
    if fam == 1:
        return W.uniform_pm1(n, seed).astype(dtype)
    if fam == 2:
        return W.small_integers(n, seed, 1 << 10, dtype)
    if fam == 3:
        return (W.uniform_pm1(n, seed) * 1e-3 + 1.0).astype(dtype)  # few rises, long runs
    x = W.uniform_pm1(n, seed).astype(dtype)
    if n > 10:
        x[rng.randrange(n)] = dtype(0.0) * -1  # a signed zero somewhere
    return x


POL = [("left_fold", 1), ("pairwise", 1), ("iterated_pairwise", 1)] + \
      [("block_dyadic", 1 << k) for k in range(0, 14)]


@pytest.mark.parametrize("case", range(150))
def test_random_scans(scr, case):
    rng = random.Random(1000 + case)
    n = draw_n(rng)
    dtype = rng.choice([np.float64, np.float32])
    policy, B = rng.choice(POL)
    x = draw_values(rng, n, dtype, W.seed_for(7, case))
    xd = torch.from_numpy(x).to(DEV)
    form = rng.choice(["inclusive", "exclusive", "include_initial", "host"])
    init = dtype(rng.choice([0.0, -0.0, 1.5, -3.25]))
    if form == "inclusive":
        got = scr.inclusive_scan(xd, policy, B).cpu().numpy()
        want = oracle.scan(x, policy, B)
    elif form == "host":
        got = scr.inclusive_scan(torch.from_numpy(x).pin_memory(), policy, B).numpy()
        want = oracle.scan(x, policy, B)
    else:
        f = scr.exclusive_scan if form == "exclusive" else scr.scan_include_initial
        got = f(xd, policy, B, init).cpu().numpy()
        want = oracle.scan_ex(x, policy, B, init, form)
    bad = same(got, want)
    assert bad is None, (n, dtype, policy, B, form, bad)


@pytest.mark.parametrize("case", range(80))
def test_random_reductions(scr, case):
    rng = random.Random(5000 + case)
    n = draw_n(rng)
    dtype = rng.choice([np.float64, np.float32])
    x = draw_values(rng, n, dtype, W.seed_for(8, case))
    xd = torch.from_numpy(x).to(DEV)
    L = rng.choice([1, 2, 3, 16, 100, 128, 1000, 1024, 4096, n, n + 5])
    init = dtype(rng.choice([0.0, -0.0, 0.5]))
    got = scr.reduce(xd, L, init).cpu().numpy()[0]
    assert same(np.array([got]), np.array([oracle.reduce(x, L, init)])) is None, (n, L, dtype)
    policy, B = rng.choice(POL)
    got = scr.reduce_policy(xd, policy, B).cpu().numpy()[0]
    want = oracle.reduce_policy(x, policy, B)
    assert same(np.array([got]), np.array([want])) is None, (n, policy, B, dtype)


@pytest.mark.parametrize("case", range(40))
def test_random_batched(scr, case):
    rng = random.Random(9000 + case)
    dtype = rng.choice([np.float64, np.float32])
    rows, cols = rng.randint(1, 3000), rng.randint(1, 400)
    buf = draw_values(rng, rows * cols, dtype, W.seed_for(9, case))
    t = torch.from_numpy(buf).to(DEV).view(rows, cols)
    dim = rng.choice([0, 1])
    n, batch = (rows, cols) if dim == 0 else (cols, rows)
    es, bs = (cols, 1) if dim == 0 else (1, cols)
    L = rng.choice([1, 3, 16, 64, 128])
    got = scr.reduce_batched(t, L, 0.25, dim=dim).cpu().numpy()
    want = oracle.reduce_batched(buf, batch, n, es, bs, L, dtype(0.25))
    assert same(got, want) is None, ("reduce", rows, cols, dim, L)
    policy, B = rng.choice(POL[:3] + [("block_dyadic", 4), ("block_dyadic", 16),
                                      ("block_dyadic", 64)])
    got = scr.inclusive_scan_batched(t, policy, B, dim=dim).cpu().numpy().reshape(-1)
    want = oracle.scan_batched(buf, batch, n, es, bs, policy, B)
    assert same(got, want) is None, ("scan", rows, cols, dim, policy, B)
