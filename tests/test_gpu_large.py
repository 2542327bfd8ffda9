"""Sequences past 2^31 elements, so that every index of every pass is 64-bit.

The values are -1, 0 or 1 (seeded), and every partial sum any tree or chain
forms is a difference of two prefix sums of them. The test first checks that
every prefix sum is below 2^22 in magnitude; then every add of every policy
is exact in binary32 and binary64, so each output of every named expression
equals the exact integer prefix sum (and the reduction the exact total),
whatever its parenthesisation. The exact sums are integer arithmetic
(torch.cumsum on int32), not the kernels under test."""
import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
N = (1 << 31) + 4099


@pytest.fixture(scope="module")
def scr():
    import scan_canonical_reduce_gb300 as m
    return m


@pytest.fixture(scope="module")
def walk():
    g = torch.Generator(device=DEV)
    g.manual_seed(0x5CA1AB1E)
    xi = torch.randint(-1, 2, (N,), dtype=torch.int8, device=DEV, generator=g)
    exact = torch.cumsum(xi, 0, dtype=torch.int32)
    # every range sum of the walk is below 2^23: exact in binary32
    assert int(exact.abs().max()) < (1 << 22)
    yield xi, exact
    del xi, exact
    torch.cuda.empty_cache()


@pytest.mark.parametrize("dt", [torch.float32, torch.float64])
def test_scans_and_reduce_past_2_31(scr, walk, dt):
    xi, exact = walk
    x = xi.to(dt)
    want = exact.to(dt)
    y = torch.empty_like(x)
    for policy, B in (("iterated_pairwise", 1), ("pairwise", 1), ("block_dyadic", 16),
                      ("block_dyadic", 256)):
        y.fill_(float("nan"))
        scr.inclusive_scan(x, policy, B, out=y)
        torch.cuda.synchronize()
        bad = torch.nonzero(y != want)
        assert bad.numel() == 0, (policy, B, dt, int(bad[0]))
    for L in (16, 1024):
        r = scr.reduce(x, L, 0.0)
        assert float(r[0]) == float(exact[-1]), (L, dt)
    del x, y, want
    torch.cuda.empty_cache()


def test_batched_past_2_31(scr):
    """A level-major column scan of 90 levels x 23,860,930 columns and a row
    reduce of 16,385 rows x 131,072 columns: 2^31 elements and more in one
    call, the per-sequence sums exact."""
    g = torch.Generator(device=DEV)
    g.manual_seed(0xC01D)
    levels, cols = 90, 23860930
    xi = torch.randint(-1, 2, (levels, cols), dtype=torch.int8, device=DEV, generator=g)
    assert xi.numel() > (1 << 31)
    exact = torch.cumsum(xi, 0, dtype=torch.int32)
    x = xi.to(torch.float32)
    y = torch.empty_like(x)
    for policy, B in (("left_fold", 1), ("block_dyadic", 16)):
        y.fill_(float("nan"))
        scr.inclusive_scan_batched(x, policy, B, dim=0, out=y)
        torch.cuda.synchronize()
        assert torch.equal(y, exact.to(torch.float32)), policy
    del xi, exact, x, y
    torch.cuda.empty_cache()
    rows, n = 16385, 131072
    xi = torch.randint(-1, 2, (rows, n), dtype=torch.int8, device=DEV, generator=g)
    assert xi.numel() > (1 << 31)
    want = xi.sum(dim=1, dtype=torch.int32).to(torch.float32)
    x = xi.to(torch.float32)
    got = scr.reduce_batched(x, 128, 0.0, dim=-1)
    assert torch.equal(got, want)
    del xi, x, got, want
    torch.cuda.empty_cache()
