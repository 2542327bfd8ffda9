"""GPU parity of the canonical scans against the oracle, 0 ULP (raw bits).

1-D scans over sizes that cover one and several 2048-element tiles, ragged
last tiles and threads, blocks inside a thread, inside a tile and spanning
tiles, the full-size benchmark shapes; in-place scans; batched column and row
scans; scan/reduce consistency including GPU scan vs GPU reduce."""
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


def bits(a):
    return np.asarray(a).tobytes()


def first_diff(a, b):
    a = np.asarray(a).view(np.uint8 if a.dtype.itemsize == 1 else
                           (np.uint64 if a.dtype.itemsize == 8 else np.uint32))
    b = np.asarray(b).view(a.dtype)
    idx = np.nonzero(a != b)[0]
    return (int(idx[0]), len(idx)) if len(idx) else None


def check_scan(scr, x, policy, B):
    got = scr.inclusive_scan(torch.from_numpy(x).to(DEV), policy, B).cpu().numpy()
    want = oracle.scan(x, policy, B)
    assert bits(got) == bits(want), (x.size, policy, B, first_diff(got, want))


SIZES = [1, 2, 3, 7, 8, 9, 15, 16, 17, 100, 255, 256, 257, 2047, 2048, 2049, 4095, 4096,
         4097, 2048 * 3 + 5, 2048 * 7, 100003, (1 << 20) + 37]


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("policy,B", [("iterated_pairwise", 1), ("pairwise", 1),
                                      ("left_fold", 1), ("block_dyadic", 1), ("block_dyadic", 2),
                                      ("block_dyadic", 4), ("block_dyadic", 8),
                                      ("block_dyadic", 16), ("block_dyadic", 32),
                                      ("block_dyadic", 256), ("block_dyadic", 2048),
                                      ("block_dyadic", 4096), ("block_dyadic", 1 << 16)])
def test_scan_sizes(scr, dtype, policy, B):
    for n in SIZES:
        x = W.signed_pow2(n, W.seed_for(3, n % 101), dtype, -20, 20)
        check_scan(scr, x, policy, B)


def test_scan_empty(scr):
    x = torch.empty(0, dtype=torch.float64, device=DEV)
    for policy, B in (("iterated_pairwise", 1), ("pairwise", 1), ("block_dyadic", 16),
                      ("left_fold", 1)):
        assert scr.inclusive_scan(x, policy, B).numel() == 0


@pytest.mark.parametrize("policy,B", [("iterated_pairwise", 1), ("pairwise", 1),
                                      ("block_dyadic", 16), ("block_dyadic", 4096),
                                      ("left_fold", 1)])
def test_scan_in_place(scr, policy, B):
    x = W.family3(2048 * 5 + 77)
    t = torch.from_numpy(x).to(DEV)
    scr.inclusive_scan(t, policy, B, out=t)
    assert bits(t.cpu().numpy()) == bits(oracle.scan(x, policy, B))


def test_scan_rejects_bad_block_and_overlap(scr):
    t = torch.zeros(100, dtype=torch.float64, device=DEV)
    with pytest.raises(ValueError):
        scr.inclusive_scan(t, "block_dyadic", 6)
    with pytest.raises(scr.CrError):
        scr.inclusive_scan(t[:90], "iterated_pairwise", 1, out=t[5:95])


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("policy,B", [("left_fold", 1), ("block_dyadic", 1),
                                      ("block_dyadic", 2), ("block_dyadic", 4),
                                      ("block_dyadic", 8), ("block_dyadic", 16),
                                      ("block_dyadic", 32), ("block_dyadic", 256),
                                      ("iterated_pairwise", 1), ("pairwise", 1)])
def test_scan_batched_columns_and_rows(scr, dtype, policy, B):
    levels, cols = 90, 1001  # 90 = 5 blocks of 16 + 10: a ragged last block
    buf = W.signed_pow2(levels * cols, W.seed_for(5, 3), dtype)
    t = torch.from_numpy(buf).to(DEV).view(levels, cols)
    got = scr.inclusive_scan_batched(t, policy, B, dim=0).cpu().numpy().reshape(-1)
    want = oracle.scan_batched(buf, cols, levels, cols, 1, policy, B)
    assert bits(got) == bits(want)
    # rows of a (cols x levels) array: elem_stride 1, batch_stride levels
    t2 = torch.from_numpy(buf).to(DEV).view(cols, levels)
    got2 = scr.inclusive_scan_batched(t2, policy, B, dim=1).cpu().numpy().reshape(-1)
    want2 = oracle.scan_batched(buf, cols, levels, 1, levels, policy, B)
    assert bits(got2) == bits(want2)


@pytest.mark.parametrize("policy,B", [("block_dyadic", 16), ("left_fold", 1)])
def test_column_scan_full_size(scr, policy, B):
    """The weather-column shape: 90 levels x 200,000 columns, level-major,
    lognormal values; every column checked."""
    levels, cols = 90, 200000
    buf = W.family5(levels, cols)
    t = torch.from_numpy(buf).to(DEV).view(levels, cols)
    got = scr.inclusive_scan_batched(t, policy, B, dim=0).cpu().numpy().reshape(-1)
    want = oracle.scan_batched(buf, cols, levels, cols, 1, policy, B)
    assert bits(got) == bits(want), first_diff(got, want)


@pytest.mark.parametrize("policy,B", [("iterated_pairwise", 1), ("block_dyadic", 16),
                                      ("block_dyadic", 256)])
def test_scan_full_size(scr, policy, B):
    """n = 2^24 and 2^28 (the benchmark sizes), U[-1, 1) values: every element
    compared with the oracle, and the scan's back element equals reduce<E>."""
    for n in (1 << 24, 1 << 28):
        x = W.family3(n)
        got = scr.inclusive_scan(torch.from_numpy(x).to(DEV), policy, B).cpu().numpy()
        want = oracle.scan(x, policy, B)
        assert bits(got) == bits(want), (n, first_diff(got, want))
        r = oracle.reduce_policy(x, policy, B)
        assert bits(got[-1]) == bits(r)


def test_scan_reduce_consistency_on_gpu(scr):
    """iterated_pairwise is the P4016 tree with L = 1 applied to every prefix,
    and -0.0 is the exact identity of init: the GPU scan's element i equals the
    GPU reduce of x[0..i] with L = 1 and init = -0.0 (two different kernels)."""
    x = W.family3((1 << 20) + 13)
    xd = torch.from_numpy(x).to(DEV)
    y = scr.inclusive_scan(xd, "iterated_pairwise").cpu().numpy()
    rng = np.random.default_rng(3)
    for i in list(rng.choice(x.size, 40, replace=False)) + [0, x.size - 1]:
        r = scr.reduce(xd[: i + 1], 1, -0.0).cpu().numpy()[0]
        assert bits(y[i]) == bits(r), i


def test_pairwise_full_size(scr):
    """1-D pairwise at the benchmark sizes: every element against the oracle.
    Its back element is the tree of the whole input when n is a power of two
    (one maximal subtree), and it equals iterated_pairwise wherever the
    prefix length has at most two set bits (two subtrees fold the same way
    from either side) - checked GPU against GPU at every such index."""
    for n in (1 << 24, (1 << 28) + 37):
        x = W.family3(n)
        xd = torch.from_numpy(x).to(DEV)
        got = scr.inclusive_scan(xd, "pairwise").cpu().numpy()
        want = oracle.scan(x, "pairwise")
        assert bits(got) == bits(want), (n, first_diff(got, want))
        it = scr.inclusive_scan(xd, "iterated_pairwise").cpu().numpy()
        m = np.arange(1, n + 1, dtype=np.uint64)
        low = m & (~m + np.uint64(1))
        rest = m - low
        two = (rest & (rest - np.uint64(1))) == 0  # popcount(i + 1) <= 2
        assert bits(got[two]) == bits(it[two])
        del it, m, low, rest, two
    x = W.family3(1 << 24)
    xd = torch.from_numpy(x).to(DEV)
    y = scr.inclusive_scan(xd, "pairwise").cpu().numpy()
    r = scr.reduce(xd, 1, -0.0).cpu().numpy()[0]
    assert bits(y[-1]) == bits(r)


@pytest.mark.parametrize("policy,B", [("iterated_pairwise", 1), ("pairwise", 1),
                                      ("left_fold", 1), ("block_dyadic", 16),
                                      ("block_dyadic", 256), ("block_dyadic", 4096)])
def test_scan_f32_large(scr, policy, B):
    """binary32 at 2^26 + 5: iterated_pairwise through the up/down passes,
    long carry chains through the parallel chain with the binary32
    classification (an estimate of the binary32 chain and a statistical
    margin; every step still checked exactly)."""
    x = W.family3((1 << 26) + 5).astype(np.float32)
    got = scr.inclusive_scan(torch.from_numpy(x).to(DEV), policy, B).cpu().numpy()
    want = oracle.scan(x, policy, B)
    assert bits(got) == bits(want), first_diff(got, want)


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("policy,B", [("left_fold", 1), ("block_dyadic", 16),
                                      ("block_dyadic", 4)])
def test_columns_pitch_and_offset(scr, dtype, policy, B):
    """Level-major columns with an even and an odd count, a row pitch wider
    than the columns, and a base one element off an aligned address, against
    the oracle: 37 levels (a ragged last block of levels), in place too."""
    levels = 37
    for ncols, pitch, off in ((1000, 1000, 0), (1001, 1001, 0), (1000, 1003, 0),
                              (1000, 1000, 1)):
        buf = W.lognormal(levels * pitch + off, W.seed_for(5, ncols % 7 + off)).astype(dtype)
        base = torch.from_numpy(buf).to(DEV)
        view = base[off:off + levels * pitch].view(levels, pitch)[:, :ncols]
        got = scr.inclusive_scan_batched(view, policy, B, dim=0).cpu().numpy()
        want = oracle.scan_batched(buf[off:].copy(), ncols, levels, pitch, 1, policy, B)
        want = want[:levels * pitch].reshape(levels, pitch)[:, :ncols]
        assert bits(got) == bits(np.ascontiguousarray(want)), (ncols, pitch, off)
        scr.inclusive_scan_batched(view, policy, B, dim=0, out=view)  # in place
        assert bits(view.cpu().numpy()) == bits(np.ascontiguousarray(want)), (ncols, pitch, off)
