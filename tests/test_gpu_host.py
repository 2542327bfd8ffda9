"""Host-buffer forms (cr_inclusive_scan_host, cr_reduce_host): inputs and
outputs in host memory, copies pipelined with the passes in chunks of tiles
(block_dyadic with B <= 2048: the carries folded chunk by chunk too).
0 ULP against the oracle for every policy and kernel path, chunk-boundary
sizes, page-locked and pageable host memory, and the benchmark size."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

POLICIES = [("iterated_pairwise", 1), ("pairwise", 1), ("left_fold", 1), ("block_dyadic", 2),
            ("block_dyadic", 16), ("block_dyadic", 256), ("block_dyadic", 2048),
            ("block_dyadic", 4096), ("block_dyadic", 1 << 16)]


@pytest.fixture(scope="module")
def scr():
    import scan_canonical_reduce_gb300 as m
    return m


def bits(a):
    return np.asarray(a).tobytes()


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("policy,B", POLICIES)
def test_scan_host(scr, dtype, policy, B):
    # 1 tile; one chunk; 8 chunks of 513 tiles with a ragged last tile
    for n in (7, 2048 * 300 + 1, 2048 * 4100 + 77):
        x = W.signed_pow2(n, W.seed_for(3, n % 41), dtype, -20, 20)
        got = scr.inclusive_scan(torch.from_numpy(x).pin_memory(), policy, B)
        assert not got.is_cuda
        assert bits(got.numpy()) == bits(oracle.scan(x, policy, B)), n


def test_scan_host_pageable_and_out(scr):
    x = W.family3(2048 * 1000 + 3)
    want = oracle.scan(x, "block_dyadic", 16)
    got = scr.inclusive_scan(torch.from_numpy(x), "block_dyadic", 16)  # pageable input
    assert bits(got.numpy()) == bits(want)
    out = torch.empty(x.size, dtype=torch.float64)  # pageable output
    scr.inclusive_scan(torch.from_numpy(x).pin_memory(), "block_dyadic", 16, out=out)
    assert bits(out.numpy()) == bits(want)


@pytest.mark.parametrize("B", [2, 16, 256, 2048])
def test_scan_host_chunked_carries(scr, B):
    """block_dyadic (B <= 2048) from host buffers folds the carries chunk by
    chunk, each segment continued from the previous one's last carry, so
    that chunks are copied out while later ones are copied in: the chain's
    stress families at chunk-edge sizes (3 whole chunks; a last chunk of one
    or two blocks; 8 chunks with a ragged last tile)."""
    from tests.test_gpu_chain import CASES
    for case in ("wide_exponents", "cancel_to_zero", "big_then_small", "halves_ties"):
        for n in (2048 * 256 * 3, 2048 * 256 * 3 + B + 1, 2048 * 2100 - 1):
            x = np.ascontiguousarray(CASES[case](n, np.float64))
            got = scr.inclusive_scan(torch.from_numpy(x).pin_memory(), "block_dyadic", B).numpy()
            want = oracle.scan(x, "block_dyadic", B)
            gn, wn = np.isnan(got), np.isnan(want)
            bad = ((got.view(np.uint64) != want.view(np.uint64)) & ~(gn & wn)) | (gn != wn)
            assert not bad.any(), (case, n, int(np.argmax(bad)))


@pytest.mark.parametrize("policy,B", [("iterated_pairwise", 1), ("block_dyadic", 16),
                                      ("block_dyadic", 256)])
def test_scan_host_full_size(scr, policy, B):
    x = W.family3(1 << 28)
    got = scr.inclusive_scan(torch.from_numpy(x).pin_memory(), policy, B)
    assert bits(got.numpy()) == bits(oracle.scan(x, policy, B))


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_reduce_host(scr, dtype):
    for n in (0, 1, 1000, (1 << 22) + 3):
        x = W.family2(n, dtype) if n else np.zeros(0, dtype=dtype)
        for L in (1, 16, 1024):
            got = scr.reduce(torch.from_numpy(x).pin_memory(), L, 0.5)
            assert not got.is_cuda
            assert bits(got.numpy()[0]) == bits(oracle.reduce(x, L, dtype(0.5))), (n, L)


@pytest.mark.parametrize("L", [1, 3, 16, 128, 1024, 5000])
def test_reduce_host_chunked(scr, L):
    """From host buffers the first pass reduces groups of its chunks as they
    arrive: sizes with a ragged tail, a last group of one chunk, and the
    benchmark size (every lane count, fp64)."""
    for n in (2048 * 1024 * 3 + 17, (1 << 24) + 5):
        x = W.family2(n)
        got = scr.reduce(torch.from_numpy(x).pin_memory(), L, -0.25)
        assert bits(got.numpy()[0]) == bits(oracle.reduce(x, L, -0.25)), (n, L)


def test_reduce_host_full_size(scr):
    x = W.family2(1 << 28)
    h = torch.from_numpy(x).pin_memory()
    for L in (16, 128, 1024):
        got = scr.reduce(h, L, 0.0)
        assert bits(got.numpy()[0]) == bits(oracle.reduce(x, L, 0.0)), L


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_reduce_batched_host(scr, dtype):
    """cr_reduce_batched_host: rows and level-major columns, padded rows,
    one group and several groups (a ragged last one), against the oracle."""
    for rows, cols in ((3, 1000), (300, 4096 + 37), (2100, 16384 + 5)):
        buf = W.signed_pow2(rows * cols, W.seed_for(4, rows % 61), dtype)
        t = torch.from_numpy(buf).view(rows, cols).pin_memory()
        for L in (1, 16, 128):
            got = scr.reduce_batched(t, L, 0.5, dim=-1)
            assert not got.is_cuda
            want = oracle.reduce_batched(buf, rows, cols, 1, cols, L, dtype(0.5))
            assert bits(got.numpy()) == bits(want), (rows, cols, L)
            gotc = scr.reduce_batched(t, L, 0.5, dim=0)
            wantc = oracle.reduce_batched(buf, cols, rows, cols, 1, L, dtype(0.5))
            assert bits(gotc.numpy()) == bits(wantc), (rows, cols, L)
    # rows with padding (batch_stride > n), pageable memory
    rows, cols, pad = 500, 3000, 13
    buf = W.signed_pow2(rows * (cols + pad), W.seed_for(4, 7), dtype)
    view = torch.from_numpy(buf).view(rows, cols + pad)[:, :cols]
    got = scr.reduce_batched(view, 16, -1.0, dim=-1)
    want = oracle.reduce_batched(buf, rows, cols, 1, cols + pad, 16, dtype(-1.0))
    assert bits(got.numpy()) == bits(want)


def test_reduce_batched_host_full_size(scr):
    """The benchmark's row reduces from host buffers (65,536 x 4,096 and
    1,024 x 262,144 binary32, L = 128), sampled rows against the oracle."""
    for rows, cols in ((65536, 4096), (1024, 262144)):
        x = W.family4(rows, cols)
        got = scr.reduce_batched(torch.from_numpy(x).pin_memory(), 128, 0.0).numpy()
        dev = scr.reduce_batched(torch.from_numpy(x).cuda(), 128, 0.0).cpu().numpy()
        assert bits(got) == bits(dev)
        rng = np.random.default_rng(2)
        for r in list(rng.choice(rows, 32, replace=False)) + [0, rows - 1]:
            want = oracle.reduce(x[r].copy(), 128, np.float32(0.0))
            assert bits(got[r]) == bits(want), r


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("policy,B", [("left_fold", 1), ("block_dyadic", 16),
                                      ("iterated_pairwise", 1), ("pairwise", 1),
                                      ("block_dyadic", 4)])
def test_scan_batched_host(scr, dtype, policy, B):
    """cr_inclusive_scan_batched_host on level-major columns (the column-scan
    shape, several groups) and on rows, against the oracle; in place too."""
    levels, ncols = 90, 20000 + 3
    buf = W.lognormal(levels * ncols, W.seed_for(5, 3)).astype(dtype)
    t = torch.from_numpy(buf).view(levels, ncols).pin_memory()
    got = scr.inclusive_scan_batched(t, policy, B, dim=0)
    assert not got.is_cuda
    want = oracle.scan_batched(buf, ncols, levels, ncols, 1, policy, B)
    assert bits(got.numpy().reshape(-1)) == bits(want)
    # rows: 700 sequences of 5000 elements
    rows, n = 700, 5000
    rb = W.signed_pow2(rows * n, W.seed_for(5, 4), dtype)
    tr = torch.from_numpy(rb).view(rows, n).pin_memory()
    gr = scr.inclusive_scan_batched(tr, policy, B, dim=-1)
    wr = oracle.scan_batched(rb, rows, n, 1, n, policy, B)
    assert bits(gr.numpy().reshape(-1)) == bits(wr)
    # in place (out is x)
    scr.inclusive_scan_batched(t, policy, B, dim=0, out=t)
    assert bits(t.numpy().reshape(-1)) == bits(want)


def test_scan_batched_host_full_size(scr):
    """The benchmark's column scans (90 x 200,000 fp64) from host buffers."""
    x = W.family5(90, 200000)
    t = torch.from_numpy(x).view(90, 200000).pin_memory()
    for policy, B in (("block_dyadic", 16), ("left_fold", 1)):
        got = scr.inclusive_scan_batched(t, policy, B, dim=0)
        want = oracle.scan_batched(x, 200000, 90, 200000, 1, policy, B)
        assert bits(got.numpy().reshape(-1)) == bits(want), policy


def test_batched_host_layout_errors(scr):
    """A layout that is neither rows nor level-major columns is unsupported
    by the host-buffer calls; an output that partially overlaps the input is
    rejected."""
    import ctypes
    L = scr.lib()
    x = torch.zeros(4000, dtype=torch.float64).pin_memory()
    out = torch.zeros(4000, dtype=torch.float64).pin_memory()
    ws = scr.workspace("cuda", None, 1 << 24)
    one = ctypes.c_double(0.0)
    # element stride 2 and sequence stride 3: neither layout
    assert L.cr_reduce_batched_host(x.data_ptr(), out.data_ptr(), 10, 10, 2, 3, 16,
                                    ctypes.byref(one), 2, ws.data_ptr(), ws.numel(),
                                    None) == 2
    assert L.cr_inclusive_scan_batched_host(x.data_ptr(), out.data_ptr(), 10, 10, 2, 30, 0, 1,
                                            2, ws.data_ptr(), ws.numel(), None) == 2
    # out one element into x's rows
    assert L.cr_inclusive_scan_batched_host(x.data_ptr(), x.data_ptr() + 8, 10, 10, 1, 10, 0,
                                            1, 2, ws.data_ptr(), ws.numel(), None) == 1
    assert L.cr_reduce_batched_host(x.data_ptr(), x.data_ptr() + 80, 10, 10, 1, 10, 16,
                                    ctypes.byref(one), 2, ws.data_ptr(), ws.numel(),
                                    None) == 1
