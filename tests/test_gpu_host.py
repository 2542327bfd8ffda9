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
