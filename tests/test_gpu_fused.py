"""The fused carry fix-up of the block_dyadic scan (carries by the parallel
exact chain, inclusive, out != x; used by default for B <= 16, forced here
for every B from 2 to 2048 through the library's test hook): the chain's
walk, checks and fill run in one cooperative pass with the fix-up
out[i] = C_{k-1} + P(i) behind them. The 1-D left fold runs the same pass
without a fix-up (the fills overlapping the walk). Against the oracle at 0 ULP, over
several chain tiles (4096 carries each) with ragged ends, and bit-equal to
the separate passes and to the recovery that runs after a failure raised
half-way through the walk (the hook sets a flag; no fault)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.test_gpu_chain import CASES

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def scr():
    import scan_canonical_reduce_gb300 as m
    yield m
    m.lib().cr_debug_fused_fixup(0)


def first_diff(a, b):
    u = np.uint64 if a.dtype.itemsize == 8 else np.uint32
    idx = np.nonzero(a.view(u) != b.view(u))[0]
    return None if idx.size == 0 else (int(idx[0]), int(idx.size))


def scan_mode(scr, x, B, mode):
    scr.lib().cr_debug_fused_fixup(mode)
    try:
        return scr.inclusive_scan(torch.from_numpy(x).to(DEV), "block_dyadic", B).cpu().numpy()
    finally:
        scr.lib().cr_debug_fused_fixup(0)


@pytest.mark.parametrize("B", [2, 4, 8, 16, 64, 256, 2048])
@pytest.mark.parametrize("tail", [0, 1, "half"])
def test_fused_against_oracle(scr, B, tail):
    """3 chain tiles and a few carries more; a ragged last block."""
    extra = {0: 0, 1: 1, "half": B // 2 + 1}[tail]
    n = B * (3 * 4096 + 5) + extra
    x = W.uniform_pm1(n, W.seed_for(31, B))
    want = oracle.scan(x, "block_dyadic", B)
    for mode in (0, 3):
        got = scan_mode(scr, x, B, mode)
        assert first_diff(got, want) is None, (n, B, mode, first_diff(got, want))


@pytest.mark.parametrize("B", [2, 16, 256, 2048])
def test_modes_agree(scr, B):
    """Fused, separate passes, and fused with the recovery: the same bits."""
    n = B * (5 * 4096 + 3) + 7
    x = W.family3(n)
    fused = scan_mode(scr, x, B, 3)
    separate = scan_mode(scr, x, B, 1)
    recovered = scan_mode(scr, x, B, 2)
    assert first_diff(fused, separate) is None
    assert first_diff(recovered, separate) is None


@pytest.mark.parametrize("case", sorted(CASES))
def test_value_families(scr, case):
    """The chain's stress inputs as block values (B = 16), every mode."""
    B = 16
    n = B * 20000 + 9
    x = np.ascontiguousarray(CASES[case](n, np.float64))
    want = oracle.scan(x, "block_dyadic", B)
    for mode in (0, 2, 3):
        got = scan_mode(scr, x, B, mode)
        gn, wn = np.isnan(got), np.isnan(want)
        bad = (got.view(np.uint64) != want.view(np.uint64)) & ~(gn & wn) | (gn != wn)
        assert not bad.any(), (case, mode, int(np.argmax(bad)))


@pytest.mark.parametrize("B", [16, 2048])
def test_binary32(scr, B):
    """Binary32 carries (about 4000: one chain tile) through every fused mode."""
    n = B * 4000 + 3
    x = W.uniform_pm1(n, W.seed_for(32, B)).astype(np.float32)
    want = oracle.scan(x, "block_dyadic", B)
    for mode in (2, 3):
        got = scan_mode(scr, x, B, mode)
        assert first_diff(got, want) is None, (mode, first_diff(got, want))


def test_short_chains(scr):
    """Chains from the parallel threshold (1024 carries) up: one tile, a
    partial tile, exactly one tile, one carry past it."""
    for K in (1025, 2000, 4097, 4098):
        for B in (2, 16):
            n = B * K - (B // 2)
            x = W.signed_pow2(n, W.seed_for(33, K), np.float64, -20, 20)
            want = oracle.scan(x, "block_dyadic", B)
            for mode in (0, 2, 3):
                got = scan_mode(scr, x, B, mode)
                assert first_diff(got, want) is None, (K, B, mode)


def test_bench_size_modes(scr):
    """n = 2^28, B = 16 (2^24 blocks, 4096 chain tiles): fused against the
    separate passes, all elements; a sample of positions against the oracle."""
    n = 1 << 28
    x = W.family3(n)
    xd = torch.from_numpy(x).to(DEV)
    scr.lib().cr_debug_fused_fixup(1)
    sep = scr.inclusive_scan(xd, "block_dyadic", 16)
    scr.lib().cr_debug_fused_fixup(0)
    fused = scr.inclusive_scan(xd, "block_dyadic", 16)
    assert bool(torch.equal(sep.view(torch.int64), fused.view(torch.int64)))
    scr.lib().cr_debug_fused_fixup(2)
    rec = scr.inclusive_scan(xd, "block_dyadic", 16)
    scr.lib().cr_debug_fused_fixup(0)
    assert bool(torch.equal(sep.view(torch.int64), rec.view(torch.int64)))
    head = 1 << 20
    want = oracle.scan(x[:head].copy(), "block_dyadic", 16)
    assert first_diff(fused[:head].cpu().numpy(), want) is None


def fold_mode(scr, x, mode, form="inclusive"):
    scr.lib().cr_debug_fused_fixup(mode)
    try:
        xd = torch.from_numpy(x).to(DEV)
        if form == "inclusive":
            return scr.inclusive_scan(xd, "left_fold", 1).cpu().numpy()
        f = scr.exclusive_scan if form == "exclusive" else scr.scan_include_initial
        return f(xd, "left_fold", 1, 0.375).cpu().numpy()
    finally:
        scr.lib().cr_debug_fused_fixup(0)


@pytest.mark.parametrize("n", [1025, 4096, 4097, 3 * 4096 + 17, 300007, (1 << 22) + 5])
def test_left_fold_fused(scr, n):
    """The 1-D left fold: fused (default), separate passes, and fused with a
    failure raised half-way through the walk; all against the oracle."""
    x = W.uniform_pm1(n, W.seed_for(34, n % 97))
    want = oracle.scan(x, "left_fold", 1)
    for mode in (0, 1, 2):
        got = fold_mode(scr, x, mode)
        assert first_diff(got, want) is None, (n, mode, first_diff(got, want))


@pytest.mark.parametrize("case", sorted(CASES))
def test_left_fold_fused_families(scr, case):
    n = 200003
    x = np.ascontiguousarray(CASES[case](n, np.float64))
    want = oracle.scan(x, "left_fold", 1)
    for mode in (0, 2):
        got = fold_mode(scr, x, mode)
        gn, wn = np.isnan(got), np.isnan(want)
        bad = (got.view(np.uint64) != want.view(np.uint64)) & ~(gn & wn) | (gn != wn)
        assert not bad.any(), (case, mode, int(np.argmax(bad)))


@pytest.mark.parametrize("form", ["exclusive", "include_initial"])
def test_left_fold_fused_shifted(scr, form):
    x = W.family3(100003)
    want = oracle.scan_ex(x, "left_fold", 1, 0.375, form)
    for mode in (0, 2):
        got = fold_mode(scr, x, mode, form)
        assert first_diff(got, want) is None, (form, mode)


RECOVERY = ("chain_fallback_kernel", "scan_local_again_kernel", "fixup_again_kernel")


@pytest.mark.parametrize("policy,B,n", [("block_dyadic", 16, 1 << 28),
                                        ("block_dyadic", 256, 1 << 28),
                                        ("left_fold", 1, 1 << 24)])
def test_parallel_chain_needs_no_recovery(scr, policy, B, n):
    """On the benchmark's value family the exact parallel chain validates
    every step: its recovery kernels (the serial chain, the local pass again,
    the fix-up again) read the chain's flag and return at once, taking
    microseconds, where a recovery of 2^20 or more steps takes milliseconds."""
    x = torch.from_numpy(W.family3(n)).to(DEV)
    y = torch.empty_like(x)
    scr.inclusive_scan(x, policy, B, out=y)
    torch.cuda.synchronize()
    scr.profile_enable(True)
    scr.inclusive_scan(x, policy, B, out=y)
    torch.cuda.synchronize()
    scr.profile_enable(False)
    prof = scr.profile_collect()
    rec = [(k, ms) for k, ms in prof if k in RECOVERY]
    assert rec, prof  # launched, as on every call
    assert all(ms < 0.5 for _, ms in rec), rec


@pytest.mark.parametrize("B", [2, 16, 256])
def test_cooperative_launch_refused(scr, B):
    """A device that refuses the cooperative launch (acted out by the
    library's hook, mode 4: nothing is launched that could fail): the chain
    runs as separate passes and a plain fix-up applies its carries; 0 ULP
    against the oracle, bit-equal to the fused pass."""
    n = B * (3 * 4096 + 5) + B // 2 + 1
    x = W.uniform_pm1(n, W.seed_for(35, B))
    want = oracle.scan(x, "block_dyadic", B)
    refused = scan_mode(scr, x, B, 4)
    assert first_diff(refused, want) is None, (B, first_diff(refused, want))
    assert first_diff(scan_mode(scr, x, B, 3), refused) is None


def test_left_fold_cooperative_launch_refused(scr):
    x = W.uniform_pm1(300007, W.seed_for(35, 1))
    want = oracle.scan(x, "left_fold", 1)
    got = fold_mode(scr, x, 4)
    assert first_diff(got, want) is None, first_diff(got, want)
