"""GPU parity of the canonical reduction against the oracle, 0 ULP (raw bits).

Cases span several tiles and pyramid levels, ragged tails (n mod L != 0 and
the case where the lanes owning the ragged row complete an extra chunk),
n < L, L = 1, L >= n, lane counts that are not powers of two, lane counts
above one block (cross-lane tree through a second pyramid), signed-zero
inits, fp64 and fp32, row- and column-batched layouts, and the full-size
benchmark shapes (sampled rows, exact-integer coverage)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def scr():
    import scan_canonical_reduce_gb300 as m
    return m


DEV = "cuda:0"


def bits(a):
    return np.asarray(a).tobytes()


def check_reduce(scr, x, L, init):
    dt = x.dtype.type
    got = scr.reduce(torch.from_numpy(x).to(DEV), L, init).cpu().numpy()[0]
    want = oracle.reduce(x, L, dt(init))
    assert bits(got) == bits(want), (x.size, L, init, got, want)


SIZES = [0, 1, 2, 3, 5, 15, 16, 17, 31, 33, 100, 255, 256, 257, 1000, 4095, 4096, 4097,
         65535, 65536, 65537, 100003, (1 << 20) + 37]
LANES = [1, 2, 3, 7, 16, 31, 128, 200, 1000, 1024, 4096]


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("L", LANES)
def test_reduce_sizes_and_lanes(scr, dtype, L):
    for n in SIZES:
        x = W.signed_pow2(n, W.seed_for(2, 17 + n % 97), dtype, -20, 20)
        check_reduce(scr, x, L, 0.5)


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("L", [1, 3, 16, 128, 1000])
def test_reduce_ragged_row_completes_a_chunk(scr, dtype, L):
    """R = 2^p - 1 full rows plus a ragged row: the lanes that own the ragged
    row have 2^p elements, so for every power-of-two chunk size their tail is a
    whole chunk."""
    for p in range(3, 15):
        for r in (1, max(1, L - 1)):
            n = L * ((1 << p) - 1) + r
            if n > (1 << 22):
                continue
            x = W.signed_pow2(n, W.seed_for(2, p * 31 + r), dtype, -20, 20)
            check_reduce(scr, x, L, -0.0)


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_reduce_inits_and_signed_zero(scr, dtype):
    x = W.signed_pow2(1000, W.seed_for(2, 5), dtype)
    for init in (0.0, -0.0, 1e30 if dtype == np.float64 else 1e20, -3.25):
        for L in (1, 16, 1024):
            check_reduce(scr, x, L, init)
    z = np.array([-0.0] * 33, dtype=dtype)
    check_reduce(scr, z, 16, -0.0)
    check_reduce(scr, z, 16, 0.0)
    check_reduce(scr, np.array([], dtype=dtype), 16, -0.0)


def test_reduce_l_one_equals_l_at_least_n(scr):
    x = W.family2((1 << 18) + 3)
    xd = torch.from_numpy(x).to(DEV)
    a = scr.reduce(xd, 1, 0.25).cpu().numpy()
    for L in (x.size, x.size + 5, 1 << 30):
        assert bits(scr.reduce(xd, L, 0.25).cpu().numpy()) == bits(a)


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_reduce_batched_rows_and_columns(scr, dtype):
    rows, cols = 300, 4096 + 37
    buf = W.signed_pow2(rows * cols, W.seed_for(4, 9), dtype)
    t = torch.from_numpy(buf).to(DEV).view(rows, cols)
    for L in (1, 16, 128, 1024):
        got = scr.reduce_batched(t, L, 0.5, dim=-1).cpu().numpy()
        want = oracle.reduce_batched(buf, rows, cols, 1, cols, L, dtype(0.5))
        assert bits(got) == bits(want), L
        gotc = scr.reduce_batched(t, L, 0.5, dim=0).cpu().numpy()
        wantc = oracle.reduce_batched(buf, cols, rows, cols, 1, L, dtype(0.5))
        assert bits(gotc) == bits(wantc), L


def test_reduce_batched_empty_and_degenerate(scr):
    t = torch.zeros(5, 0, dtype=torch.float64, device=DEV)
    assert scr.reduce_batched(t, 16, 2.0).cpu().tolist() == [2.0] * 5
    t = torch.zeros(0, 7, dtype=torch.float64, device=DEV)
    assert scr.reduce_batched(t, 16, 2.0).numel() == 0


@pytest.mark.parametrize("rows,cols", [(65536, 4096), (1024, 262144)])
def test_reduce_batched_full_size_sampled(scr, rows, cols):
    """The benchmark's row-reduce shapes in the benchmark's launch; the oracle
    recomputes sampled rows one by one."""
    x = W.family4(rows, cols)
    got = scr.reduce_batched(torch.from_numpy(x).to(DEV), 128, 0.0).cpu().numpy()
    rng = np.random.default_rng(1)
    for r in list(rng.choice(rows, 64, replace=False)) + [0, rows - 1]:
        want = oracle.reduce(x[r].copy(), 128, np.float32(0.0))
        assert bits(got[r]) == bits(want), r


@pytest.mark.parametrize("n", [(1 << 28), (1 << 28) + 37])
def test_reduce_full_size_fp64(scr, n):
    """n = 2^28 and 2^28 + 37 (the benchmark size), family-2 values, 0 ULP."""
    x = W.family2(n)
    xd = torch.from_numpy(x).to(DEV)
    for L in (16, 128, 1024):
        got = scr.reduce(xd, L, 0.0).cpu().numpy()[0]
        want = oracle.reduce(x, L, 0.0)
        assert bits(got) == bits(want), (n, L)


def test_reduce_exact_integers_two_to_thirty(scr):
    """Coverage at 2^30 elements: integer values |x| <= 2^20 make every partial
    sum exact, so any tree over all elements equals the exact integer sum."""
    n = 1 << 30
    g = torch.Generator(device=DEV).manual_seed(5)
    xi = torch.randint(-(1 << 20), (1 << 20) + 1, (n,), device=DEV, generator=g,
                       dtype=torch.int32)
    exact = int(xi.to(torch.int64).sum().item())
    x = xi.to(torch.float64)
    del xi
    for L in (16, 1024):
        got = scr.reduce(x, L, 7.0).item()
        assert got == float(exact + 7)


@pytest.mark.parametrize("dtype,L", [(np.float32, 128), (np.float64, 64)])
def test_reduce_rows_one_warp_per_row(scr, dtype, L):
    """Many contiguous rows with L = one warp's 16-byte vector width and
    n = P L take the one-warp-per-row kernel: every row against the oracle,
    for lane lengths P around the register blocks of 8 and the stack depths;
    a misaligned start, a padded row stride and a row stride that breaks
    16-byte alignment (general passes) give the same results."""
    rows = 2048
    for P in (1, 7, 8, 9, 32, 63, 64, 100, 1100, 2100):
        cols = P * L
        x = W.signed_pow2(rows * cols, W.seed_for(4, P), dtype, -20, 20).reshape(rows, cols)
        got = scr.reduce_batched(torch.from_numpy(x).to(DEV), L, 0.25).cpu().numpy()
        want = oracle.reduce_batched(x.reshape(-1), rows, cols, 1, cols, L, dtype(0.25))
        assert bits(got) == bits(want), P
    P = 9
    cols = P * L
    x = W.signed_pow2(rows * (cols + 8) + 1, W.seed_for(4, 99), dtype, -20, 20)
    base = torch.from_numpy(x).to(DEV)
    for pad, off in ((0, 1), (8, 0), (1, 0)):
        stride = cols + pad
        view = base[off:off + rows * stride].view(rows, stride)[:, :cols]
        got = scr.reduce_batched(view, L, -1.0).cpu().numpy()
        want = oracle.reduce_batched(x[off:].copy(), rows, cols, 1, stride, L, dtype(-1.0))
        assert bits(got) == bits(want), (pad, off)


def _oracle_reduce_all(x, lanes, init):
    """oracle.reduce for several lane counts at once (the oracle is
    single-threaded; its ctypes calls release the GIL)."""
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(len(lanes)) as ex:
        futs = {L: ex.submit(oracle.reduce, x, L, init) for L in lanes}
        return {L: f.result() for L, f in futs.items()}


@pytest.mark.parametrize("n", [(1 << 28), (1 << 28) + 37])
def test_reduce_full_size_fp32(scr, n):
    """The sweep's binary32 rows at n = 2^28 and 2^28 + 37 (family-2 values:
    reassociation changes the bits), L = 16, 128 and 1024, 0 ULP: the deepest
    binary32 pyramids."""
    x = W.family2(n, np.float32)
    xd = torch.from_numpy(x).to(DEV)
    lanes = (16, 128, 1024)
    want = _oracle_reduce_all(x, lanes, np.float32(0.0))
    for L in lanes:
        got = scr.reduce(xd, L, 0.0).cpu().numpy()[0]
        assert bits(got) == bits(want[L]), (n, L)


def test_reduce_full_size_fp64_two_to_thirty(scr):
    """n = 2^30, family-2 values (not integers: every level of the pyramid,
    the third included, decides bits), L = 16 and 1024, 0 ULP."""
    n = 1 << 30
    x = W.family2(n)
    xd = torch.from_numpy(x).to(DEV)
    lanes = (16, 1024)
    want = _oracle_reduce_all(x, lanes, 0.0)
    for L in lanes:
        got = scr.reduce(xd, L, 0.0).cpu().numpy()[0]
        assert bits(got) == bits(want[L]), L


@pytest.mark.parametrize("L", [16, 128])
def test_reduce_uniform01_two_to_twenty(scr, L):
    """The golden-value setup's shape: binary64, n = 2^20, U[0, 1) values,
    init +0.0, L = 16 and 128, 0 ULP."""
    x = W.family1(1 << 20)
    check_reduce(scr, x, L, 0.0)
