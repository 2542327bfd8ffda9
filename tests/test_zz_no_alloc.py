"""cr_reduce_noalloc: the canonical reduction for callers that cannot
allocate device memory (e.g. a plugin whose host framework owns all device
memory, or a path that must not pay cudaMalloc's possible device-wide
synchronisation). Its scratch is a 16 MiB device array built into libcr.

Called here through the C ABI (ctypes) and compared, bit for bit, with
cr_reduce on a caller-provided workspace and with the oracle, twice in a row:
the shared array keeps the previous call's contents, so the second call checks
that nothing stale leaks into a result (a large call followed by a small one
included). Runs alone in a fresh process or after the other tests."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def lib():
    import scan_canonical_reduce_gb300 as scr
    return scr.lib()


def call_reduce(lib, x, L, init, out, ws, stream):
    dt = 2 if x.dtype == torch.float64 else 1
    ini = ctypes.c_double(init) if dt == 2 else ctypes.c_float(init)
    return lib.cr_reduce(x.data_ptr(), x.numel(), L, ctypes.byref(ini), dt, out.data_ptr(),
                         ws.data_ptr(), ws.numel(), stream)


def call_noalloc(lib, x, L, init, out, stream):
    dt = 2 if x.dtype == torch.float64 else 1
    ini = ctypes.c_double(init) if dt == 2 else ctypes.c_float(init)
    return lib.cr_reduce_noalloc(x.data_ptr(), x.numel(), L, ctypes.byref(ini), dt,
                                 out.data_ptr(), stream)


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_noalloc_matches_reduce_twice(lib, dtype):
    stream = torch.cuda.current_stream(DEV).cuda_stream
    tdt = torch.float64 if dtype == np.float64 else torch.float32
    # (2^26 + 3, 16) then (1000, 7): a small call right after a large one
    cases = [(1, 16), (100003, 16), ((1 << 20) + 37, 128), ((1 << 24) + 5, 1024),
             ((1 << 26) + 3, 16), (1000, 7), ((1 << 22) + 1, 1)]
    for n, L in cases:
        xh = W.signed_pow2(n, W.seed_for(2, n % 89), dtype)
        x = torch.from_numpy(xh).to(DEV)
        nb = lib.cr_reduce_workspace_bytes(n, L, 2 if tdt == torch.float64 else 1)
        ws = torch.empty(nb, dtype=torch.uint8, device=DEV)
        ref = torch.empty(1, dtype=tdt, device=DEV)
        assert call_reduce(lib, x, L, 0.5, ref, ws, stream) == 0
        want = np.asarray(oracle.reduce(xh, L, dtype(0.5))).tobytes()
        for _ in range(2):  # two calls in a row on the shared array
            out = torch.full((1,), float("nan"), dtype=tdt, device=DEV)
            assert call_noalloc(lib, x, L, 0.5, out, stream) == 0
            torch.cuda.synchronize()
            got = out.cpu().numpy().tobytes()
            assert got == ref.cpu().numpy().tobytes(), (n, L)
            assert got == want, (n, L)


def test_noalloc_rejects_oversized_call(lib):
    """n = 2^30 with L = 1024 needs about 34 MiB of scratch: rejected before
    anything is enqueued (the small buffer below is never read, and out keeps
    its NaN)."""
    x = torch.zeros(16, dtype=torch.float64, device=DEV)
    out = torch.full((1,), float("nan"), dtype=torch.float64, device=DEV)
    before = lib.cr_launch_count()
    ini = ctypes.c_double(0.0)
    rc = lib.cr_reduce_noalloc(x.data_ptr(), 1 << 30, 1024, ctypes.byref(ini), 2,
                               out.data_ptr(), torch.cuda.current_stream(DEV).cuda_stream)
    assert rc == 3  # CR_ERR_WORKSPACE
    torch.cuda.synchronize()
    launches = lib.cr_launch_count()
    assert launches == before
    assert np.isnan(out.cpu().numpy()[0])
    assert lib.cr_reduce_noalloc(x.data_ptr(), 16, 0, ctypes.byref(ini), 2, out.data_ptr(),
                                 None) == 1  # L < 1
