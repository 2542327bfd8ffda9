"""cr_reduce_noalloc: the canonical reduction for callers that cannot
allocate device memory (e.g. a plugin whose host framework owns all device
memory, or a path that must not pay cudaMalloc's possible device-wide
synchronisation). Its scratch is a 16 MiB device array built into libcr.

Called here through the C ABI (ctypes) and compared, bit for bit, with
cr_reduce on a caller-provided workspace, twice in a row: the shared array
keeps the previous call's contents, so the second call checks that nothing
stale leaks into a result. Runs alone in a fresh process or after the other
tests."""
import ctypes

import numpy as np
import pytest
import torch

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
    cases = [(1, 16), (1000, 7), (100003, 16), ((1 << 20) + 37, 128), ((1 << 24) + 5, 1024),
             ((1 << 26) + 3, 16), ((1 << 22) + 1, 1)]
    for n, L in cases:
        x = torch.from_numpy(W.signed_pow2(n, W.seed_for(2, n % 89), dtype)).to(DEV)
        nb = lib.cr_reduce_workspace_bytes(n, L, 2 if tdt == torch.float64 else 1)
        ws = torch.empty(nb, dtype=torch.uint8, device=DEV)
        ref = torch.empty(1, dtype=tdt, device=DEV)
        assert call_reduce(lib, x, L, 0.5, ref, ws, stream) == 0
        for _ in range(2):  # two calls in a row on the shared array
            out = torch.full((1,), float("nan"), dtype=tdt, device=DEV)
            assert call_noalloc(lib, x, L, 0.5, out, stream) == 0
            torch.cuda.synchronize()
            assert out.cpu().numpy().tobytes() == ref.cpu().numpy().tobytes(), (n, L)


def test_noalloc_rejects_oversized_call(lib):
    """n = 2^30 with L = 1024 needs about 34 MiB of scratch: rejected before
    anything is enqueued (the small buffer below is never read)."""
    x = torch.zeros(16, dtype=torch.float64, device=DEV)
    out = torch.zeros(1, dtype=torch.float64, device=DEV)
    ini = ctypes.c_double(0.0)
    rc = lib.cr_reduce_noalloc(x.data_ptr(), 1 << 30, 1024, ctypes.byref(ini), 2,
                               out.data_ptr(), torch.cuda.current_stream(DEV).cuda_stream)
    assert rc == 3  # CR_ERR_WORKSPACE
    assert lib.cr_reduce_noalloc(x.data_ptr(), 16, 0, ctypes.byref(ini), 2, out.data_ptr(),
                                 None) == 1  # L < 1
