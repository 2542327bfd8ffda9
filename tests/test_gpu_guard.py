"""Accesses stay inside their buffers: a stand-in for a device memory checker,
which this pool does not run. Every call family runs through the C ABI on
buffers placed inside larger allocations whose surroundings hold a canary
byte pattern, with workspaces of exactly the size the matching
*_workspace_bytes call returns. Afterwards the canaries are intact, the
input is unchanged (out-of-place calls), and in pitched layouts every
element between the outputs still holds the canary. Output values are the
parity tests' business; here they are only checked against the binding's
result for the same call."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
GUARD = 1 << 16
CANARY = 0xA5
F64, F32 = 2, 1
POL = {"left_fold": 0, "pairwise": 1, "iterated_pairwise": 2, "block_dyadic": 3}


@pytest.fixture(scope="module")
def scr():
    import scan_canonical_reduce_gb300 as m
    return m


class Guarded:
    """nbytes of device memory between two canary bands of GUARD bytes."""

    def __init__(self, nbytes, fill=CANARY):
        self.nbytes = int(nbytes)
        self.fill = fill
        self.buf = torch.full((GUARD + self.nbytes + GUARD,), fill, dtype=torch.uint8,
                              device=DEV)
        self.ptr = self.buf.data_ptr() + GUARD  # 256-byte aligned like the allocation

    def view(self, dtype):
        return self.buf[GUARD:GUARD + self.nbytes].view(dtype)

    def bands_intact(self):
        return bool((self.buf[:GUARD] == self.fill).all()) and \
            bool((self.buf[GUARD + self.nbytes:] == self.fill).all())


def guarded_input(values):
    """The input between bands of all-ones bytes, a NaN in either precision:
    a read past the input that reached a result would make it NaN, and the
    comparison with the binding's result would fail."""
    g = Guarded(values.nbytes, fill=0xFF)
    g.view(torch.float64 if values.dtype == np.float64 else torch.float32).copy_(
        torch.from_numpy(values))
    return g


def init_of(dt, v):
    return ctypes.c_double(v) if dt == F64 else ctypes.c_float(v)


def run(lib, code, ws):
    """The call's status, then its device-side status word (after a sync)."""
    assert code == 0, lib.cr_status_string(code)
    assert lib.cr_sync_status(ws.ptr, None) == 0
    torch.cuda.synchronize()


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_reduce(scr, dtype):
    lib = scr.lib()
    dt = F64 if dtype == np.float64 else F32
    tdt = torch.float64 if dt == F64 else torch.float32
    n = (1 << 20) + 37
    xv = W.family2(n, dtype)
    for L in (1, 16, 1000):
        x = guarded_input(xv)
        before = x.buf.clone()
        out = Guarded(xv.itemsize)
        ws = Guarded(lib.cr_reduce_workspace_bytes(n, L, dt))
        run(lib, lib.cr_reduce(x.ptr, n, L, ctypes.byref(init_of(dt, 0.5)), dt, out.ptr, ws.ptr,
                               ws.nbytes, None), ws)
        assert torch.equal(x.buf, before), L
        assert out.bands_intact() and ws.bands_intact(), L
        want = scr.reduce(torch.from_numpy(xv).to(DEV), L, 0.5)
        assert torch.equal(out.view(tdt), want), L


def test_reduce_batched_rows_and_pitched_columns(scr):
    lib = scr.lib()
    rows, cols = 300, 5000
    xv = W.family4(rows, cols).astype(np.float64).ravel()
    x = guarded_input(xv)
    before = x.buf.clone()
    out = Guarded(rows * 8)
    ws = Guarded(lib.cr_reduce_batched_workspace_bytes(rows, cols, 128, F64))
    run(lib, lib.cr_reduce_batched(x.ptr, out.ptr, rows, cols, 1, cols, 128,
                                   ctypes.byref(init_of(F64, 0.0)), F64, ws.ptr, ws.nbytes,
                                   None), ws)
    assert torch.equal(x.buf, before) and out.bands_intact() and ws.bands_intact()
    # columns of a level-major array with a pitch wider than its columns
    levels, ncols, pitch = 90, 20000, 20003
    xv = W.family5(levels, pitch)
    x = guarded_input(xv)
    before = x.buf.clone()
    out = Guarded(ncols * 8)
    ws = Guarded(lib.cr_reduce_batched_workspace_bytes(ncols, levels, 16, F64))
    run(lib, lib.cr_reduce_batched(x.ptr, out.ptr, ncols, levels, pitch, 1, 16,
                                   ctypes.byref(init_of(F64, 0.0)), F64, ws.ptr, ws.nbytes,
                                   None), ws)
    assert torch.equal(x.buf, before) and out.bands_intact() and ws.bands_intact()
    want = scr.reduce_batched(torch.from_numpy(xv).to(DEV).view(levels, pitch)[:, :ncols], 16,
                              0.0, dim=0)
    assert torch.equal(out.view(torch.float64), want)


@pytest.mark.parametrize("policy,B", [("iterated_pairwise", 1), ("pairwise", 1),
                                      ("left_fold", 1), ("block_dyadic", 16),
                                      ("block_dyadic", 256), ("block_dyadic", 4096)])
@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_scan(scr, policy, B, dtype):
    lib = scr.lib()
    dt = F64 if dtype == np.float64 else F32
    tdt = torch.float64 if dt == F64 else torch.float32
    n = (1 << 20) + 37
    xv = W.family3(n).astype(dtype)
    want = scr.inclusive_scan(torch.from_numpy(xv).to(DEV), policy, B)
    nb = lib.cr_scan_workspace_bytes(n, POL[policy], B, dt)
    # out of place
    x = guarded_input(xv)
    before = x.buf.clone()
    out = Guarded(xv.nbytes)
    ws = Guarded(nb)
    run(lib, lib.cr_inclusive_scan(x.ptr, out.ptr, n, POL[policy], B, dt, ws.ptr, ws.nbytes,
                                   None), ws)
    assert torch.equal(x.buf, before) and out.bands_intact() and ws.bands_intact()
    assert torch.equal(out.view(tdt), want)
    # in place
    x = guarded_input(xv)
    ws = Guarded(nb)
    run(lib, lib.cr_inclusive_scan(x.ptr, x.ptr, n, POL[policy], B, dt, ws.ptr, ws.nbytes,
                                   None), ws)
    assert x.bands_intact() and ws.bands_intact()
    assert torch.equal(x.view(tdt), want)


@pytest.mark.parametrize("policy,B", [("left_fold", 1), ("block_dyadic", 16),
                                      ("iterated_pairwise", 1), ("pairwise", 1)])
def test_scan_batched_pitched_columns(scr, policy, B):
    """out uses x's strides: the pitch's gap elements must keep the canary."""
    lib = scr.lib()
    levels, ncols, pitch = 90, 20000, 20003
    xv = W.family5(levels, pitch)
    x = guarded_input(xv)
    before = x.buf.clone()
    out = Guarded(xv.nbytes)
    ws = Guarded(lib.cr_scan_batched_workspace_bytes(ncols, levels, POL[policy], B, F64))
    run(lib, lib.cr_inclusive_scan_batched(x.ptr, out.ptr, ncols, levels, pitch, 1, POL[policy],
                                           B, F64, ws.ptr, ws.nbytes, None), ws)
    assert torch.equal(x.buf, before) and out.bands_intact() and ws.bands_intact()
    o = out.buf[GUARD:GUARD + out.nbytes].view(levels, pitch * 8)
    assert bool((o[:, ncols * 8:] == CANARY).all())  # the gaps of every level
    xd = torch.from_numpy(xv).to(DEV).view(levels, pitch)[:, :ncols]
    want = scr.inclusive_scan_batched(xd, policy, B, dim=0)
    assert torch.equal(out.view(torch.float64).view(levels, pitch)[:, :ncols], want)


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("policy,B", [("iterated_pairwise", 1), ("block_dyadic", 16),
                                      ("left_fold", 1), ("pairwise", 1)])
def test_scan_ex(scr, mode, policy, B):
    lib = scr.lib()
    n = (1 << 20) + 37
    m = n + 1 if mode == 2 else n
    xv = W.family3(n)
    x = guarded_input(xv)
    before = x.buf.clone()
    out = Guarded(m * 8)
    ws = Guarded(lib.cr_scan_ex_workspace_bytes(n, POL[policy], B, mode, F64))
    run(lib, lib.cr_scan_ex(x.ptr, out.ptr, n, POL[policy], B, mode,
                            ctypes.byref(init_of(F64, 0.25)), F64, ws.ptr, ws.nbytes, None), ws)
    assert torch.equal(x.buf, before) and out.bands_intact() and ws.bands_intact()
    f = scr.exclusive_scan if mode == 1 else scr.scan_include_initial
    want = f(torch.from_numpy(xv).to(DEV), policy, B, 0.25)
    assert torch.equal(out.view(torch.float64), want)


def test_scan_ex_batched_include_initial_columns(scr):
    lib = scr.lib()
    levels, ncols, pitch = 90, 20000, 20003
    xv = W.family5(levels, pitch)
    x = guarded_input(xv)
    before = x.buf.clone()
    out = Guarded((levels + 1) * pitch * 8)
    ws = Guarded(lib.cr_scan_ex_batched_workspace_bytes(ncols, levels, POL["block_dyadic"], 16, 2,
                                                        F64))
    run(lib, lib.cr_scan_ex_batched(x.ptr, out.ptr, ncols, levels, pitch, 1, pitch, 1,
                                    POL["block_dyadic"], 16, 2, ctypes.byref(init_of(F64, 0.25)),
                                    F64, ws.ptr, ws.nbytes, None), ws)
    assert torch.equal(x.buf, before) and out.bands_intact() and ws.bands_intact()
    o = out.buf[GUARD:GUARD + out.nbytes].view(levels + 1, pitch * 8)
    assert bool((o[:, ncols * 8:] == CANARY).all())


@pytest.mark.parametrize("policy,B", [("left_fold", 1), ("block_dyadic", 16),
                                      ("block_dyadic", 4096), ("pairwise", 1)])
def test_reduce_policy(scr, policy, B):
    lib = scr.lib()
    n = (1 << 20) + 37
    xv = W.family3(n)
    x = guarded_input(xv)
    before = x.buf.clone()
    out = Guarded(8)
    ws = Guarded(lib.cr_reduce_policy_workspace_bytes(n, POL[policy], B, F64))
    run(lib, lib.cr_reduce_policy(x.ptr, n, POL[policy], B, F64, out.ptr, ws.ptr, ws.nbytes,
                                  None), ws)
    assert torch.equal(x.buf, before) and out.bands_intact() and ws.bands_intact()
    want = scr.reduce_policy(torch.from_numpy(xv).to(DEV), policy, B)
    assert torch.equal(out.view(torch.float64), want)


def test_host_buffer_calls(scr):
    """Host buffers inside larger host arrays and the device buffer inside
    canary bands: the pipelined copies stay in range on both sides."""
    lib = scr.lib()
    n = (1 << 22) + 37
    xv = W.family3(n)
    pad = GUARD // 8
    host_out = np.full(n + 2 * pad, np.nan)
    dev = Guarded(lib.cr_inclusive_scan_host_workspace_bytes(n, POL["block_dyadic"], 16, F64))
    xh = np.ascontiguousarray(xv)
    rc = lib.cr_inclusive_scan_host(xh.ctypes.data, host_out[pad:].ctypes.data, n,
                                    POL["block_dyadic"], 16, F64, dev.ptr, dev.nbytes, None)
    assert rc == 0
    torch.cuda.synchronize()
    assert dev.bands_intact()
    assert np.isnan(host_out[:pad]).all() and np.isnan(host_out[pad + n:]).all()
    want = scr.inclusive_scan(torch.from_numpy(xv).to(DEV), "block_dyadic", 16).cpu().numpy()
    assert host_out[pad:pad + n].tobytes() == want.tobytes()
    dev = Guarded(lib.cr_reduce_host_workspace_bytes(n, 16, F64))
    out = ctypes.c_double(float("nan"))
    rc = lib.cr_reduce_host(xh.ctypes.data, n, 16, ctypes.byref(init_of(F64, 0.5)), F64,
                            ctypes.addressof(out), dev.ptr, dev.nbytes, None)
    assert rc == 0
    torch.cuda.synchronize()
    assert dev.bands_intact()
    assert out.value == float(scr.reduce(torch.from_numpy(xv).to(DEV), 16, 0.5)[0])
