"""GB300 canonical reduce / scan: a thin Python binding of libcr (C ABI).

Every computation runs in libcr's CUDA kernels (``csrc/``, declared in
``include/cr.h``); this module only marshals torch tensors, streams and the
workspace into the C calls. PyTorch provides device memory and streams. There
is no CPU path: if the CUDA library has not been built, importing the binding
raises.

What is computed ("Canonical Parallel Reduction and Scan", github README
andyD123/canonical-reduce):
  * ``reduce(x, L, init)``: P4016R0's canonical reduction - lanes i mod L,
    each reduced by the iterative pairwise (shift-reduce) tree, lane results
    combined by the same tree, then op(init, R) once;
  * ``inclusive_scan(x, policy, B)``: P4229R0's prefix observations of the
    named expression policies left_fold, pairwise, iterated_pairwise,
    block_dyadic<B>;
  * batched/strided variants of both over one axis of a 2-D tensor.
Results are bit-identical to the named expression on any GPU and launch shape.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libcr.so")

CR_F32, CR_F64 = 1, 2
POLICIES = {"left_fold": 0, "pairwise": 1, "iterated_pairwise": 2, "block_dyadic": 3}
MODES = {"exclusive": 1, "include_initial": 2}  # cr_scan_mode
STATUS = {0: "CR_OK", 1: "CR_ERR_INVALID_ARG", 2: "CR_ERR_UNSUPPORTED",
          3: "CR_ERR_WORKSPACE", 4: "CR_ERR_CUDA", 5: "CR_ERR_TIMEOUT"}

# every symbol include/cr.h declares: name -> (restype, argtypes)
_P, _I64, _I32, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
_INT = ctypes.c_int
SIGNATURES = {
    "cr_reduce_workspace_bytes": (_SZ, [_I64, _I32, _INT]),
    "cr_reduce": (_INT, [_P, _I64, _I32, _P, _INT, _P, _P, _SZ, _P]),
    "cr_reduce_noalloc": (_INT, [_P, _I64, _I32, _P, _INT, _P, _P]),
    "cr_reduce_batched_workspace_bytes": (_SZ, [_I64, _I64, _I32, _INT]),
    "cr_reduce_batched": (_INT, [_P, _P, _I64, _I64, _I64, _I64, _I32, _P, _INT, _P, _SZ, _P]),
    "cr_scan_workspace_bytes": (_SZ, [_I64, _INT, _I64, _INT]),
    "cr_inclusive_scan": (_INT, [_P, _P, _I64, _INT, _I64, _INT, _P, _SZ, _P]),
    "cr_scan_batched_workspace_bytes": (_SZ, [_I64, _I64, _INT, _I64, _INT]),
    "cr_inclusive_scan_batched": (_INT, [_P, _P, _I64, _I64, _I64, _I64, _INT, _I64, _INT, _P,
                                         _SZ, _P]),
    "cr_reduce_policy_workspace_bytes": (_SZ, [_I64, _INT, _I64, _INT]),
    "cr_reduce_policy": (_INT, [_P, _I64, _INT, _I64, _INT, _P, _P, _SZ, _P]),
    "cr_scan_ex_workspace_bytes": (_SZ, [_I64, _INT, _I64, _INT, _INT]),
    "cr_scan_ex": (_INT, [_P, _P, _I64, _INT, _I64, _INT, _P, _INT, _P, _SZ, _P]),
    "cr_scan_ex_batched_workspace_bytes": (_SZ, [_I64, _I64, _INT, _I64, _INT, _INT]),
    "cr_scan_ex_batched": (_INT, [_P, _P, _I64, _I64, _I64, _I64, _I64, _I64, _INT, _I64, _INT,
                                  _P, _INT, _P, _SZ, _P]),
    "cr_inclusive_scan_host_workspace_bytes": (_SZ, [_I64, _INT, _I64, _INT]),
    "cr_inclusive_scan_host": (_INT, [_P, _P, _I64, _INT, _I64, _INT, _P, _SZ, _P]),
    "cr_reduce_host_workspace_bytes": (_SZ, [_I64, _I32, _INT]),
    "cr_reduce_host": (_INT, [_P, _I64, _I32, _P, _INT, _P, _P, _SZ, _P]),
    "cr_reduce_batched_host_workspace_bytes": (_SZ, [_I64, _I64, _I32, _INT]),
    "cr_reduce_batched_host": (_INT, [_P, _P, _I64, _I64, _I64, _I64, _I32, _P, _INT, _P, _SZ,
                                      _P]),
    "cr_inclusive_scan_batched_host_workspace_bytes": (_SZ, [_I64, _I64, _INT, _I64, _INT]),
    "cr_inclusive_scan_batched_host": (_INT, [_P, _P, _I64, _I64, _I64, _I64, _INT, _I64, _INT,
                                              _P, _SZ, _P]),
    "cr_sync_status": (_INT, [_P, _P]),
    "cr_status_string": (ctypes.c_char_p, [_INT]),
    "cr_version": (_INT, []),
    "cr_launch_count": (ctypes.c_uint64, []),
    "cr_debug_skip_publish": (None, [_I64]),
    "cr_debug_fused_fixup": (None, [_INT]),
    "cr_profile_enable": (None, [_INT]),
    "cr_profile_select": (None, [_INT]),
    "cr_profile_collect": (_INT, [_P, _P, _INT]),
    "cr_kernel_name": (ctypes.c_char_p, [_INT]),
    "cr_measure_add_peak_scratch_bytes": (_SZ, []),
    "cr_add_pairs_int": (_INT, [_P, _P, _P, _I64, _P]),
    "cr_measure_int_add_rate": (_INT, [_P, _SZ, _P, ctypes.POINTER(ctypes.c_double)]),
    "cr_measure_add_peak": (_INT, [_INT, _P, _SZ, _P, ctypes.POINTER(ctypes.c_double),
                                   ctypes.POINTER(ctypes.c_double)]),
}


class CrError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__("%s failed: %s (%s)" % (what, STATUS.get(code, code),
                                                 lib().cr_status_string(code).decode()))


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libcr (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                "libcr.so is missing (%s): build it first with "
                "`python -c 'import __graft_entry__ as g; g.build()'`" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


lib()  # fail at import time when the CUDA library is absent


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float64:
        return CR_F64
    if t.dtype == torch.float32:
        return CR_F32
    raise TypeError("libcr computes in float32 or float64, got %s" % t.dtype)


def _stream_ptr(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _resolve(device) -> torch.device:
    """A CUDA device with an explicit index ('cuda' means the current one)."""
    d = torch.device(device)
    if d.type != "cuda":
        raise ValueError("libcr runs on CUDA devices, got %s" % d)
    return d if d.index is not None else torch.device("cuda", torch.cuda.current_device())


class _Workspace:
    """One growing device workspace per (device, stream); calls on one stream
    are ordered, so they may share it."""

    def __init__(self):
        self._bufs = {}
        self._lock = threading.Lock()

    def get(self, device: torch.device, stream, nbytes: int) -> torch.Tensor:
        device = _resolve(device)
        s = torch.cuda.current_stream(device) if stream is None else stream
        key = (device.index, int(s.cuda_stream))
        with self._lock:
            buf = self._bufs.get(key)
            if buf is None or buf.numel() < nbytes:
                with torch.cuda.stream(s):  # allocated on the stream that uses it
                    buf = torch.empty(max(nbytes, 4096), dtype=torch.uint8, device=device)
                self._bufs[key] = buf
            return buf


_WS = _Workspace()


def workspace(device, stream=None, nbytes: int = 4096) -> torch.Tensor:
    """The binding's cached workspace for (device, stream), at least nbytes:
    a uint8 device tensor that grows on demand and is reused by every call
    on that stream (calls on one stream run in order). A capture into a CUDA
    graph should make one call first, so that no allocation happens inside
    the capture."""
    return _WS.get(torch.device(device), stream, nbytes)


def _check(code: int, what: str) -> None:
    if code != 0:
        raise CrError(code, what)


def _init_buffer(init, dt_code):
    if dt_code == CR_F64:
        return ctypes.c_double(float(init))
    return ctypes.c_float(float(init))


def _on_device(x: torch.Tensor, stream=None):
    """Host tensors are copied in on the call's stream (asynchronously from
    pinned memory); the caller copies the result back with _to_host."""
    if x.is_cuda:
        return x, False
    s = torch.cuda.current_stream() if stream is None else stream
    with torch.cuda.stream(s):
        return x.to("cuda", non_blocking=True), True


def _to_host(o: torch.Tensor, stream=None) -> torch.Tensor:
    """Device result -> a pinned host tensor, copied on the call's stream,
    which is then synchronised."""
    s = torch.cuda.current_stream(o.device) if stream is None else stream
    h = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    with torch.cuda.stream(s):
        h.copy_(o, non_blocking=True)
    s.synchronize()
    return h


# ---------------------------------------------------------------- reduce
def reduce(x: torch.Tensor, L: int, init=0.0, out: torch.Tensor | None = None,
           stream=None) -> torch.Tensor:
    """Canonical reduction of a 1-D tensor: op(init, tree over lane trees).

    Returns a 1-element tensor of x's dtype on x's device (a host tensor in
    gives a host tensor back, through pinned-memory copies)."""
    if x.dim() != 1:
        raise ValueError("reduce expects a 1-D tensor; use reduce_batched for 2-D")
    if not x.is_cuda:  # host buffers: one C call copies in, reduces, copies out
        xc = x.contiguous()
        dt = _dtype_code(xc)
        n = xc.numel()
        o = out if out is not None else torch.empty(1, dtype=xc.dtype, pin_memory=True)
        nb = lib().cr_reduce_host_workspace_bytes(n, int(L), dt)
        if nb == 0:
            raise ValueError("invalid reduce arguments (n=%d, L=%d)" % (n, L))
        dev = torch.device("cuda", torch.cuda.current_device())
        ws = _WS.get(dev, stream, nb)
        ini = _init_buffer(init, dt)
        _check(lib().cr_reduce_host(xc.data_ptr() if n else None, n, int(L), ctypes.byref(ini),
                                    dt, o.data_ptr(), ws.data_ptr(), ws.numel(),
                                    _stream_ptr(stream)), "cr_reduce_host")
        return o
    xd, host = _on_device(x.contiguous() if x.is_cuda else x, stream)
    xd = xd.contiguous()
    dt = _dtype_code(xd)
    n = xd.numel()
    o = out if out is not None else torch.empty(1, dtype=xd.dtype, device=xd.device)
    sp = _stream_ptr(stream)
    nb = lib().cr_reduce_workspace_bytes(n, int(L), dt)
    if nb == 0:
        raise ValueError("invalid reduce arguments (n=%d, L=%d)" % (n, L))
    ws = _WS.get(xd.device, stream, nb)
    ini = _init_buffer(init, dt)
    _check(lib().cr_reduce(xd.data_ptr() if n else None, n, int(L), ctypes.byref(ini), dt,
                           o.data_ptr(), ws.data_ptr(), ws.numel(), sp), "cr_reduce")
    return _to_host(o, stream) if host else o


def reduce_batched(x: torch.Tensor, L: int, init=0.0, dim: int = -1,
                   out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """One canonical reduction per line of a 2-D tensor along ``dim`` (any
    strides): dim=-1 reduces rows, dim=0 reduces columns."""
    if x.dim() != 2:
        raise ValueError("reduce_batched expects a 2-D tensor")
    if not x.is_cuda:  # host buffers: one C call, transfers pipelined with the kernels
        return _reduce_batched_host(x, L, init, dim, out, stream)
    xd, host = _on_device(x, stream)
    dt = _dtype_code(xd)
    d = dim % 2
    n = xd.shape[d]
    batch = xd.shape[1 - d]
    es, bs = xd.stride(d), xd.stride(1 - d)
    o = out if out is not None else torch.empty(batch, dtype=xd.dtype, device=xd.device)
    sp = _stream_ptr(stream)
    nb = lib().cr_reduce_batched_workspace_bytes(batch, n, int(L), dt)
    if nb == 0:
        raise ValueError("invalid reduce_batched arguments")
    ws = _WS.get(xd.device, stream, nb)
    ini = _init_buffer(init, dt)
    _check(lib().cr_reduce_batched(xd.data_ptr(), o.data_ptr(), batch, n, es, bs, int(L),
                                   ctypes.byref(ini), dt, ws.data_ptr(), ws.numel(), sp),
           "cr_reduce_batched")
    return _to_host(o, stream) if host else o


def _host_layout(x: torch.Tensor, dim: int):
    """(n, batch, elem_stride, batch_stride) of the lines of a 2-D tensor along
    dim, and x itself or a contiguous copy when its layout is neither rows nor
    level-major columns (the layouts the host-buffer calls move in groups)."""
    d = dim % 2
    n, batch = x.shape[d], x.shape[1 - d]
    es, bs = x.stride(d), x.stride(1 - d)
    rows = es == 1 and (bs >= n or batch == 1)
    cols = bs == 1 and (es >= batch or n == 1)
    if not (rows or cols or batch <= 1 or n <= 1):
        x = x.contiguous()
        es, bs = x.stride(d), x.stride(1 - d)
    return x, n, batch, es, bs


def _reduce_batched_host(x, L, init, dim, out, stream):
    x, n, batch, es, bs = _host_layout(x, dim)
    dt = _dtype_code(x)
    o = out if out is not None else torch.empty(batch, dtype=x.dtype, pin_memory=True)
    if o.is_cuda or o.numel() != batch or o.dtype != x.dtype or not o.is_contiguous():
        raise ValueError("out must be a contiguous host tensor of %d elements" % batch)
    nb = lib().cr_reduce_batched_host_workspace_bytes(batch, n, int(L), dt)
    if nb == 0:
        raise ValueError("invalid reduce_batched arguments")
    dev = torch.device("cuda", torch.cuda.current_device())
    ws = _WS.get(dev, stream, nb)
    ini = _init_buffer(init, dt)
    _check(lib().cr_reduce_batched_host(x.data_ptr() if x.numel() else None, o.data_ptr(),
                                        batch, n, es, bs, int(L), ctypes.byref(ini), dt,
                                        ws.data_ptr(), ws.numel(), _stream_ptr(stream)),
           "cr_reduce_batched_host")
    return o


# ------------------------------------------------------------------ scan
def _policy(policy) -> int:
    return POLICIES[policy] if isinstance(policy, str) else int(policy)


def inclusive_scan(x: torch.Tensor, policy="iterated_pairwise", B: int = 1,
                   out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Inclusive scan of a 1-D tensor under a named expression policy.
    ``out`` may be ``x`` itself (in place)."""
    if x.dim() != 1:
        raise ValueError("inclusive_scan expects a 1-D tensor")
    if not x.is_cuda:  # host buffers: one C call, transfers pipelined with the passes
        xc = x.contiguous()
        dt = _dtype_code(xc)
        n = xc.numel()
        o = out if out is not None else torch.empty(n, dtype=xc.dtype, pin_memory=True)
        if o.is_cuda or o.numel() != n or o.dtype != xc.dtype or not o.is_contiguous():
            raise ValueError("out must be a contiguous host tensor like x")
        p = _policy(policy)
        nb = lib().cr_inclusive_scan_host_workspace_bytes(n, p, int(B), dt)
        if nb == 0:
            raise ValueError("invalid scan arguments (policy=%s, B=%d)" % (policy, B))
        dev = torch.device("cuda", torch.cuda.current_device())
        ws = _WS.get(dev, stream, nb)
        _check(lib().cr_inclusive_scan_host(xc.data_ptr(), o.data_ptr(), n, p, int(B), dt,
                                            ws.data_ptr(), ws.numel(), _stream_ptr(stream)),
               "cr_inclusive_scan_host")
        return o
    xd, host = _on_device(x, stream)
    xd = xd.contiguous()
    dt = _dtype_code(xd)
    n = xd.numel()
    o = out if out is not None else torch.empty_like(xd)
    p = _policy(policy)
    sp = _stream_ptr(stream)
    nb = lib().cr_scan_workspace_bytes(n, p, int(B), dt)
    if nb == 0:
        raise ValueError("invalid scan arguments (policy=%s, B=%d)" % (policy, B))
    ws = _WS.get(xd.device, stream, nb)
    _check(lib().cr_inclusive_scan(xd.data_ptr(), o.data_ptr(), n, p, int(B), dt,
                                   ws.data_ptr(), ws.numel(), sp), "cr_inclusive_scan")
    return _to_host(o, stream) if host else o


def inclusive_scan_batched(x: torch.Tensor, policy="left_fold", B: int = 1, dim: int = 0,
                           out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Independent inclusive scans along ``dim`` of a 2-D tensor (dim=0 scans
    each column of a level-major array along its levels); the result has x's
    strides."""
    if x.dim() != 2:
        raise ValueError("inclusive_scan_batched expects a 2-D tensor")
    if not x.is_cuda:  # host buffers: one C call, transfers pipelined with the kernels
        xh, n, batch, es, bs = _host_layout(x, dim)
        dt = _dtype_code(xh)
        o = out if out is not None else torch.empty_strided(
            xh.shape, xh.stride(), dtype=xh.dtype, pin_memory=True)
        if o.is_cuda or o.stride() != xh.stride() or o.dtype != xh.dtype:
            raise ValueError("out must be a host tensor with x's strides")
        p = _policy(policy)
        nb = lib().cr_inclusive_scan_batched_host_workspace_bytes(batch, n, p, int(B), dt)
        if nb == 0:
            raise ValueError("invalid scan arguments")
        dev = torch.device("cuda", torch.cuda.current_device())
        ws = _WS.get(dev, stream, nb)
        _check(lib().cr_inclusive_scan_batched_host(
            xh.data_ptr() if xh.numel() else None, o.data_ptr() if o.numel() else None, batch,
            n, es, bs, p, int(B), dt, ws.data_ptr(), ws.numel(), _stream_ptr(stream)),
            "cr_inclusive_scan_batched_host")
        return o
    xd, host = _on_device(x, stream)
    dt = _dtype_code(xd)
    d = dim % 2
    n, batch = xd.shape[d], xd.shape[1 - d]
    es, bs = xd.stride(d), xd.stride(1 - d)
    o = out if out is not None else torch.empty_strided(xd.shape, xd.stride(), dtype=xd.dtype,
                                                        device=xd.device)
    if o.stride() != xd.stride():
        raise ValueError("out must have x's strides")
    p = _policy(policy)
    sp = _stream_ptr(stream)
    nb = lib().cr_scan_batched_workspace_bytes(batch, n, p, int(B), dt)
    if nb == 0:
        raise ValueError("invalid scan arguments")
    ws = _WS.get(xd.device, stream, nb)
    _check(lib().cr_inclusive_scan_batched(xd.data_ptr(), o.data_ptr(), batch, n, es, bs, p,
                                           int(B), dt, ws.data_ptr(), ws.numel(), sp),
           "cr_inclusive_scan_batched")
    return _to_host(o, stream) if host else o


def reduce_policy(x: torch.Tensor, policy="iterated_pairwise", B: int = 1,
                  out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """reduce<E>(x): the root of the named expression whose prefixes
    inclusive_scan observes (1-element tensor; x must not be empty)."""
    if x.dim() != 1:
        raise ValueError("reduce_policy expects a 1-D tensor")
    xd, host = _on_device(x, stream)
    xd = xd.contiguous()
    dt = _dtype_code(xd)
    n = xd.numel()
    p = _policy(policy)
    o = out if out is not None else torch.empty(1, dtype=xd.dtype, device=xd.device)
    sp = _stream_ptr(stream)
    nb = lib().cr_reduce_policy_workspace_bytes(n, p, int(B), dt)
    if nb == 0:
        raise ValueError("invalid reduce_policy arguments (n=%d, policy=%s, B=%d)" %
                         (n, policy, B))
    ws = _WS.get(xd.device, stream, nb)
    _check(lib().cr_reduce_policy(xd.data_ptr(), n, p, int(B), dt, o.data_ptr(), ws.data_ptr(),
                                  ws.numel(), sp), "cr_reduce_policy")
    return _to_host(o, stream) if host else o


def _scan_ex(x, policy, B, init, mode, out, stream, what):
    if x.dim() != 1:
        raise ValueError("%s expects a 1-D tensor" % what)
    xd, host = _on_device(x, stream)
    xd = xd.contiguous()
    dt = _dtype_code(xd)
    n = xd.numel()
    md = MODES[mode]
    m = n + (1 if md == 2 else 0)
    o = out if out is not None else torch.empty(m, dtype=xd.dtype, device=xd.device)
    if o.dim() != 1 or not o.is_contiguous() or o.numel() < m or o.dtype != xd.dtype:
        raise ValueError("out must be a contiguous 1-D tensor of %d elements of x's dtype" % m)
    p = _policy(policy)
    sp = _stream_ptr(stream)
    nb = lib().cr_scan_ex_workspace_bytes(n, p, int(B), md, dt)
    if nb == 0:
        raise ValueError("invalid scan arguments (policy=%s, B=%d)" % (policy, B))
    ws = _WS.get(xd.device, stream, nb)
    ini = _init_buffer(init, dt)
    _check(lib().cr_scan_ex(xd.data_ptr() if n else None, o.data_ptr(), n, p, int(B), md,
                            ctypes.byref(ini), dt, ws.data_ptr(), ws.numel(), sp), "cr_scan_ex")
    return _to_host(o, stream) if host else o


def exclusive_scan(x: torch.Tensor, policy="iterated_pairwise", B: int = 1, init=0.0,
                   out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Exclusive scan of a 1-D tensor: out[0] = init, out[k] = init op y[k-1]
    with y the inclusive scan of the policy (n outputs; ``out`` may be ``x``)."""
    return _scan_ex(x, policy, B, init, "exclusive", out, stream, "exclusive_scan")


def scan_include_initial(x: torch.Tensor, policy="iterated_pairwise", B: int = 1, init=0.0,
                         out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The include_initial form: n + 1 outputs, out[0] = init and
    out[k] = init op y[k-1] for k = 1..n."""
    return _scan_ex(x, policy, B, init, "include_initial", out, stream, "scan_include_initial")


def _scan_ex_batched(x, policy, B, init, dim, mode, out, stream, what):
    if x.dim() != 2:
        raise ValueError("%s expects a 2-D tensor" % what)
    xd, host = _on_device(x, stream)
    dt = _dtype_code(xd)
    d = dim % 2
    n, batch = xd.shape[d], xd.shape[1 - d]
    es, bs = xd.stride(d), xd.stride(1 - d)
    md = MODES[mode]
    m = n + (1 if md == 2 else 0)
    shape = (m, batch) if d == 0 else (batch, m)
    o = out if out is not None else torch.empty(shape, dtype=xd.dtype, device=xd.device)
    if tuple(o.shape) != shape or o.dtype != xd.dtype:
        raise ValueError("out must have shape %s and x's dtype" % (shape,))
    oes, obs = o.stride(d), o.stride(1 - d)
    p = _policy(policy)
    sp = _stream_ptr(stream)
    nb = lib().cr_scan_ex_batched_workspace_bytes(batch, n, p, int(B), md, dt)
    if nb == 0:
        raise ValueError("invalid scan arguments")
    ws = _WS.get(xd.device, stream, nb)
    ini = _init_buffer(init, dt)
    _check(lib().cr_scan_ex_batched(xd.data_ptr() if xd.numel() else None, o.data_ptr(), batch,
                                    n, es, bs, oes, obs, p, int(B), md, ctypes.byref(ini), dt,
                                    ws.data_ptr(), ws.numel(), sp), "cr_scan_ex_batched")
    return _to_host(o, stream) if host else o


def exclusive_scan_batched(x: torch.Tensor, policy="left_fold", B: int = 1, init=0.0,
                           dim: int = 0, out: torch.Tensor | None = None,
                           stream=None) -> torch.Tensor:
    """Independent exclusive scans along ``dim`` of a 2-D tensor."""
    return _scan_ex_batched(x, policy, B, init, dim, "exclusive", out, stream,
                            "exclusive_scan_batched")


def scan_include_initial_batched(x: torch.Tensor, policy="left_fold", B: int = 1, init=0.0,
                                 dim: int = 0, out: torch.Tensor | None = None,
                                 stream=None) -> torch.Tensor:
    """Independent include_initial scans along ``dim``: n levels give n + 1
    values (e.g. cell values to interface values of a level-major column
    array, the first being init)."""
    return _scan_ex_batched(x, policy, B, init, dim, "include_initial", out, stream,
                            "scan_include_initial_batched")


def sync_status(device=None, stream=None) -> None:
    """Synchronise the stream and raise if the last call on its workspace
    reported a device-side timeout."""
    dev = _resolve("cuda" if device is None else device)
    sp = _stream_ptr(stream)
    ws = _WS.get(dev, stream, 4096)
    _check(lib().cr_sync_status(ws.data_ptr(), sp), "cr_sync_status")


def launch_count() -> int:
    """Kernels libcr has enqueued since it was loaded."""
    return int(lib().cr_launch_count())


def profile_enable(on: bool = True) -> None:
    """Bracket every later libcr launch with CUDA events on its stream."""
    lib().cr_profile_enable(1 if on else 0)


def profile_select(kernel=None) -> None:
    """Record only the launches of the kernel named ``kernel`` (a name
    profile_collect returns) while profiling is on; None records every one."""
    kid = -1
    if kernel is not None:
        for i in range(256):  # ids run from 0 until the name is "unknown"
            nm = lib().cr_kernel_name(i).decode()
            if nm == "unknown":
                break
            if nm == kernel:
                kid = i
                break
        if kid < 0:
            raise ValueError("no libcr kernel named %r" % kernel)
    lib().cr_profile_select(kid)


def profile_collect():
    """[(kernel name, device ms)] of the launches recorded since the last call."""
    cap = 1 << 16
    ids = (ctypes.c_int * cap)()
    ms = (ctypes.c_float * cap)()
    n = lib().cr_profile_collect(ids, ms, cap)
    return [(lib().cr_kernel_name(ids[i]).decode(), float(ms[i])) for i in range(min(n, cap))]


def measure_add_peak(dtype=torch.float64, device="cuda", stream=None):
    """(adds per second over the GPU, dependent-add latency in ns) of
    round-to-nearest adds of ``dtype``, measured by libcr's calibration
    kernels on ``device``."""
    dt = CR_F64 if dtype == torch.float64 else CR_F32
    with torch.cuda.device(torch.device(device)):
        nb = lib().cr_measure_add_peak_scratch_bytes()
        scratch = torch.empty(max(int(nb), 256), dtype=torch.uint8, device=device)
        rate, lat = ctypes.c_double(0), ctypes.c_double(0)
        _check(lib().cr_measure_add_peak(dt, scratch.data_ptr(), scratch.numel(),
                                         _stream_ptr(stream), ctypes.byref(rate),
                                         ctypes.byref(lat)), "cr_measure_add_peak")
    return rate.value, lat.value


def add_pairs_int(a: torch.Tensor, b: torch.Tensor, stream=None) -> torch.Tensor:
    """Elementwise binary64 a + b through libcr's integer-pipe add."""
    if a.dtype != torch.float64 or b.dtype != torch.float64 or a.shape != b.shape:
        raise TypeError("float64 tensors of one shape")
    a, b = a.contiguous(), b.contiguous()
    out = torch.empty_like(a)
    _check(lib().cr_add_pairs_int(a.data_ptr(), b.data_ptr(), out.data_ptr(), a.numel(),
                                  _stream_ptr(stream)), "cr_add_pairs_int")
    return out


def measure_int_add_rate(device="cuda", stream=None) -> float:
    """Adds per second of the integer-pipe binary64 add over the GPU."""
    with torch.cuda.device(torch.device(device)):
        nb = lib().cr_measure_add_peak_scratch_bytes()
        scratch = torch.empty(max(int(nb), 256), dtype=torch.uint8, device=device)
        rate = ctypes.c_double(0)
        _check(lib().cr_measure_int_add_rate(scratch.data_ptr(), scratch.numel(),
                                             _stream_ptr(stream), ctypes.byref(rate)),
               "cr_measure_int_add_rate")
    return rate.value


__all__ = ["reduce", "reduce_batched", "reduce_policy", "inclusive_scan",
           "inclusive_scan_batched",
           "exclusive_scan", "scan_include_initial", "exclusive_scan_batched",
           "scan_include_initial_batched", "MODES", "sync_status", "lib", "workspace", "launch_count", "profile_enable", "profile_collect", "measure_add_peak", "add_pairs_int", "measure_int_add_rate", "CrError", "POLICIES", "SIGNATURES"]
