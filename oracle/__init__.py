"""Oracle: plain single-threaded CPU evaluation of the canonical reduction
(P4016R0) and the canonical scan policies (P4229R0).

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package. It shares
no code with the CUDA library (``scan_canonical_reduce_gb300``) and imports
nothing from it.

Definitions follow "Canonical Parallel Reduction and Scan" (github README
andyD123/canonical-reduce), sections "P4016R0 - Key Design Points" and
"P4229R0 - Summary / Key Design Points"; the C++ source ``cro.cpp`` states
each definition and each reading next to its code.

All arrays are numpy arrays; float64 inputs are evaluated in binary64 and
float32 inputs in binary32 (the page fixes the element type as the
arithmetic type: no widening).
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import build as _build

POLICIES = {
    "left_fold": 0,
    "pairwise": 1,
    "iterated_pairwise": 2,
    "block_dyadic": 3,
    "block_dyadic_alt": 4,
}

_lib = None


def lib() -> ctypes.CDLL:
    """Load (building first if needed) the oracle's shared library."""
    global _lib
    if _lib is None:
        path = _build.build()
        _lib = ctypes.CDLL(path)
        _declare(_lib)
    return _lib


def _declare(L: ctypes.CDLL) -> None:
    P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    D, F, U64 = ctypes.c_double, ctypes.c_float, ctypes.c_uint64
    sig = {
        "cro_tree_f64": (D, [P, I64, I64]),
        "cro_tree_f32": (F, [P, I64, I64]),
        "cro_reduce_f64": (D, [P, I64, I64, I64, D]),
        "cro_reduce_f32": (F, [P, I64, I64, I64, F]),
        "cro_reduce_modp": (U64, [P, I64, I64, U64]),
        "cro_reduce_batched_f64": (None, [P, P, I64, I64, I64, I64, I64, D]),
        "cro_reduce_batched_f32": (None, [P, P, I64, I64, I64, I64, I64, F]),
        "cro_scan_f64": (I32, [P, I64, P, I64, I64, I32, I64]),
        "cro_scan_f32": (I32, [P, I64, P, I64, I64, I32, I64]),
        "cro_scan_modp": (I32, [P, P, I64, I32, I64]),
        "cro_scan_batched_f64": (I32, [P, P, I64, I64, I64, I64, I32, I64]),
        "cro_scan_batched_f32": (I32, [P, P, I64, I64, I64, I64, I32, I64]),
        "cro_scan_ex_f64": (I32, [P, I64, P, I64, I64, I32, I64, D, I32]),
        "cro_scan_ex_f32": (I32, [P, I64, P, I64, I64, I32, I64, F, I32]),
        "cro_scan_ex_modp": (I32, [P, P, I64, I32, I64, U64, I32]),
        "cro_scan_ex_batched_f64": (I32, [P, P, I64, I64, I64, I64, I64, I64, I32, I64, D,
                                          I32]),
        "cro_scan_ex_batched_f32": (I32, [P, P, I64, I64, I64, I64, I64, I64, I32, I64, F,
                                          I32]),
        "cro_sym_scan_ex": (I64, [I64, I32, I64, I32, I64, P, I64]),
        "cro_reduce_policy_f64": (I32, [P, I64, I32, I64, P]),
        "cro_reduce_policy_f32": (I32, [P, I64, I32, I64, P]),
        "cro_reduce_policy_modp": (I32, [P, I64, I32, I64, P]),
        "cro_sym_tree": (I64, [I64, P, I64]),
        "cro_sym_reduce": (I64, [I64, I64, P, I64]),
        "cro_sym_scan": (I64, [I64, I32, I64, I64, P, I64]),
        "cro_sym_reduce_policy": (I64, [I64, I32, I64, P, I64]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _kind(x: np.ndarray) -> str:
    if x.dtype == np.float64:
        return "f64"
    if x.dtype == np.float32:
        return "f32"
    raise TypeError("oracle evaluates float64 or float32 arrays, got %s" % x.dtype)


def _policy(p) -> int:
    return POLICIES[p] if isinstance(p, str) else int(p)


def tree(v: np.ndarray) -> np.floating:
    """tree(v_0..v_{m-1}) for a 1-D array with m >= 1."""
    v = np.ascontiguousarray(v)
    if v.size < 1:
        raise ValueError("tree() needs at least one operand")
    k = _kind(v)
    fn = getattr(lib(), "cro_tree_" + k)
    return v.dtype.type(fn(_ptr(v), v.size, 1))


def reduce(x: np.ndarray, L: int, init=0.0) -> np.floating:
    """Canonical reduction op(init, tree(R_0..R_{m-1})) of a 1-D array."""
    x = np.ascontiguousarray(x)
    if L < 1:
        raise ValueError("L must be >= 1")
    k = _kind(x)
    init = x.dtype.type(init)
    fn = getattr(lib(), "cro_reduce_" + k)
    return x.dtype.type(fn(_ptr(x), x.size, 1, int(L), init))


def reduce_strided(buf: np.ndarray, offset: int, n: int, stride: int, L: int,
                   init=0.0) -> np.floating:
    """Canonical reduction of buf[offset + i*stride], i < n (flat buffer)."""
    assert buf.flags.c_contiguous and buf.ndim == 1
    k = _kind(buf)
    if n > 0:
        last = offset + (n - 1) * stride
        assert 0 <= offset < buf.size and 0 <= last < buf.size
    fn = getattr(lib(), "cro_reduce_" + k)
    return buf.dtype.type(fn(_ptr(buf) + offset * buf.itemsize, n, stride, int(L),
                             buf.dtype.type(init)))


def reduce_batched(buf: np.ndarray, batch: int, n: int, elem_stride: int,
                   batch_stride: int, L: int, init=0.0) -> np.ndarray:
    """One canonical reduction per sequence b: buf[b*batch_stride + i*elem_stride]."""
    assert buf.flags.c_contiguous and buf.ndim == 1
    k = _kind(buf)
    _check_extent(buf, batch, n, elem_stride, batch_stride)
    out = np.empty(batch, dtype=buf.dtype)
    fn = getattr(lib(), "cro_reduce_batched_" + k)
    fn(_ptr(buf), _ptr(out), batch, n, elem_stride, batch_stride, int(L),
       buf.dtype.type(init))
    return out


def scan(x: np.ndarray, policy, B: int = 1) -> np.ndarray:
    """Inclusive scan of a 1-D array under a named policy."""
    x = np.ascontiguousarray(x)
    k = _kind(x)
    y = np.empty_like(x)
    rc = getattr(lib(), "cro_scan_" + k)(_ptr(x), 1, _ptr(y), 1, x.size, _policy(policy),
                                         int(B))
    if rc:
        raise ValueError("bad policy or block size")
    return y


def scan_batched(buf: np.ndarray, batch: int, n: int, elem_stride: int,
                 batch_stride: int, policy, B: int = 1) -> np.ndarray:
    """Batched inclusive scans; the result uses the input's strides (a copy of
    ``buf`` with every scanned position overwritten)."""
    assert buf.flags.c_contiguous and buf.ndim == 1
    k = _kind(buf)
    _check_extent(buf, batch, n, elem_stride, batch_stride)
    y = buf.copy()
    rc = getattr(lib(), "cro_scan_batched_" + k)(_ptr(buf), _ptr(y), batch, n, elem_stride,
                                                 batch_stride, _policy(policy), int(B))
    if rc:
        raise ValueError("bad policy or block size")
    return y


SCAN_MODES = {"exclusive": 0, "include_initial": 1}


def _mode(mode) -> int:
    return SCAN_MODES[mode] if isinstance(mode, str) else int(mode)


def scan_ex(x: np.ndarray, policy, B: int = 1, init=0.0, mode="exclusive") -> np.ndarray:
    """Exclusive scan (n outputs) or include_initial (n + 1 outputs) of a 1-D
    array: out[0] = init, out[k] = init + inclusive[k - 1]."""
    x = np.ascontiguousarray(x)
    k = _kind(x)
    md = _mode(mode)
    y = np.empty(x.size + (1 if md == 1 else 0), dtype=x.dtype)
    rc = getattr(lib(), "cro_scan_ex_" + k)(_ptr(x), 1, _ptr(y), 1, x.size, _policy(policy),
                                            int(B), x.dtype.type(init), md)
    if rc:
        raise ValueError("bad policy, block size or mode")
    return y


def scan_ex_batched(buf: np.ndarray, batch: int, n: int, elem_stride: int, batch_stride: int,
                    policy, B: int, init, mode, out: np.ndarray, out_elem_stride: int,
                    out_batch_stride: int) -> np.ndarray:
    """Batched exclusive / include_initial scans into ``out`` (1-D, its own
    strides); returns ``out``."""
    assert buf.flags.c_contiguous and buf.ndim == 1
    assert out.flags.c_contiguous and out.ndim == 1 and out.dtype == buf.dtype
    k = _kind(buf)
    md = _mode(mode)
    _check_extent(buf, batch, n, elem_stride, batch_stride)
    _check_extent(out, batch, n + (1 if md == 1 else 0), out_elem_stride, out_batch_stride)
    rc = getattr(lib(), "cro_scan_ex_batched_" + k)(
        _ptr(buf), _ptr(out), batch, n, elem_stride, batch_stride, out_elem_stride,
        out_batch_stride, _policy(policy), int(B), buf.dtype.type(init), md)
    if rc:
        raise ValueError("bad policy, block size or mode")
    return out


def reduce_policy(x: np.ndarray, policy, B: int = 1) -> np.floating:
    """reduce<E>(x): the root of the named expression, from its own definition."""
    x = np.ascontiguousarray(x)
    k = _kind(x)
    out = np.empty(1, dtype=x.dtype)
    rc = getattr(lib(), "cro_reduce_policy_" + k)(_ptr(x), x.size, _policy(policy), int(B),
                                                  _ptr(out))
    if rc:
        raise ValueError("bad policy, block size or empty input")
    return out[0]


# ---- the non-associative integer operator (structure checks only)
def reduce_modp(x: np.ndarray, L: int, init: int) -> int:
    x = np.ascontiguousarray(x, dtype=np.uint64)
    return int(lib().cro_reduce_modp(_ptr(x), x.size, int(L), int(init)))


def scan_modp(x: np.ndarray, policy, B: int = 1) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.uint64)
    y = np.empty_like(x)
    if lib().cro_scan_modp(_ptr(x), _ptr(y), x.size, _policy(policy), int(B)):
        raise ValueError("bad policy or block size")
    return y


def scan_ex_modp(x: np.ndarray, policy, B: int, init: int, mode) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.uint64)
    md = _mode(mode)
    y = np.empty(x.size + (1 if md == 1 else 0), dtype=np.uint64)
    if lib().cro_scan_ex_modp(_ptr(x), _ptr(y), x.size, _policy(policy), int(B), int(init), md):
        raise ValueError("bad policy, block size or mode")
    return y


def reduce_policy_modp(x: np.ndarray, policy, B: int = 1) -> int:
    x = np.ascontiguousarray(x, dtype=np.uint64)
    out = np.empty(1, dtype=np.uint64)
    if lib().cro_reduce_policy_modp(_ptr(x), x.size, _policy(policy), int(B), _ptr(out)):
        raise ValueError("bad policy, block size or empty input")
    return int(out[0])


# ---- symbolic expressions (operands x0, x1, ...; init I)
def _text(fn, *args) -> str:
    need = fn(*args, None, 0)
    if need < 0:
        raise ValueError("bad arguments")
    buf = ctypes.create_string_buffer(int(need) + 1)
    fn(*args, buf, need + 1)
    return buf.value.decode()


def sym_tree(m: int) -> str:
    return _text(lib().cro_sym_tree, m)


def sym_reduce(n: int, L: int) -> str:
    return _text(lib().cro_sym_reduce, n, L)


def sym_scan(n: int, policy, B: int, i: int) -> str:
    return _text(lib().cro_sym_scan, n, _policy(policy), B, i)


def sym_scan_ex(n: int, policy, B: int, mode, k: int) -> str:
    return _text(lib().cro_sym_scan_ex, n, _policy(policy), B, _mode(mode), k)


def sym_reduce_policy(n: int, policy, B: int = 1) -> str:
    return _text(lib().cro_sym_reduce_policy, n, _policy(policy), B)


def _check_extent(buf, batch, n, es, bs):
    if batch <= 0 or n <= 0:
        return
    lo = min(0, (batch - 1) * bs) + min(0, (n - 1) * es)
    hi = max(0, (batch - 1) * bs) + max(0, (n - 1) * es)
    if lo < 0 or hi >= buf.size:
        raise ValueError("strided view exceeds the buffer")
