"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module holds only input generation: it computes no part of the canonical
reduction or scan. Both the CUDA path and the oracle consume the arrays it
returns, generated once on the host.

Random bits come from SplitMix64 used as a counter-based generator: element i
of stream ``seed`` is ``mix(seed + (i + 1) * 0x9E3779B97F4A7C15)`` with the
finaliser of Steele, Lea and Flood, "Fast splittable pseudorandom number
generators" (OOPSLA 2014). Uniform and power-of-two-scaled values are built
from those bits exactly (integer arithmetic, no libm); the normal and
lognormal families use Box-Muller through numpy's log/sqrt/cos/exp.

Workload families (the sizes are those of the benchmark configurations):
  1. canonical reduce, fp64, n = 2^20, L in {16, 128}, init 0.0, x ~ U[0,1)
  2. canonical reduce sweep, fp64/fp32, n = 2^20..2^30 (+ odd n such as
     2^28 + 37), L in {16, 128, 1024}, x = random sign * 2^e * m with e an
     integer uniform in [-20, 20] and m uniform in [1, 2) (all mantissa bits
     random), so that reassociation changes the bits
  3. canonical inclusive scan, fp64, n in {2^24, 2^28}, x ~ U[-1, 1)
  4. batched row reduce, fp32, 65,536 x 4,096 and 1,024 x 262,144, L = 128,
     x = z * 10^u_row, z ~ N(0, 1), u_row ~ U(-3, 3)
  5. batched column scan, fp64, 90 levels x 200,000 columns stored
     level-major (element (k, c) at k * 200000 + c), x = exp(z), z ~ N(0, 1)
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 20
_THREADS = max(1, min(16, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
                                else (os.cpu_count() or 1)))

SEED_BASE = 0xC0DE0000


def seed_for(cfg_id: int, sub: int = 0) -> int:
    """Fixed seed of workload family ``cfg_id`` (1..5), sub-stream ``sub``."""
    return (SEED_BASE + cfg_id + (sub << 8)) & 0xFFFFFFFFFFFFFFFF


class _Stream:
    """Chunked SplitMix64 bits with reused work buffers (fresh pages are slow)."""

    def __init__(self, chunk: int):
        self.base = np.arange(1, chunk + 1, dtype=np.uint64)
        self.t = np.empty(chunk, dtype=np.uint64)

    def bits(self, seed: int, start: int, z: np.ndarray) -> np.ndarray:
        c = z.size
        t = self.t[:c]
        with np.errstate(over="ignore"):
            np.add(self.base[:c], np.uint64(start), out=z)      # counter i + 1
            np.multiply(z, GOLDEN, out=z)
            np.add(z, np.uint64(seed & 0xFFFFFFFFFFFFFFFF), out=z)
            np.right_shift(z, np.uint64(30), out=t)
            np.bitwise_xor(z, t, out=z)
            np.multiply(z, _M1, out=z)
            np.right_shift(z, np.uint64(27), out=t)
            np.bitwise_xor(z, t, out=z)
            np.multiply(z, _M2, out=z)
            np.right_shift(z, np.uint64(31), out=t)
            np.bitwise_xor(z, t, out=z)
        return z


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Bits of elements [start, start + count) of stream ``seed`` (uint64)."""
    out = np.empty(count, dtype=np.uint64)
    st = _Stream(min(count, _CHUNK) if count else 1)
    for s in range(0, count, _CHUNK):
        c = min(_CHUNK, count - s)
        st.bits(seed, start + s, out[s:s + c])
    return out


def _fill(n: int, seed: int, dtype, fn) -> np.ndarray:
    """out[i] = fn(bits of stream ``seed`` at i, bits of stream ``seed ^ 0x5A5A``
    at i) built chunk by chunk. Large arrays are built by several threads, each
    on its own chunks (numpy's arithmetic releases the GIL); every element
    depends on its index alone, so the result does not depend on the split."""
    out = np.empty(n, dtype=dtype)
    if n == 0:
        return out
    two = fn.__code__.co_argcount == 2
    nchunks = (n + _CHUNK - 1) // _CHUNK

    def work(first: int, step: int) -> None:
        c0 = min(_CHUNK, n)
        st = _Stream(c0)
        u = np.empty(c0, dtype=np.uint64)
        v = np.empty(c0, dtype=np.uint64)
        for j in range(first, nchunks, step):
            s = j * _CHUNK
            c = min(_CHUNK, n - s)
            uu = st.bits(seed, s, u[:c])
            out[s:s + c] = fn(uu, st.bits(seed ^ 0x5A5A, s, v[:c])) if two else fn(uu)

    workers = min(_THREADS, nchunks)
    if workers <= 1:
        work(0, 1)
    else:
        with ThreadPoolExecutor(workers) as ex:
            for f in [ex.submit(work, w, workers) for w in range(workers)]:
                f.result()
    return out


def uniform01(n: int, seed: int) -> np.ndarray:
    """x ~ U[0, 1): the top 53 bits times 2^-53 (exact), float64."""
    return _fill(n, seed, np.float64,
                 lambda u: (u >> np.uint64(11)).astype(np.float64) * 2.0 ** -53)


def uniform_pm1(n: int, seed: int) -> np.ndarray:
    """x ~ U[-1, 1): top 53 bits times 2^-52, minus 1 (exact), float64."""
    return _fill(n, seed, np.float64,
                 lambda u: (u >> np.uint64(11)).astype(np.float64) * 2.0 ** -52 - 1.0)


def signed_pow2(n: int, seed: int, dtype=np.float64, emin: int = -20,
                emax: int = 20) -> np.ndarray:
    """x = sign * 2^e * m built bit by bit: sign from bit 63 of stream ``seed``,
    all mantissa bits from its low bits (m uniform in [1, 2)), and e uniform
    in [emin, emax] from stream ``seed ^ 0x5A5A`` by multiply-shift."""
    span = emax - emin + 1
    dtype = np.dtype(dtype)

    def make(u, v):
        e = (((v >> np.uint64(11)) * np.uint64(span)) >> np.uint64(53)).astype(np.int64) + emin
        sign = u >> np.uint64(63)
        if dtype == np.float64:
            bits = (sign << np.uint64(63)) | ((e + 1023).astype(np.uint64) << np.uint64(52)) \
                | (u & np.uint64((1 << 52) - 1))
            return bits.view(np.float64)
        bits = (sign << np.uint64(31)) | ((e + 127).astype(np.uint64) << np.uint64(23)) \
            | (u & np.uint64((1 << 23) - 1))
        return bits.astype(np.uint32).view(np.float32)

    return _fill(n, seed, dtype, make)


def small_integers(n: int, seed: int, bound: int, dtype=np.float64) -> np.ndarray:
    """Integer-valued x uniform in [-bound, bound] (exactly representable)."""
    span = 2 * bound + 1
    return _fill(n, seed, dtype,
                 lambda u: ((((u >> np.uint64(11)) * np.uint64(span)) >> np.uint64(53))
                                  .astype(np.int64) - bound).astype(dtype))


def standard_normal(n: int, seed: int) -> np.ndarray:
    """z ~ N(0, 1) by Box-Muller from streams ``seed`` and ``seed ^ 0x5A5A``, float64."""
    def make(u, v):
        u1 = ((u >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53  # (0, 1]
        u2 = (v >> np.uint64(11)).astype(np.float64) * 2.0 ** -53          # [0, 1)
        return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return _fill(n, seed, np.float64, make)


def row_scaled_normal(rows: int, cols: int, seed: int) -> np.ndarray:
    """Family 4: z * 10^u_row, z ~ N(0,1), u_row ~ U(-3, 3); float32, row-major."""
    z = standard_normal(rows * cols, seed).reshape(rows, cols)
    urow = (splitmix64(seed ^ 0x3C3C, 0, rows) >> np.uint64(11)).astype(np.float64) \
        * 2.0 ** -53 * 6.0 - 3.0
    return (z * (10.0 ** urow)[:, None]).astype(np.float32)


def lognormal(n: int, seed: int) -> np.ndarray:
    """Family 5: exp(z), z ~ N(0, 1); float64."""
    return np.exp(standard_normal(n, seed))


# ---------------------------------------------------------------- families
def family1(n: int = 1 << 20) -> np.ndarray:
    return uniform01(n, seed_for(1))


def family2(n: int, dtype=np.float64) -> np.ndarray:
    return signed_pow2(n, seed_for(2, 1 if np.dtype(dtype) == np.float32 else 0), dtype)


def family3(n: int) -> np.ndarray:
    return uniform_pm1(n, seed_for(3))


def family4(rows: int = 65536, cols: int = 4096, first_rows: int | None = None) -> np.ndarray:
    """The rows x cols matrix, or only its first ``first_rows`` rows (the same
    values: element i and row r's scale depend on i and r alone)."""
    k = rows if first_rows is None else min(first_rows, rows)
    return row_scaled_normal(k, cols, seed_for(4, 0 if rows == 65536 else 1))


def family5(levels: int = 90, cols: int = 200000) -> np.ndarray:
    """Level-major (levels x cols) array, flattened: element (k, c) at k*cols + c."""
    return lognormal(levels * cols, seed_for(5))
