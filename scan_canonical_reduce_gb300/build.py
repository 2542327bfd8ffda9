"""Builds libcr.so, the CUDA library of this package, for sm_103a (GB300).

Each translation unit is compiled in parallel with nvcc, then linked into a
shared library next to this file (``_build/libcr.so``). The flags keep every
floating-point add an explicit round-to-nearest operation: no FMA
contraction, no flush-to-zero, IEEE division and square root, never
--use_fast_math.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libcr.so")
SOURCES = ["cr_api.cu", "cr_calibrate.cu", "cr_chain.cu", "cr_host_batched.cu", "cr_launch.cu",
           "cr_noalloc.cu", "cr_reduce.cu", "cr_reduce_policy.cu", "cr_scan.cu"]
HEADERS = ["cr_chain.h", "cr_chain_map.h", "cr_device.cuh", "cr_launch.h", "cr_plan.h",
           "cr_scan.h"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVFLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17", "--fmad=false", "-ftz=false", "-prec-div=true",
    "-prec-sqrt=true", "-Xcompiler", "-fPIC", "-Xcompiler", "-fno-fast-math",
    "-I", os.path.join(ROOT, "include"), "-I", CSRC,
]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libcr")
    return cand


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    deps = [src] + [os.path.join(CSRC, h) for h in HEADERS] + [
        os.path.join(ROOT, "include", "cr.h"), __file__]
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, defines=(), out_dir: str | None = None) -> str:
    """Compiles the sources (those changed since their object, or all with
    force) and links the library; returns its path. `defines` ("NAME=value"
    strings) override the decomposition knobs of the sources (run lengths,
    tiles a block, fill blocks), which change no result; a build with
    defines goes to its own out_dir and is always complete."""
    out = OUT_DIR if out_dir is None else out_dir
    if defines and out_dir is None:
        raise ValueError("a build with overridden knobs needs its own out_dir")
    lib = os.path.join(out, "libcr.so")
    os.makedirs(out, exist_ok=True)
    nvcc = _nvcc()
    flags = NVFLAGS + ["-D" + d for d in defines]
    force = force or bool(defines)
    objs, jobs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(out, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, s):
            jobs.append([nvcc, *flags, "-c", s, "-o", o])
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            for r in ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs):
                if verbose or r.returncode:
                    print(r.stdout + r.stderr)
                if r.returncode:
                    raise RuntimeError("nvcc failed: " + " ".join(r.args))
    if force or jobs or not os.path.exists(lib):
        tmp = lib + ".tmp.%d" % os.getpid()
        subprocess.run([nvcc, *ARCH, "-shared", "--cudart", "static", "-o", tmp, *objs], check=True)
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
