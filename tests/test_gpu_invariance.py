"""Invariance under the decomposition: libcr built with other compile-time
block widths, run lengths and leaf-item targets of the reduce, other tiles a block in the
scans' up pass and other fill blocks in the fused chain pass forms the same
nodes in other blocks and passes, so every call returns the default build's
bits. The inputs are sized so that each knob changes the schedule: several
reduce passes, up-pass groups of 1 to 8 tiles, 32 chain tiles shared by 5 or
32 fill blocks."""
import concurrent.futures as cf
import ctypes
import importlib.util
import os

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

VARIANTS = {
    "short_runs": ["CR_REDUCE_THREADS=128", "CR_REDUCE_MAX_RUN=16", "CR_REDUCE_LEAF_ITEMS=5000",
                   "CR_UP_LOG_TILES=0", "CR_MAX_FILL_BLOCKS=5"],
    "long_groups": ["CR_REDUCE_MAX_RUN=64", "CR_REDUCE_LEAF_ITEMS=64", "CR_UP_LOG_TILES=3",
                    "CR_MAX_FILL_BLOCKS=200"],
}


@pytest.fixture(scope="module")
def scr():
    import scan_canonical_reduce_gb300 as m
    return m


@pytest.fixture(scope="module")
def variant_libs(scr, tmp_path_factory):
    spec = importlib.util.spec_from_file_location(
        "_cr_build_variants", os.path.join(ROOT, "scan_canonical_reduce_gb300", "build.py"))
    build = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(build)
    base = tmp_path_factory.mktemp("variants")
    with cf.ThreadPoolExecutor(len(VARIANTS)) as ex:
        futs = {name: ex.submit(build.build, False, False, defs, str(base / name))
                for name, defs in VARIANTS.items()}
        paths = {name: f.result() for name, f in futs.items()}
    libs = {}
    for name, path in paths.items():
        L = ctypes.CDLL(path)
        for fn_name, (res, args) in scr.SIGNATURES.items():
            fn = getattr(L, fn_name)
            fn.restype = res
            fn.argtypes = args
        libs[name] = L
    return libs


def outputs(scr):
    """Every call's result bytes on fixed seeded inputs."""
    res = {}
    n = (1 << 21) + 37
    for dt in (np.float64, np.float32):
        x = torch.from_numpy(W.family2((1 << 22) + 37, dt)).to(DEV)
        for L in (1, 16, 128, 1000, 4096):
            res["reduce", dt, L] = scr.reduce(x, L, 0.5).cpu().numpy().tobytes()
    x4 = torch.from_numpy(W.family4(300, 5000)).to(DEV)
    res["rows"] = scr.reduce_batched(x4, 128, 0.0, dim=-1).cpu().numpy().tobytes()
    res["cols"] = scr.reduce_batched(x4, 16, 0.0, dim=0).cpu().numpy().tobytes()
    x3 = torch.from_numpy(W.family3(n)).to(DEV)
    for policy, B in (("iterated_pairwise", 1), ("pairwise", 1), ("left_fold", 1),
                      ("block_dyadic", 16), ("block_dyadic", 256), ("block_dyadic", 4096)):
        res["scan", policy, B] = scr.inclusive_scan(x3, policy, B).cpu().numpy().tobytes()
    res["excl"] = scr.exclusive_scan(x3, "pairwise", 1, 0.25).cpu().numpy().tobytes()
    res["incl_init"] = scr.scan_include_initial(x3, "block_dyadic", 16, 0.25).cpu().numpy().tobytes()
    for policy, B in (("block_dyadic", 16), ("block_dyadic", 4096), ("left_fold", 1)):
        res["reduce_policy", policy, B] = scr.reduce_policy(x3, policy, B).cpu().numpy().tobytes()
    x3f = x3.float()
    for policy, B in (("iterated_pairwise", 1), ("pairwise", 1), ("block_dyadic", 16)):
        res["scan32", policy, B] = scr.inclusive_scan(x3f, policy, B).cpu().numpy().tobytes()
    x5 = torch.from_numpy(W.family5(90, 20000)).to(DEV).view(90, 20000)
    for policy, B in (("left_fold", 1), ("block_dyadic", 16)):
        res["colscan", policy, B] = scr.inclusive_scan_batched(x5, policy, B, dim=0).cpu().numpy().tobytes()
    torch.cuda.synchronize()
    return res


@pytest.mark.parametrize("variant", sorted(VARIANTS))
def test_same_bits_under_other_decompositions(scr, variant_libs, variant):
    want = outputs(scr)
    default_lib = scr._lib
    variant_lib = variant_libs[variant]
    launched_default = default_lib.cr_launch_count()
    launched_variant = variant_lib.cr_launch_count()
    scr._lib = variant_lib
    try:
        got = outputs(scr)
    finally:
        scr._lib = default_lib
    # the calls ran in the variant's kernels, none in the default build's
    assert variant_lib.cr_launch_count() > launched_variant
    assert default_lib.cr_launch_count() == launched_default
    assert want.keys() == got.keys()
    differ = [k for k in want if want[k] != got[k]]
    assert not differ, (variant, differ)
