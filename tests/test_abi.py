"""The C ABI library: builds, loads, exports every function include/cr.h
declares, and rejects bad arguments on the host (no GPU needed: argument
checks and workspace sizing run before any CUDA call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cr.h")


@pytest.fixture(scope="module")
def scr():
    import __graft_entry__
    __graft_entry__.build()
    import scan_canonical_reduce_gb300 as m
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cr_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(scr):
    names = declared_functions()
    assert len(names) >= 11
    lib = ctypes.CDLL(scr.LIB_PATH)
    for name in names:
        assert hasattr(lib, name), name
    # and the binding declares a signature for each
    assert sorted(scr.SIGNATURES) == names


def test_status_strings_and_version(scr):
    L = scr.lib()
    for code in range(6):
        assert L.cr_status_string(code)
    assert L.cr_status_string(99) == b"unknown status"
    assert L.cr_version() >= 100


def test_workspace_sizes(scr):
    L = scr.lib()
    for n in (0, 1, 17, 1 << 20, (1 << 28) + 37):
        for lanes in (1, 16, 128, 1024):
            for dt in (1, 2):
                nb = L.cr_reduce_workspace_bytes(n, lanes, dt)
                assert nb >= 256 and nb % 256 == 0
    assert L.cr_reduce_workspace_bytes(-1, 16, 2) == 0
    assert L.cr_reduce_workspace_bytes(10, 0, 2) == 0
    assert L.cr_reduce_workspace_bytes(10, 16, 3) == 0
    assert L.cr_reduce_batched_workspace_bytes(65536, 4096, 128, 1) >= 256
    assert L.cr_scan_workspace_bytes(100, 3, 3, 2) == 0   # B not a power of two
    assert L.cr_scan_workspace_bytes(100, 9, 1, 2) == 0   # unknown policy
    assert L.cr_scan_workspace_bytes(100, 3, 16, 2) >= 256


def test_host_side_argument_errors(scr):
    L = scr.lib()
    one = ctypes.c_double(0.0)
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: checks fail first
    # n < 0, L < 1, bad dtype, missing init/out
    assert L.cr_reduce(fake, -1, 16, ctypes.byref(one), 2, fake, fake, 1 << 20, None) == 1
    assert L.cr_reduce(fake, 10, 0, ctypes.byref(one), 2, fake, fake, 1 << 20, None) == 1
    assert L.cr_reduce(fake, 10, 16, ctypes.byref(one), 7, fake, fake, 1 << 20, None) == 1
    assert L.cr_reduce(fake, 10, 16, None, 2, fake, fake, 1 << 20, None) == 1
    assert L.cr_reduce(fake, 10, 16, ctypes.byref(one), 2, None, fake, 1 << 20, None) == 1
    # misaligned element pointer
    assert L.cr_reduce(ctypes.c_void_p(0x10004), 10, 16, ctypes.byref(one), 2, fake, fake,
                       1 << 20, None) == 1
    # workspace missing / misaligned / too small
    assert L.cr_reduce(fake, 10, 16, ctypes.byref(one), 2, fake, None, 1 << 20, None) == 3
    assert L.cr_reduce(fake, 10, 16, ctypes.byref(one), 2, fake, ctypes.c_void_p(0x10008),
                       1 << 20, None) == 3
    assert L.cr_reduce(fake, 1 << 20, 16, ctypes.byref(one), 2, fake, fake, 256, None) == 3
    # scans: bad policy, B not a power of two, partial overlap
    assert L.cr_inclusive_scan(fake, fake, 10, 9, 1, 2, fake, 1 << 20, None) == 1
    assert L.cr_inclusive_scan(fake, fake, 10, 3, 6, 2, fake, 1 << 20, None) == 1
    assert L.cr_inclusive_scan(fake, ctypes.c_void_p(0x10008), 10, 2, 1, 2, fake, 1 << 20,
                               None) == 1
    assert L.cr_reduce_batched(fake, fake, -1, 10, 1, 10, 16, ctypes.byref(one), 2, fake,
                               1 << 20, None) == 1


def test_scan_ex_host_side_argument_errors(scr):
    """Exclusive / include_initial: bad mode, missing init, an output range
    that partially overlaps the input (the include_initial output is one
    element longer), in-place batched calls with other output strides."""
    L = scr.lib()
    one = ctypes.c_double(0.0)
    fake = ctypes.c_void_p(0x10000)
    assert L.cr_scan_ex_workspace_bytes(100, 2, 1, 0, 2) == 0   # mode 0 is not a mode here
    assert L.cr_scan_ex_workspace_bytes(100, 2, 1, 3, 2) == 0
    assert L.cr_scan_ex_workspace_bytes(100, 3, 6, 1, 2) == 0   # B not a power of two
    for mode in (1, 2):
        assert L.cr_scan_ex_workspace_bytes(100, 3, 16, mode, 2) >= 256
        assert L.cr_scan_ex_workspace_bytes(0, 0, 1, mode, 1) >= 256
        assert L.cr_scan_ex_batched_workspace_bytes(7, 90, 3, 16, mode, 2) >= 256
    assert L.cr_scan_ex(fake, fake, 10, 2, 1, 5, ctypes.byref(one), 2, fake, 1 << 20,
                        None) == 1
    assert L.cr_scan_ex(fake, fake, 10, 2, 1, 1, None, 2, fake, 1 << 20, None) == 1
    # out starts one element before x: overlaps, not in place
    assert L.cr_scan_ex(ctypes.c_void_p(0x10008), fake, 10, 2, 1, 2, ctypes.byref(one), 2,
                        fake, 1 << 20, None) == 1
    # include_initial writes n + 1 elements: out ending inside x overlaps
    assert L.cr_scan_ex(fake, ctypes.c_void_p(0x10000 - 8 * 5), 10, 2, 1, 2, ctypes.byref(one),
                        2, fake, 1 << 20, None) == 1
    # in place batched with different output strides
    assert L.cr_scan_ex_batched(fake, fake, 4, 10, 4, 1, 5, 1, 0, 1, 2, ctypes.byref(one), 2,
                                fake, 1 << 20, None) == 1
    # workspace too small
    assert L.cr_scan_ex(fake, ctypes.c_void_p(0x10000000), 1 << 20, 3, 16, 1, ctypes.byref(one),
                        2, fake, 256, None) == 3


def test_binding_fails_loudly_without_library(tmp_path, scr):
    """The binding has no CPU fallback: with the library absent it raises."""
    import importlib.util
    import shutil
    pkg = tmp_path / "scan_canonical_reduce_gb300"
    shutil.copytree(os.path.dirname(scr.__file__), pkg,
                    ignore=shutil.ignore_patterns("_build", "__pycache__"))
    spec = importlib.util.spec_from_file_location("scr_nolib", pkg / "__init__.py")
    mod = importlib.util.module_from_spec(spec)
    with pytest.raises(ImportError):
        spec.loader.exec_module(mod)


def test_reduce_policy_host_side_argument_errors(scr):
    """reduce<E> of an empty input has no root; bad policy or block size."""
    L = scr.lib()
    fake = ctypes.c_void_p(0x10000)
    assert L.cr_reduce_policy_workspace_bytes(0, 2, 1, 2) == 0
    assert L.cr_reduce_policy_workspace_bytes(10, 3, 6, 2) == 0
    for p, B in ((0, 1), (1, 1), (2, 1), (3, 16), (3, 1 << 20)):
        assert L.cr_reduce_policy_workspace_bytes(1 << 20, p, B, 2) >= 256
    assert L.cr_reduce_policy(fake, 0, 2, 1, 2, fake, fake, 1 << 20, None) == 1
    assert L.cr_reduce_policy(fake, 10, 9, 1, 2, fake, fake, 1 << 20, None) == 1
    assert L.cr_reduce_policy(fake, 10, 2, 1, 2, None, fake, 1 << 20, None) == 1
    assert L.cr_reduce_policy(fake, 1 << 20, 3, 16, 2, fake, fake, 256, None) == 3


def test_stride_errors(scr):
    """Negative strides, and zero output strides that would send two outputs
    to one element, are rejected on the host (nothing is enqueued)."""
    L = scr.lib()
    one = ctypes.c_double(0.0)
    fake = ctypes.c_void_p(0x10000)
    ws = ctypes.c_void_p(0x100000)
    for es, bs in ((-1, 10), (10, -1)):
        assert L.cr_reduce_batched(fake, ws, 4, 10, es, bs, 16, ctypes.byref(one), 2, fake,
                                   1 << 20, None) == 1
        assert L.cr_inclusive_scan_batched(fake, ws, 4, 10, es, bs, 0, 1, 2, fake, 1 << 20,
                                           None) == 1
    # zero strides: a read-only repeat is fine for a reduce (fails later, on the
    # fake workspace being too small, not on the strides)
    assert L.cr_reduce_batched(fake, ws, 4, 10, 0, 0, 16, ctypes.byref(one), 2, fake, 8,
                               None) == 3
    # scans: two outputs of one sequence, or two sequences, on one element
    assert L.cr_inclusive_scan_batched(fake, ws, 4, 10, 0, 1, 0, 1, 2, fake, 1 << 20, None) == 1
    assert L.cr_inclusive_scan_batched(fake, ws, 4, 10, 4, 0, 0, 1, 2, fake, 1 << 20, None) == 1
    assert L.cr_scan_ex_batched(fake, ws, 4, 10, 4, 1, 0, 1, 0, 1, 2, ctypes.byref(one), 2,
                                fake, 1 << 20, None) == 1
    assert L.cr_scan_ex_batched(fake, ws, 4, 10, 4, 1, 4, -1, 0, 1, 2, ctypes.byref(one), 2,
                                fake, 1 << 20, None) == 1
    # one sequence of one output may use a zero output stride (workspace check next)
    assert L.cr_scan_ex_batched(fake, ws, 1, 0, 1, 1, 0, 0, 0, 1, 2, ctypes.byref(one), 2,
                                fake, 8, None) == 3


def test_batched_overlap_errors(scr):
    """Batched layouts whose outputs would meet: equal output strides with two
    or more sequences of two or more outputs, and an output that partially
    overlaps a densely laid out input (rows or level-major columns). A zero
    output stride in an empty batch, and interleaved (non-dense) layouts,
    are not rejected for that reason (the fake workspace fails next)."""
    L = scr.lib()
    one = ctypes.c_double(0.0)
    x = 0x10000
    ws = ctypes.c_void_p(0x100000)

    def p(addr):
        return ctypes.c_void_p(addr)

    # out == x with element and sequence strides both 1: (b + 1, k) is (b, k + 1)
    assert L.cr_inclusive_scan_batched(p(x), p(x), 2, 10, 1, 1, 0, 1, 2, ws, 1 << 20,
                                       None) == 1
    assert L.cr_scan_ex_batched(p(x), p(0x90000), 2, 10, 1, 10, 1, 1, 0, 1, 2,
                                ctypes.byref(one), 2, ws, 1 << 20, None) == 1
    # an empty batch may carry any output strides
    assert L.cr_scan_ex_batched(p(x), p(0x90000), 0, 10, 1, 10, 0, 0, 0, 1, 2,
                                ctypes.byref(one), 2, ws, 8, None) == 3
    # rows of 10: out one element after x overlaps every row but the first
    assert L.cr_inclusive_scan_batched(p(x), p(x + 8), 4, 10, 1, 10, 0, 1, 2, ws, 1 << 20,
                                       None) == 1
    # level-major columns: out one level below x
    assert L.cr_inclusive_scan_batched(p(x), p(x + 8 * 4), 4, 10, 4, 1, 0, 1, 2, ws, 1 << 20,
                                       None) == 1
    # include_initial output rows of 11 ending inside the input rows
    assert L.cr_scan_ex_batched(p(x + 8 * 40 - 8), p(x), 4, 10, 1, 10, 1, 11, 0, 1, 2,
                                ctypes.byref(one), 2, ws, 1 << 20, None) == 1
    # a batched reduce writing its results into its own rows
    assert L.cr_reduce_batched(p(x), p(x + 16), 4, 10, 1, 10, 16, ctypes.byref(one), 2, ws,
                               1 << 20, None) == 1
    # interleaved: x on even elements, out on odd ones (not dense): allowed
    assert L.cr_inclusive_scan_batched(p(x), p(x + 8), 4, 10, 2, 20, 0, 1, 2, ws, 8,
                                       None) == 3
    assert L.cr_reduce_batched(p(x), p(x + 8 * 40), 4, 10, 1, 10, 16, ctypes.byref(one), 2,
                               ws, 8, None) == 3


def test_batched_host_argument_errors(scr):
    """The host-buffer batched calls check their arguments, the device
    buffer and the host layout before any CUDA call."""
    L = scr.lib()
    one = ctypes.c_double(0.0)
    x, o = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x90000)
    ws = ctypes.c_void_p(0x100000)
    need = L.cr_reduce_batched_host_workspace_bytes(10, 10, 16, 2)
    assert need >= 256 and need % 256 == 0
    assert L.cr_reduce_batched_host_workspace_bytes(10, 10, 0, 2) == 0
    assert L.cr_inclusive_scan_batched_host_workspace_bytes(10, 10, 3, 3, 2) == 0
    # negative strides, bad dtype
    assert L.cr_reduce_batched_host(x, o, 10, 10, -1, 10, 16, ctypes.byref(one), 2, ws,
                                    need, None) == 1
    assert L.cr_reduce_batched_host(x, o, 10, 10, 1, 10, 16, ctypes.byref(one), 7, ws,
                                    need, None) == 1
    # the device buffer too small
    assert L.cr_reduce_batched_host(x, o, 10, 10, 1, 10, 16, ctypes.byref(one), 2, ws,
                                    need - 256, None) == 3
    # neither rows nor level-major columns
    assert L.cr_reduce_batched_host(x, o, 10, 10, 2, 3, 16, ctypes.byref(one), 2, ws,
                                    need, None) == 2
    sneed = L.cr_inclusive_scan_batched_host_workspace_bytes(10, 10, 0, 1, 2)
    assert L.cr_inclusive_scan_batched_host(x, o, 10, 10, 2, 30, 0, 1, 2, ws, sneed,
                                            None) == 2
    # a zero stride sends two outputs to one element
    assert L.cr_inclusive_scan_batched_host(x, o, 10, 10, 0, 1, 0, 1, 2, ws, sneed,
                                            None) == 2
    # empty batches need no GPU
    assert L.cr_reduce_batched_host(x, o, 0, 10, 1, 10, 16, ctypes.byref(one), 2, ws, 256,
                                    None) == 0
    assert L.cr_inclusive_scan_batched_host(x, o, 10, 0, 1, 0, 0, 1, 2, ws, 256, None) == 0


def test_pairwise_binary64_workspace_keeps_quads(scr):
    """The binary64 pairwise scan's up pass keeps 16 bytes a thread (a quad
    and the thread's root, 8 elements a thread): its workspace exceeds the
    binary32 one by at least 2 bytes an element; iterated_pairwise keeps
    none."""
    L = scr.lib()
    n = 1 << 24
    pw64 = L.cr_scan_workspace_bytes(n, 1, 1, 2)
    pw32 = L.cr_scan_workspace_bytes(n, 1, 1, 1)
    ip64 = L.cr_scan_workspace_bytes(n, 2, 1, 2)
    assert pw64 >= pw32 + 2 * n
    assert ip64 < 2 * n


def test_profile_select_takes_any_id(scr):
    """Selecting a kernel, an id out of range or none records nothing by
    itself and needs no device."""
    L = scr.lib()
    for kid in (0, 5, -1, 10 ** 6):
        L.cr_profile_select(kid)
    L.cr_profile_select(-1)
    assert L.cr_profile_collect(None, None, 0) == 0
    with pytest.raises(ValueError):
        scr.profile_select("no_such_kernel")


def test_build_overrides_need_their_own_directory():
    """A build with overridden decomposition knobs never replaces the
    package's own library."""
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_cr_build_check", os.path.join(ROOT, "scan_canonical_reduce_gb300", "build.py"))
    build = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(build)
    with pytest.raises(ValueError):
        build.build(defines=["CR_REDUCE_MAX_RUN=16"])
