"""The oracle's pins catch plausible mistakes in it.

Each mutant is a copy of oracle/cro.cpp with one slip planted (CPU only,
built into a temporary directory; the oracle's own source and library are
untouched): an operand order swapped in a tree merge, the final fold or the
carry; init applied on the wrong side; the lanes rotated; the merge rule
loosened; pairwise folded like iterated_pairwise; the reduce<block_dyadic>
chain reversed; the exclusive form folding init on the wrong side; the adds
evaluated in a wider type. Every mutant must fail at least one pin of
tests/test_oracle.py and tests/test_oracle_scan_ex.py, and the unmutated copy,
built the same way, must pass them all.
"""
import concurrent.futures as cf
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
from oracle import build as obuild
from tests import test_oracle as T
from tests import test_oracle_scan_ex as TX

# (name, text in cro.cpp, its replacement)
MUTANTS = [
    ("merge_operands_swapped", "val.push_back(op(lower, upper));",
     "val.push_back(op(upper, lower));"),
    ("final_fold_operands_swapped", "k >= 0; --k) acc = op(val[k], acc);",
     "k >= 0; --k) acc = op(acc, val[k]);"),
    ("init_on_the_right", "return op(init, across.collapse_from_top(op));",
     "return op(across.collapse_from_top(op), init);"),
    ("lanes_rotated", "for (int64_t i = j; i < n; i += L) lane.push(",
     "for (int64_t i = (j + 1) % m; i < n; i += L) lane.push("),
    ("merge_rule_loosened", "size[size.size() - 1] == size[size.size() - 2]",
     "size[size.size() - 1] <= size[size.size() - 2]"),
    ("pairwise_folded_from_the_top", "    y[i * ys] = st.fold_from_bottom(op);",
     "    y[i * ys] = st.collapse_from_top(op);"),
    ("block_carry_on_the_right", "y[i * ys] = (k == 0) ? p : op(carry, p);",
     "y[i * ys] = (k == 0) ? p : op(p, carry);"),
    ("block_chain_reversed", "carry = (k == 0) ? t : op(carry, t);",
     "carry = (k == 0) ? t : op(t, carry);"),
    ("reduce_policy_chain_reversed", "c = op(c, tree(x + k0 * xs, len, xs, op));",
     "c = op(tree(x + k0 * xs, len, xs, op), c);"),
    ("exclusive_init_on_the_right", "out[k * os] = op(init, y[(size_t)(k - 1)]);",
     "out[k * os] = op(y[(size_t)(k - 1)], init);"),
    ("adds_widened", "double operator()(double a, double b) const { return a + b; }",
     "double operator()(double a, double b) const { return (long double)a + b; }"),
]


def _checks():
    """The pins, as (name, callable) pairs; each raises when it fails."""
    f64 = np.float64
    return [
        ("golden_expressions", T.test_golden_expressions),
        ("golden_worked_values", T.test_golden_worked_values),
        ("tree_shapes", lambda: [T.test_tree_shape_matches_independent_codings(m)
                                 for m in range(1, 40)]),
        ("reduce_shapes", lambda: [T.test_reduce_shape_lanes(n, L) for n in range(0, 20)
                                   for L in (1, 2, 3, 5, 16)]),
        ("reduce_bruteforce", lambda: [T.test_reduce_bruteforce_modp(n, L)
                                       for n in range(1, 8) for L in (1, 2, 3)]),
        ("scan_bruteforce", lambda: [T.test_scan_bruteforce_modp(p, B) for p, B in
                                     (("left_fold", 1), ("iterated_pairwise", 1),
                                      ("pairwise", 1), ("block_dyadic", 2))]),
        ("adversarial_doubles", T.test_adversarial_doubles_bruteforce),
        ("exact_integers", lambda: T.test_reduce_exact_integers_f64(1000, 16)),
        ("left_fold_numpy", T.test_left_fold_is_numpy_accumulate),
        ("block_dyadic_limits", T.test_block_dyadic_limits),
        ("pairwise_vs_iterated", T.test_pairwise_back_vs_iterated),
        ("consistency", lambda: [T.test_scan_reduce_consistency(p, B, f64) for p, B in
                                 (("iterated_pairwise", 1), ("block_dyadic", 4))]),
        ("scan_ex_bruteforce", lambda: [TX.test_bruteforce_modp(p, B, mode)
                                        for p, B in (("left_fold", 1), ("block_dyadic", 2))
                                        for mode in ("exclusive", "include_initial")]),
    ]


def _build(tmp, name, patch):
    with open(obuild.SRC) as f:
        src = f.read()
    if patch is not None:
        old, new = patch
        assert src.count(old) == 1, "mutation anchor not found once: %s" % name
        src = src.replace(old, new)
    cpp = os.path.join(tmp, name + ".cpp")
    so = os.path.join(tmp, name + ".so")
    with open(cpp, "w") as f:
        f.write(src)
    subprocess.run(["g++", *obuild.CXXFLAGS, cpp, "-o", so], check=True)
    return so


def _failing_checks(so):
    """Names of the pins that fail with the oracle library at `so`."""
    saved = oracle.lib()
    lib = ctypes.CDLL(so)
    oracle._declare(lib)
    oracle._lib = lib
    failed = []
    try:
        for name, fn in _checks():
            try:
                fn()
            except Exception:  # an assertion, or a shape or type error: caught either way
                failed.append(name)
    finally:
        oracle._lib = saved
    return failed


@pytest.fixture(scope="module")
def builds(tmp_path_factory):
    tmp = str(tmp_path_factory.mktemp("cro_mutants"))
    jobs = [("unmutated", None)] + [(n, (a, b)) for n, a, b in MUTANTS]
    with cf.ThreadPoolExecutor(max_workers=min(8, len(jobs))) as ex:
        paths = list(ex.map(lambda j: _build(tmp, j[0], j[1]), jobs))
    return dict(zip([j[0] for j in jobs], paths))


def test_unmutated_copy_passes_every_pin(builds):
    assert _failing_checks(builds["unmutated"]) == []


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_mutant_is_caught(builds, name):
    if name == "adds_widened" and np.finfo(np.longdouble).nmant != 63:
        # only x87's 64-bit significand rounds twice often enough to show
        pytest.skip("long double is not the x87 extended format here")
    failed = _failing_checks(builds[name])
    assert failed, "no pin caught the planted mistake %s" % name
