"""Pins of the oracle's exclusive scan and include_initial form.

Definitions: the page "Vertical scan redesign: research notes", section B.2
(inclusive/exclusive duality: the exclusive scan emits the carry before each
element, its first entry is init, and include_initial is the inclusive scan
with init emitted one level upstream, n + 1 values), with init placed as in
P4016R0 on "Canonical Parallel Reduction and Scan" (combined once, as the
left operand, after the named expression). So out[0] = init and
out[k] = init + inclusive[k - 1].

Each pin is independent of the oracle's own code: hand-derived expressions
and IEEE examples live in tests/golden; here, brute force over every
parenthesisation with a non-associative operator and an independently coded
expression shape, exact integer cumulative sums, -0.0 as the exact identity,
and the page's statement that exclusive = include_initial minus its last
level.
"""
import random

import numpy as np
import pytest

import oracle
import workloads as W
from tests.test_oracle import MODP, all_trees, eval_expr, tree_split

POLICIES = [("left_fold", 1), ("iterated_pairwise", 1), ("pairwise", 1), ("block_dyadic", 2),
            ("block_dyadic", 4)]


def inclusive_shape(names, policy, B):
    """The inclusive scan's expression at the last of `names`, coded from the
    policy definitions independently of the oracle."""
    if policy == "left_fold":
        e = names[0]
        for v in names[1:]:
            e = "(%s+%s)" % (e, v)
        return e
    if policy == "iterated_pairwise":
        return tree_split(names)
    if policy == "pairwise":  # maximal aligned power-of-two runs, folded from the left
        runs, start, m = [], 0, len(names)
        for bit in reversed(range(m.bit_length())):
            if (m >> bit) & 1:
                runs.append(tree_split(names[start:start + (1 << bit)]))
                start += 1 << bit
        e = runs[0]
        for r in runs[1:]:
            e = "(%s+%s)" % (e, r)
        return e
    if policy == "block_dyadic":  # block trees chained from the left
        blocks = [names[k:k + B] for k in range(0, len(names), B)]
        e = tree_split(blocks[0])
        for blk in blocks[1:]:
            e = "(%s+%s)" % (e, tree_split(blk))
        return e
    raise AssertionError(policy)


@pytest.mark.parametrize("policy,B", POLICIES)
@pytest.mark.parametrize("mode", ["exclusive", "include_initial"])
def test_bruteforce_modp(policy, B, mode):
    rng = random.Random("%s-%d-%s" % (policy, B, mode))
    for n in range(0, 8):
        x = [rng.randrange(MODP) for _ in range(n)]
        init = rng.randrange(MODP)
        y = oracle.scan_ex_modp(np.array(x, dtype=np.uint64), policy, B, init, mode)
        m = n + 1 if mode == "include_initial" else n
        assert y.size == m
        env = {"I": init, **{"x%d" % i: v for i, v in enumerate(x)}}
        names = ["x%d" % i for i in range(n)]
        for k in range(m):
            # every operand once, in order, init first
            assert int(y[k]) in all_trees([init] + x[:k])
            assert int(y[k]) == eval_expr(oracle.sym_scan_ex(n, policy, B, mode, k), env)
            want = "I" if k == 0 else "(I+%s)" % inclusive_shape(names[:k], policy, B)
            assert int(y[k]) == eval_expr(want, env), (k, want)


@pytest.mark.parametrize("policy,B", POLICIES + [("block_dyadic", 256)])
def test_exact_integers(policy, B):
    """Integer values below 2^20 and n ~ 10^5: every sum is exact, so
    include_initial = init followed by init + the running sums."""
    n = 100003
    x = W.small_integers(n, W.seed_for(9, 41), 1 << 20)
    init = -777.0
    want = np.concatenate([[0], np.cumsum(x.astype(np.int64))]).astype(np.float64) + init
    got = oracle.scan_ex(x, policy, B, init, "include_initial")
    assert np.array_equal(got, want)
    ex = oracle.scan_ex(x, policy, B, init, "exclusive")
    assert np.array_equal(ex, want[:-1])


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("policy,B", POLICIES + [("block_dyadic", 16)])
def test_minus_zero_init_shifts_inclusive(dtype, policy, B):
    """-0.0 is the exact identity of IEEE addition (no NaN in the input):
    with it the exclusive scan is the inclusive scan moved one place right."""
    for n in (1, 2, 9, 1000, 4099):
        x = W.signed_pow2(n, W.seed_for(9, n + 5), dtype, -30, 30)
        inc = oracle.scan(x, policy, B)
        z = dtype(-0.0)
        ex = oracle.scan_ex(x, policy, B, z, "exclusive")
        ii = oracle.scan_ex(x, policy, B, z, "include_initial")
        assert ex.tobytes() == np.concatenate([[z], inc[:-1]]).astype(dtype).tobytes()
        assert ii.tobytes() == np.concatenate([[z], inc]).astype(dtype).tobytes()


@pytest.mark.parametrize("policy,B", POLICIES)
def test_exclusive_is_include_initial_minus_last_level(policy, B):
    for n in (0, 1, 5, 300):
        x = W.family3(n + 1)[:n].copy()
        a = oracle.scan_ex(x, policy, B, 0.375, "exclusive")
        b = oracle.scan_ex(x, policy, B, 0.375, "include_initial")
        assert a.tobytes() == b[:-1].tobytes()
        assert b.size == n + 1 and b[0] == 0.375


@pytest.mark.parametrize("mode", ["exclusive", "include_initial"])
def test_batched_matches_1d(mode):
    """Level-major columns (the column-scan layout) and contiguous rows, each
    written with the output's own strides."""
    levels, cols = 13, 7
    extra = 1 if mode == "include_initial" else 0
    buf = W.signed_pow2(levels * cols, W.seed_for(9, 77))
    for policy, B in POLICIES:
        out = np.full((levels + extra) * cols, np.nan)
        oracle.scan_ex_batched(buf, cols, levels, cols, 1, policy, B, 1.5, mode, out, cols, 1)
        for c in range(cols):
            want = oracle.scan_ex(buf[c::cols].copy(), policy, B, 1.5, mode)
            assert out[c::cols].tobytes() == want.tobytes()
        out2 = np.full(cols * (levels + extra), np.nan)
        oracle.scan_ex_batched(buf, cols, levels, 1, levels, policy, B, 1.5, mode, out2, 1,
                               levels + extra)
        for r in range(cols):
            want = oracle.scan_ex(buf[r * levels:(r + 1) * levels].copy(), policy, B, 1.5, mode)
            assert out2[r * (levels + extra):(r + 1) * (levels + extra)].tobytes() == \
                want.tobytes()
