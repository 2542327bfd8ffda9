"""Pins of the oracle to things other than itself.

Each check is chosen so that a plausible slip in the oracle (a dropped or
duplicated operand, a swapped operand order, a wrong tree shape, a lane index
off by one, init applied in the wrong place or twice) fails at least one:

* hand-derived expressions and hand-evaluated IEEE examples (tests/golden);
* two independent codings of the tree shape (level-wise pairing with the odd
  operand carried up, and the recursive split at the largest power of two);
* brute force over every parenthesisation of tiny inputs with a
  non-associative, non-commutative operator;
* exact integer arithmetic at large n (any tree gives the exact sum);
* special cases that reduce to one another or to numpy's sequential
  accumulate; scan/reduce consistency per policy.

Definitions: "Canonical Parallel Reduction and Scan" (github README
andyD123/canonical-reduce), P4016R0 and P4229R0 Key Design Points.
"""
import os
import random

import numpy as np
import pytest

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
MODP = (1 << 61) - 1


def modp_op(a, b):
    return (3 * a + 5 * b + 1) % MODP


# ---------------------------------------------------------------- goldens
def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


def test_golden_expressions():
    n_checked = 0
    for line in _golden_lines("expressions.txt"):
        lhs, rhs = [s.strip() for s in line.split("=", 1)]
        f = lhs.split()
        if f[0] == "tree":
            got = oracle.sym_tree(int(f[1]))
        elif f[0] == "reduce":
            got = oracle.sym_reduce(int(f[1]), int(f[2]))
        elif f[0] == "scan":
            got = oracle.sym_scan(int(f[3]), f[1], int(f[2]), int(f[4]))
        elif f[0] == "reduce_policy":
            got = oracle.sym_reduce_policy(int(f[3]), f[1], int(f[2]))
        elif f[0] == "scan_ex":
            got = oracle.sym_scan_ex(int(f[4]), f[2], int(f[3]), f[1], int(f[5]))
        else:
            raise AssertionError(line)
        assert got == rhs, line
        n_checked += 1
    assert n_checked >= 30


def _num(tok, dt):
    return dt(float(tok))


def test_golden_worked_values():
    n_checked = 0
    for line in _golden_lines("worked_values.txt"):
        head, ops, exp = [s.strip() for s in line.split("|")]
        h = head.split()
        dt = np.float64 if h[1] == "f64" else np.float32
        x = np.array([float(t) for t in ops.split()], dtype=dt)
        if h[0] == "reduce":
            got = oracle.reduce(x, int(h[2]), dt(float(h[4])))
            want = dt(float(exp))
            assert got.tobytes() == want.tobytes(), (line, got)
        elif h[0] == "reduce_policy":
            got = oracle.reduce_policy(x, h[2], int(h[3]))
            assert got.tobytes() == dt(float(exp)).tobytes(), (line, got)
        elif h[0] == "scan":
            got = oracle.scan(x, h[2], int(h[3]))
            want = np.array([float(t) for t in exp.split()], dtype=dt)
            assert got.tobytes() == want.tobytes(), (line, got)
        elif h[0] == "scan_ex":
            got = oracle.scan_ex(x, h[3], int(h[4]), dt(float(h[5])), h[2])
            want = np.array([float(t) for t in exp.split()], dtype=dt)
            assert got.tobytes() == want.tobytes(), (line, got)
        else:
            raise AssertionError(line)
        n_checked += 1
    assert n_checked >= 15


# ------------------------------------------------ independent tree codings
def tree_levelwise(items):
    """Pair neighbours level by level; an odd last item moves up unchanged."""
    items = list(items)
    while len(items) > 1:
        nxt = ["(%s+%s)" % (items[k], items[k + 1]) for k in range(0, len(items) - 1, 2)]
        if len(items) % 2:
            nxt.append(items[-1])
        items = nxt
    return items[0]


def tree_split(items):
    """Recursive: split a power-of-two run in halves, any other run after its
    largest power-of-two prefix."""
    m = len(items)
    if m == 1:
        return items[0]
    p = 1 << (m.bit_length() - 1)
    if p == m:
        p //= 2
    return "(%s+%s)" % (tree_split(items[:p]), tree_split(items[p:]))


@pytest.mark.parametrize("m", list(range(1, 130)) + [255, 256, 257, 600, 1000])
def test_tree_shape_matches_independent_codings(m):
    names = ["x%d" % i for i in range(m)]
    want = tree_split(names)
    assert tree_levelwise(names) == want
    assert oracle.sym_tree(m) == want


@pytest.mark.parametrize("n,L", [(n, L) for n in range(0, 40) for L in (1, 2, 3, 4, 5, 7, 8, 16, 50)])
def test_reduce_shape_lanes(n, L):
    """reduce = (I + tree over lane results), lane j = operands i with i mod L = j,
    lanes with no operand left out."""
    if n == 0:
        assert oracle.sym_reduce(n, L) == "I"
        return
    lanes = [["x%d" % i for i in range(j, n, L)] for j in range(min(n, L))]
    want = "(I+%s)" % tree_split([tree_split(l) for l in lanes])
    assert oracle.sym_reduce(n, L) == want


# ------------------------------------------------------------- brute force
def all_trees(vals):
    """Values of every binary parenthesisation of vals (in order) under modp_op."""
    if len(vals) == 1:
        return {vals[0]}
    out = set()
    for k in range(1, len(vals)):
        for a in all_trees(vals[:k]):
            for b in all_trees(vals[k:]):
                out.add(modp_op(a, b))
    return out


def eval_expr(expr, env):
    """Evaluate expression text like '(I+((x0+x1)+x2))' with modp_op."""
    pos = 0

    def parse():
        nonlocal pos
        if expr[pos] == "(":
            pos += 1
            a = parse()
            assert expr[pos] == "+"
            pos += 1
            b = parse()
            assert expr[pos] == ")"
            pos += 1
            return modp_op(a, b)
        k = pos
        while pos < len(expr) and expr[pos] not in "+()":
            pos += 1
        return env[expr[k:pos]]

    v = parse()
    assert pos == len(expr)
    return v


@pytest.mark.parametrize("n,L", [(n, L) for n in range(1, 8) for L in (1, 2, 3, 5, 9)])
def test_reduce_bruteforce_modp(n, L):
    rng = random.Random(1000 * n + L)
    x = [rng.randrange(MODP) for _ in range(n)]
    init = rng.randrange(MODP)
    got = oracle.reduce_modp(np.array(x, dtype=np.uint64), L, init)
    # leaves in lane order, init first: every operand used once, in that order
    order = [init] + [x[i] for j in range(min(n, L)) for i in range(j, n, L)]
    assert got in all_trees(order)
    env = {"I": init, **{"x%d" % i: v for i, v in enumerate(x)}}
    assert got == eval_expr(oracle.sym_reduce(n, L), env)
    # the shape is the one the independent coding gives, not just any tree
    lanes = [["x%d" % i for i in range(j, n, L)] for j in range(min(n, L))]
    assert got == eval_expr("(I+%s)" % tree_split([tree_split(l) for l in lanes]), env)


@pytest.mark.parametrize("policy,B", [("left_fold", 1), ("iterated_pairwise", 1),
                                      ("pairwise", 1), ("block_dyadic", 2),
                                      ("block_dyadic", 4), ("block_dyadic_alt", 2)])
def test_scan_bruteforce_modp(policy, B):
    rng = random.Random("%s-%d" % (policy, B))
    for n in range(1, 8):
        x = [rng.randrange(MODP) for _ in range(n)]
        y = oracle.scan_modp(np.array(x, dtype=np.uint64), policy, B)
        env = {"x%d" % i: v for i, v in enumerate(x)}
        for i in range(n):
            assert int(y[i]) in all_trees(x[:i + 1])
            assert int(y[i]) == eval_expr(oracle.sym_scan(n, policy, B, i), env)


def test_adversarial_doubles_bruteforce():
    """Mixed 2^+-50 magnitudes: the oracle's float value is the float value of
    its own expression (evaluated here independently) and in general differs
    from other parenthesisations."""
    rng = random.Random(7)
    for n in range(2, 8):
        for L in (1, 2, 3):
            x = [rng.choice([-1, 1]) * 2.0 ** rng.randint(-50, 50) * (1 + rng.random())
                 for _ in range(n)]
            init = 2.0 ** rng.randint(-50, 50)
            got = oracle.reduce(np.array(x), L, init)
            lanes = [[x[i] for i in range(j, n, L)] for j in range(min(n, L))]

            def tree_val(v):
                if len(v) == 1:
                    return v[0]
                p = 1 << (len(v).bit_length() - 1)
                if p == len(v):
                    p //= 2
                return tree_val(v[:p]) + tree_val(v[p:])

            want = init + tree_val([tree_val(l) for l in lanes])
            assert got.tobytes() == np.float64(want).tobytes()


# ----------------------------------------------------------- exact integers
@pytest.mark.parametrize("n", [1, 2, 3, 17, 1000, 4097, (1 << 16) + 37, 1 << 20])
@pytest.mark.parametrize("L", [1, 3, 16, 128, 1024])
def test_reduce_exact_integers_f64(n, L):
    x = W.small_integers(n, W.seed_for(9, n % 251), 1 << 20)
    init = 12345.0
    want = float(int(x.astype(np.int64).sum()) + 12345)
    assert oracle.reduce(x, L, init) == want


@pytest.mark.parametrize("n", [1, 5, 1000, (1 << 20) - 3])
@pytest.mark.parametrize("L", [1, 16, 128])
def test_reduce_exact_integers_f32(n, L):
    x = W.small_integers(n, W.seed_for(9, 7 + n % 13), 8, np.float32)
    want = np.float32(int(x.astype(np.int64).sum()) - 3)
    assert oracle.reduce(x, L, np.float32(-3.0)) == want


@pytest.mark.slow
def test_reduce_exact_integers_large():
    n = (1 << 26) + 37
    x = W.small_integers(n, W.seed_for(9, 99), 1 << 20)
    want = float(int(x.astype(np.int64).sum()))
    for L in (16, 1024):
        assert oracle.reduce(x, L, 0.0) == want


@pytest.mark.parametrize("policy,B", [("left_fold", 1), ("iterated_pairwise", 1),
                                      ("pairwise", 1), ("block_dyadic", 16),
                                      ("block_dyadic", 256), ("block_dyadic_alt", 16)])
def test_scan_exact_integers(policy, B):
    n = 100003
    x = W.small_integers(n, W.seed_for(9, 3), 1 << 20)
    want = np.cumsum(x.astype(np.int64)).astype(np.float64)
    assert np.array_equal(oracle.scan(x, policy, B), want)


# ------------------------------------------------------------ special cases
def _adversarial(n, seed, dtype=np.float64):
    return W.signed_pow2(n, seed, dtype, -30, 30)


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_lane_count_one_equals_lane_count_at_least_n(dtype):
    for n in (1, 2, 7, 64, 100, 1000):
        x = _adversarial(n, W.seed_for(9, n), dtype)
        init = dtype(0.25)
        a = oracle.reduce(x, 1, init)
        for L in (n, n + 1, 10 * n):
            assert oracle.reduce(x, L, init).tobytes() == a.tobytes()


def test_empty_and_single():
    x = np.array([], dtype=np.float64)
    assert oracle.reduce(x, 16, 3.5) == 3.5
    for L in (1, 2, 100):
        v = oracle.reduce(np.array([1e-300]), L, 1.0)
        assert v == 1.0 + 1e-300


def test_minus_zero_init_is_identity():
    for n in (1, 3, 1000, 4099):
        x = _adversarial(n, W.seed_for(9, n + 1))
        a = oracle.reduce(x, 1, -0.0)
        b = oracle.reduce_policy(x, "iterated_pairwise")
        assert a.tobytes() == b.tobytes()


def test_left_fold_is_numpy_accumulate():
    """numpy's add.accumulate is a strictly sequential left-to-right fold."""
    for dtype in (np.float64, np.float32):
        x = _adversarial(5000, W.seed_for(9, 5), dtype)
        assert np.array_equal(oracle.scan(x, "left_fold"), np.add.accumulate(x))
        assert np.array_equal(oracle.scan(x, "block_dyadic", 1), np.add.accumulate(x))


def test_block_dyadic_limits():
    for n in (1, 5, 16, 17, 100, 1000):
        x = _adversarial(n, W.seed_for(9, 2 * n))
        ip = oracle.scan(x, "iterated_pairwise")
        for B in (n, 2 * n, 1 << 20):
            assert np.array_equal(oracle.scan(x, "block_dyadic", B), ip)
        assert np.array_equal(oracle.scan(x, "block_dyadic", 1), oracle.scan(x, "left_fold"))
        # reading B sits the other way round
        assert np.array_equal(oracle.scan(x, "block_dyadic_alt", 1), ip)
        assert np.array_equal(oracle.scan(x, "block_dyadic_alt", max(n, 1)),
                              oracle.scan(x, "left_fold"))


def test_pairwise_back_vs_iterated():
    differs = 0
    for n in range(1, 300):
        x = _adversarial(n, W.seed_for(9, 3 * n))
        a = oracle.scan(x, "pairwise")[-1]
        b = oracle.scan(x, "iterated_pairwise")[-1]
        if bin(n).count("1") <= 2:
            assert a.tobytes() == b.tobytes(), n
        elif a.tobytes() != b.tobytes():
            differs += 1
    assert differs > 50  # the two policies are really different expressions


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_batched_rows_and_columns_match_1d(dtype):
    rows, cols = 7, 301
    buf = _adversarial(rows * cols, W.seed_for(9, 77), dtype)
    m = buf.reshape(rows, cols)
    # rows: batch_stride = cols, elem_stride = 1
    out = oracle.reduce_batched(buf, rows, cols, 1, cols, 16, 0.5)
    for r in range(rows):
        assert out[r].tobytes() == oracle.reduce(m[r].copy(), 16, 0.5).tobytes()
    # columns: level-major, elem_stride = cols, batch_stride = 1
    outc = oracle.reduce_batched(buf, cols, rows, cols, 1, 3, 0.5)
    for c in range(cols):
        assert outc[c].tobytes() == oracle.reduce(m[:, c].copy(), 3, 0.5).tobytes()
    for policy, B in (("left_fold", 1), ("block_dyadic", 4), ("iterated_pairwise", 1)):
        y = oracle.scan_batched(buf, cols, rows, cols, 1, policy, B).reshape(rows, cols)
        for c in range(0, cols, 37):
            assert np.array_equal(y[:, c], oracle.scan(m[:, c].copy(), policy, B))


@pytest.mark.parametrize("policy,B", [("left_fold", 1), ("iterated_pairwise", 1),
                                      ("block_dyadic", 1), ("block_dyadic", 2),
                                      ("block_dyadic", 4), ("block_dyadic", 16),
                                      ("block_dyadic_alt", 4)])
@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_scan_reduce_consistency(policy, B, dtype):
    """inclusive_scan<E>(xs)[i] == reduce<E>(xs[0..i+1)) for the policies that
    claim it; reduce<E> is evaluated from its own definition."""
    n = 300
    x = _adversarial(n, W.seed_for(9, 11), dtype)
    y = oracle.scan(x, policy, B)
    for i in range(n):
        r = oracle.reduce_policy(x[:i + 1].copy(), policy, B)
        assert y[i].tobytes() == r.tobytes(), i


def test_pairwise_is_not_consistent_in_general():
    x = _adversarial(300, W.seed_for(9, 12))
    y = oracle.scan(x, "pairwise")
    bad = sum(y[i].tobytes() != oracle.reduce_policy(x[:i + 1].copy(), "pairwise").tobytes()
              for i in range(300))
    assert bad > 0


def test_lane_count_changes_result_few_ulps():
    """Family-1 data (n = 2^20, U[0,1)): L = 16 and L = 128 both evaluate valid
    trees, so they agree to within a few ulps but need not be equal."""
    x = W.family1(1 << 20)
    a = oracle.reduce(x, 16, 0.0)
    b = oracle.reduce(x, 128, 0.0)
    ulps = abs(int(a.view(np.int64)) - int(b.view(np.int64)))
    assert ulps < 200
    assert abs(a - x.sum()) < 1e-6 * x.sum()


def test_splitmix64_published_first_output():
    """SplitMix64 with state 0: first output 0xe220a8397b1dcdaf (the value the
    published reference implementation prints)."""
    assert int(W.splitmix64(0, 0, 1)[0]) == 0xE220A8397B1DCDAF
