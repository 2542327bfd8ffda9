"""bench.py's host-side pieces (CPU, no GPU): the per-row rates (algorithmic
GB/s against the measured and the nominal HBM figures, elements/s, adds/s
against the add rate of the row's type), the element count of every row of
the step, and the oracle sample's input rows."""
import pytest

import bench


def test_rate_stats_by_hand():
    # 8 GB read in 2 ms = 4000 GB/s; 2^28 elements; 2^28 adds
    r = ("reduce_f64_L16", "reduce", {"L": 16}, 8 * 10**9, 1 << 28, "f64")
    s = bench.rate_stats(r, 2.0, 8000.0, 0.5e12, 40e12)
    assert s["gb_s"] == 4000.0
    assert s["hbm_frac"] == 0.5
    assert s["hbm_frac_nominal"] == pytest.approx(4000.0 / 7900.0, abs=1e-4)
    assert s["elems_per_s"] == pytest.approx(bench.N / 2e-3)
    assert s["adds_per_s"] == pytest.approx((1 << 28) / 2e-3)
    assert s["alu_frac"] == pytest.approx((1 << 28) / 2e-3 / 0.5e12, abs=1e-4)


def test_rate_stats_f32_uses_the_f32_add_rate():
    r = ("reduce_rows_f32_L128", "rows", {"L": 128}, 10**9, 10**9, "f32")
    s = bench.rate_stats(r, 1.0, None, 0.5e12, 40e12)
    assert s["hbm_frac"] is None
    assert s["alu_frac"] == pytest.approx(1e12 / 40e12, abs=1e-4)
    assert s["elems_per_s"] == pytest.approx(bench.ROWS_R * bench.ROWS_C / 1e-3)


def test_every_row_has_its_element_count():
    """Element counts and algorithmic bytes per element of every row: the
    step's rows and the extras (the reduce sweep over n, the binary32 scans,
    the U[0, 1) reduce at 2^20 and the 1,024 x 262,144 row reduce)."""
    rows_b = bench.ROWS_B[0] * bench.ROWS_B[1]
    for r in bench.rows_spec() + bench.extra_rows():
        kind, p = r[1], r[2]
        want = {"reduce": p.get("n", bench.N), "reduce_u01": 1 << 20, "scan": bench.N,
                "scan_ex": bench.N, "rows": bench.ROWS_R * bench.ROWS_C, "rows_b": rows_b,
                "cols": bench.COLS_LEVELS * bench.COLS_N}[kind]
        assert bench.row_elems(r) == want, r[0]
        es = 4 if r[5] == "f32" else 8
        per = r[3] / bench.row_elems(r)
        if kind in ("reduce", "reduce_u01"):
            assert per == es, (r[0], per)
        elif kind in ("scan", "cols"):
            assert per == 2 * es, (r[0], per)
        elif kind == "scan_ex":
            assert 16 <= per < 16.01, (r[0], per)
        else:  # row reduces: the input and one output a row
            assert 4 <= per < 4.01, (r[0], per)
    names = [r[0] for r in bench.extra_rows()]
    assert len(names) == len(set(names))
    for dt in ("f64", "f32"):
        for n in bench.SWEEP_N:
            for L in (16, 128, 1024):
                assert "sweep_reduce_%s_n%s_L%d" % (dt, bench.size_tag(n), L) in names
    assert bench.size_tag((1 << 28) + 37) == "2e28p37"


def test_family4_first_rows_is_the_matrix_prefix():
    """The reference arm's row sample generates only the rows it times: the
    same values as the first rows of the full matrix (per-element counters,
    per-row scales), for the bench shape's seed and another."""
    import numpy as np
    import workloads as W
    for rows in (65536, 300):
        full = W.family4(rows, 4)
        part = W.family4(rows, 4, first_rows=37)
        assert part.shape == (37, 4)
        assert np.array_equal(part.view(np.uint32), full[:37].view(np.uint32))


def test_ncu_traffic_needs_the_captured_sources(monkeypatch):
    """The recorded ncu traffic of a kernel is reported only while its source
    files hash as they did at the capture; any change drops it (None)."""
    rec = bench.NCU_TRAFFIC["scan_onepass_kernel"]
    monkeypatch.setattr(bench, "source_digest", lambda name: rec["sources"].get(name))
    assert bench.ncu_traffic("scan_onepass_kernel") == rec["bytes"]
    monkeypatch.setattr(bench, "source_digest", lambda name: "0" * 16)
    assert bench.ncu_traffic("scan_onepass_kernel") is None
    assert bench.ncu_traffic("no_such_kernel") is None


def test_clock_samples_inside_the_timed_window():
    """Only samples stamped inside the timed region count (with their throttle
    reasons); with none inside, all samples are reported and the count says
    so; unparsable lines are skipped."""
    import datetime

    def line(t, sm, cap):
        stamp = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return "%s, %d, 2070, 900.0, Not Active, Not Active, Not Active, %s" % (
            stamp, sm, "Active" if cap else "Not Active")

    t = 1.8e9
    lines = [line(t - 0.3, 900, True), line(t + 0.01, 2070, False),
             line(t + 0.03, 2055, False), "not a sample"]
    c = bench.summarize_clock_lines(lines, (t, t + 0.05), 20)
    assert c["samples"] == 2 and c["samples_in_timed_region"] == 2
    assert c["sm_mhz"] == pytest.approx(2062.5) and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == []  # the power-cap sample lies before the window
    c = bench.summarize_clock_lines(lines, (t + 1, t + 2), 20)
    assert c["samples"] == 3 and c["samples_in_timed_region"] == 0
    assert c["reasons"] == ["sw_power_cap"]
