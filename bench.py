#!/usr/bin/env python
"""Benchmark of the canonical reduce / scan hot path on GB300.

One step = one pass over every row of the hot path, each on its own seeded
synthetic input (inputs larger than L2, resident in HBM before the timed
region):
  reduce_f64_L{16,128,1024}  canonical reduce, fp64, n = 2^28, family-2 values
  scan_iterated_pairwise     inclusive scan, fp64, n = 2^28, U[-1, 1)
  scan_block_dyadic_{16,256} inclusive scan, fp64, n = 2^28, U[-1, 1)
  reduce_rows_f32_L128       batched row reduce, fp32, 65,536 x 4,096
  colscan_{block_dyadic16,left_fold}  batched column scan, fp64, 90 x 200,000
value = algorithmic bytes of all rows / device time of the step (GB/s);
e2e   = the same through the public API with pinned host buffers, the
        host->device copy of the inputs and the device->host copy of every
        result inside the timed region.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]
  python bench.py --one-row {reduce,scan,rows,cols} [--n --L --policy --B --rows
                  --cols --levels --dtype --warmup --steps]   (one row, for ncu)

With N > 1 (torchrun) every rank runs the same step on its own GPU
(replicas: the rows are independent problems, no exchange); rank 0 prints.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "canonical reduce/scan GB/s (fp64, N=2^28) & % of HBM roofline; 0-ULP vs oracle"
N = 1 << 28
COLS_LEVELS, COLS_N = 90, 200000
ROWS_R, ROWS_C = 65536, 4096


# ------------------------------------------------------- algorithmic counts
def popcount_sum(n: int) -> int:
    """sum of popcount(j) for j = 1..n."""
    total, bit = 0, 0
    while (1 << bit) <= n:
        period = 1 << (bit + 1)
        full = (n + 1) // period
        total += full * (1 << bit) + max(0, (n + 1) % period - (1 << bit))
        bit += 1
    return total


def adds_iterated(n: int) -> int:
    """Adds of an iterated_pairwise scan: every complete aligned node
    (n - popcount(n)) plus popcount(i+1) - 1 right-nested combinations."""
    return (n - bin(n).count("1")) + (popcount_sum(n) - n)


def adds_block_dyadic(n: int, B: int) -> int:
    full, rem = divmod(n, B)
    a = full * adds_iterated(B) + (adds_iterated(rem) if rem else 0)
    return a + max(0, n - B) + max(0, -(-n // B) - 2)  # carries applied + chain


def adds_pairwise(n: int) -> int:
    """Adds of a pairwise scan: every complete aligned node (n - popcount(n))
    plus one left-nested combination per prefix length that is not a power
    of two."""
    return (n - bin(n).count("1")) + (n - n.bit_length())


SWEEP_N = (1 << 20, 1 << 24, 1 << 28, (1 << 28) + 37, 1 << 30)
N_MAX = 1 << 30
ROWS_B = (1024, 262144)


def size_tag(n: int) -> str:
    """2^k, or 2^k + r, as "2e<k>" or "2e<k>p<r>"."""
    k = n.bit_length() - 1
    r = n - (1 << k)
    return "2e%d" % k + ("p%d" % r if r else "")


def extra_rows():
    """Rows beyond the headline step, timed on their own after it and
    reported under "extras"; not part of value: the next policies, the
    reduce sweep over sizes, binary32 and lane counts, the U[0, 1) reduce at
    2^20 and the 1,024 x 262,144 row reduce."""
    rs = [("scan_pairwise", "scan", {"policy": "pairwise", "B": 1}, 16 * N,
           adds_pairwise(N), "f64"),
          # init combined once with each of the n - 1 (n) observations
          ("scan_iterated_pairwise_exclusive", "scan_ex",
           {"policy": "iterated_pairwise", "B": 1, "mode": "exclusive"}, 16 * N,
           adds_iterated(N) - 1 + (N - 1), "f64"),
          ("scan_block_dyadic_16_include_initial", "scan_ex",
           {"policy": "block_dyadic", "B": 16, "mode": "include_initial"}, 16 * N + 8,
           adds_block_dyadic(N, 16) + N, "f64")]
    # binary32 scans of the same input rounded to binary32 (the carry chains
    # of left_fold and block_dyadic through the estimated-chain classification)
    for pol, B in (("iterated_pairwise", 1), ("pairwise", 1), ("block_dyadic", 16),
                   ("block_dyadic", 256), ("left_fold", 1)):
        name = "scan_%s%s_f32" % (pol, "_%d" % B if pol == "block_dyadic" else "")
        adds = {"iterated_pairwise": adds_iterated(N), "pairwise": adds_pairwise(N),
                "block_dyadic": adds_block_dyadic(N, B), "left_fold": N - 1}[pol]
        rs.append((name, "scan", {"policy": pol, "B": B, "dt": "f32"}, 8 * N, adds, "f32"))
    for dt, es in (("f64", 8), ("f32", 4)):
        for n in SWEEP_N:
            for L in (16, 128, 1024):
                rs.append(("sweep_reduce_%s_n%s_L%d" % (dt, size_tag(n), L), "reduce",
                           {"L": L, "n": n, "dt": dt}, es * n, n, dt))
    for L in (16, 128):
        rs.append(("reduce_u01_f64_n2e20_L%d" % L, "reduce_u01", {"L": L, "n": 1 << 20},
                   8 << 20, 1 << 20, "f64"))
    r, c = ROWS_B
    rs.append(("reduce_rows_f32_L128_%dx%d" % (r, c), "rows_b", {"L": 128, "rows": r,
                                                                  "cols": c},
               4 * r * c + 4 * r, r * c, "f32"))
    return rs


def rows_spec():
    """(name, kind, params, algorithmic bytes, algorithmic adds, dtype)."""
    rs = []
    for L in (16, 128, 1024):
        rs.append(("reduce_f64_L%d" % L, "reduce", {"L": L}, 8 * N, N, "f64"))
    rs.append(("scan_iterated_pairwise", "scan", {"policy": "iterated_pairwise", "B": 1},
               16 * N, adds_iterated(N), "f64"))
    for B in (16, 256):
        rs.append(("scan_block_dyadic_%d" % B, "scan", {"policy": "block_dyadic", "B": B},
                   16 * N, adds_block_dyadic(N, B), "f64"))
    rs.append(("reduce_rows_f32_L128", "rows", {"L": 128},
               4 * ROWS_R * ROWS_C + 4 * ROWS_R, ROWS_R * ROWS_C, "f32"))
    for pol, B in (("block_dyadic", 16), ("left_fold", 1)):
        name = "colscan_%s%s" % (pol, B if pol == "block_dyadic" else "")
        adds = COLS_N * (adds_block_dyadic(COLS_LEVELS, B) if pol == "block_dyadic"
                         else COLS_LEVELS - 1)
        rs.append((name, "cols", {"policy": pol, "B": B}, 16 * COLS_LEVELS * COLS_N, adds,
                   "f64"))
    return rs


HBM_NOMINAL_GBS = 7900.0  # GB300's nominal HBM3e bandwidth (8 stacks)


def row_elems(r) -> int:
    """Input elements of a row: n for the 1-D rows, rows x cols, levels x columns."""
    kind, p = r[1], r[2]
    if kind == "rows":
        return ROWS_R * ROWS_C
    if kind == "rows_b":
        return p["rows"] * p["cols"]
    if kind == "cols":
        return COLS_LEVELS * COLS_N
    return p.get("n", N)


def rate_stats(r, ms: float, hbm_peak, dadd_rate: float, fadd_rate: float) -> dict:
    """One row's rates at a median time of ms: algorithmic GB/s against the
    measured copy peak and the nominal HBM figure, elements/s, and adds/s
    against the measured add rate of the row's type."""
    sec = ms * 1e-3
    gbs = r[3] / sec / 1e9
    add_rate = r[4] / sec
    peak_add = dadd_rate if r[5] == "f64" else fadd_rate
    return {"ms": round(ms, 4), "gb_s": round(gbs, 1),
            "hbm_frac": round(gbs / hbm_peak, 4) if hbm_peak else None,
            "hbm_frac_nominal": round(gbs / HBM_NOMINAL_GBS, 4),
            "elems_per_s": row_elems(r) / sec,
            "adds_per_s": add_rate, "alu_frac": round(add_rate / peak_add, 4),
            "bytes": r[3], "adds": r[4], "dtype": r[5]}


# ----------------------------------------------------------------- inputs
def host_inputs():
    """Every row's input, generated once on the host. The reduce rows of the
    step and of the size sweep read prefixes of one 2^30-element array per
    type (the generator is counter-based: family2(n) is the first n elements
    of family2(2^30))."""
    return {
        "f2": W.family2(N_MAX),                  # reduce (step: the first 2^28)
        "f2f": W.family2(N_MAX, np.float32),     # binary32 reduce sweep
        "f1": W.family1(1 << 20),                # U[0, 1) reduce at 2^20
        "f3": W.family3(N),                      # 1-D scans
        "f4": W.family4(ROWS_R, ROWS_C),         # row reduce
        "f4b": W.family4(*ROWS_B),               # row reduce, 1,024 x 262,144
        "f5": W.family5(COLS_LEVELS, COLS_N),    # column scans
    }


# ------------------------------------------------------------- ranks
def job_config(world: int) -> dict:
    """The workload both arms name: every hot-path row at its full size."""
    return {"workload": "all hot-path rows at n = 2^28 fp64 (reduce L=16/128/1024, "
                        "iterated_pairwise and block_dyadic<16>/<256> scans) + 65536x4096 "
                        "fp32 row reduce + 90x200000 fp64 column scans",
            "n": N, "l2": "every input larger than L2 (>=144 MB); no flush",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def max_over_ranks(x: float, dist, dev) -> float:
    """The largest value of x over the ranks (a job takes as long as its
    slowest rank); x itself on one process. dev: a device of the process
    group's backend (the rank's GPU for NCCL, the CPU for gloo)."""
    if not dist or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_step: int, steps: int, world: int, seconds: float) -> float:
    """Whole-job throughput of `world` replicas: every rank processed
    bytes_per_step each step; the job's time is the slowest rank's."""
    return bytes_per_step * steps * world / seconds / 1e9


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons while running,
    every INTERVAL_MS; stop() keeps the samples stamped inside the timed
    window (all of them if none falls inside)."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 20

    def __init__(self, gpu_uuid: str | None):
        self.uuid = gpu_uuid
        self.proc = None
        self.lines = []

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
               "-lms", str(self.INTERVAL_MS)]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self, window=None):
        """window: (t0, t1) in time.time() seconds, the timed region."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        return summarize_clock_lines(self.lines, window, self.INTERVAL_MS)


def summarize_clock_lines(lines, window, interval_ms):
    """Median SM clock, max clock and the throttle reasons seen, over the
    samples stamped inside `window` (local-time stamps of nvidia-smi), or over
    all samples when none is inside."""
    import datetime
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    samples = []  # (seconds, sm, max, reasons)
    for l in lines:
        f = [x.strip() for x in l.split(",")]
        if len(f) < 8:
            continue
        try:
            ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            sm, mx = float(f[1]), float(f[2])
        except ValueError:
            continue
        samples.append((ts, sm, mx, {nm for nm, v in zip(names, f[4:8])
                                     if v.lower().startswith("active")}))
    inside = [x for x in samples if window and window[0] <= x[0] <= window[1]]
    use = inside or samples
    reasons = set().union(*(x[3] for x in use)) if use else set()
    return {"sm_mhz": statistics.median(x[1] for x in use) if use else None,
            "sm_max_mhz": max(x[2] for x in use) if use else None,
            "samples": len(use), "samples_in_timed_region": len(inside),
            "interval_ms": interval_ms, "reasons": sorted(reasons)}


# ------------------------------------------------------------- GPU arm
def run_native(args):
    import torch

    import scan_canonical_reduce_gb300 as scr

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.gpus != world:
        raise SystemExit("--gpus %d but WORLD_SIZE=%d" % (args.gpus, world))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    rows = rows_spec()
    hin = host_inputs()
    # device-resident inputs and outputs
    x2_all = torch.from_numpy(hin["f2"]).to(dev)
    x2 = x2_all[:N]
    x2f_all = torch.from_numpy(hin["f2f"]).to(dev)
    x1 = torch.from_numpy(hin["f1"]).to(dev)
    x4b = torch.from_numpy(hin["f4b"]).to(dev)
    x3 = torch.from_numpy(hin["f3"]).to(dev)
    x3f = x3.float()  # the 1-D scan input rounded to binary32
    y_scan32 = torch.empty_like(x3f)
    x4 = torch.from_numpy(hin["f4"]).to(dev)
    x5 = torch.from_numpy(hin["f5"]).to(dev).view(COLS_LEVELS, COLS_N)
    y_scan = torch.empty_like(x3)
    y_scan1 = torch.empty(N + 1, dtype=x3.dtype, device=dev)  # include_initial: n + 1
    y_cols = torch.empty_like(x5)
    r_out = torch.empty(1, dtype=torch.float64, device=dev)
    r_out32 = torch.empty(1, dtype=torch.float32, device=dev)
    rows_out = torch.empty(ROWS_R, dtype=torch.float32, device=dev)
    rows_out_b = torch.empty(ROWS_B[0], dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def run_row(row):
        name, kind, p = row[0], row[1], row[2]
        if kind == "reduce":
            if p.get("dt", "f64") == "f32":
                scr.reduce(x2f_all[:p["n"]], p["L"], 0.0, out=r_out32)
            else:
                scr.reduce(x2_all[:p.get("n", N)], p["L"], 0.0, out=r_out)
        elif kind == "reduce_u01":
            scr.reduce(x1, p["L"], 0.0, out=r_out)
        elif kind == "rows_b":
            scr.reduce_batched(x4b, p["L"], 0.0, dim=-1, out=rows_out_b)
        elif kind == "scan":
            if p.get("dt", "f64") == "f32":
                scr.inclusive_scan(x3f, p["policy"], p["B"], out=y_scan32)
            else:
                scr.inclusive_scan(x3, p["policy"], p["B"], out=y_scan)
        elif kind == "scan_ex":
            if p["mode"] == "exclusive":
                scr.exclusive_scan(x3, p["policy"], p["B"], 0.5, out=y_scan)
            else:
                scr.scan_include_initial(x3, p["policy"], p["B"], 0.5, out=y_scan1)
        elif kind == "rows":
            scr.reduce_batched(x4, p["L"], 0.0, dim=-1, out=rows_out)
        elif kind == "cols":
            scr.inclusive_scan_batched(x5, p["policy"], p["B"], dim=0, out=y_cols)

    def step():
        for row in rows:
            run_row(row)

    # ALU roofline denominators, measured on this GPU by libcr's calibration
    dadd_rate, dadd_lat = scr.measure_add_peak(torch.float64, dev)
    fadd_rate, _ = scr.measure_add_peak(torch.float32, dev)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    # ---- per-kernel breakdown: K more steps with every libcr launch
    # bracketed by CUDA events on its stream (not the timed region: the
    # events add a little to each launch)
    scr.profile_select(None)
    scr.profile_enable(True)
    row_launches = {r[0]: [] for r in rows}
    for _ in range(args.steps):
        for row in rows:
            before = scr.launch_count()
            run_row(row)
            row_launches[row[0]].append(scr.launch_count() - before)
    torch.cuda.synchronize(dev)
    scr.profile_enable(False)
    prof = scr.profile_collect()
    kern = {}
    for name, ms in prof:
        k = kern.setdefault(name, [0, 0.0])
        k[0] += 1
        k[1] += ms
    top_kernel = max(kern, key=lambda k: kern[k][1]) if kern else None

    # ---- timed region: K steps, per-row events on the stream; of the
    # launches, only the dominant kernel's carry events (its duration for
    # the roofline)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    sampler = ClockSampler(uuid)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    launches0 = scr.launch_count()
    scr.profile_select(top_kernel)
    scr.profile_enable(top_kernel is not None)
    ev = {r[0]: [] for r in rows}
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    t0.record(stream)
    for _ in range(args.steps):
        for row in rows:
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            run_row(row)
            b.record(stream)
            ev[row[0]].append((a, b))
    t1.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    scr.profile_enable(False)
    scr.profile_select(None)
    launches = scr.launch_count() - launches0
    prof_top = scr.profile_collect()
    clocks = sampler.stop((wall0, wall1))
    ms_total = max_over_ranks(t0.elapsed_time(t1), dist, dev)
    if dist:
        dist.barrier()

    step_bytes = sum(r[3] for r in rows)
    ms_per_step = ms_total / args.steps
    value = job_gbs(step_bytes, args.steps, world, ms_total * 1e-3)
    peaks = measured_peaks()
    hbm_peak = peaks.get("hbm_gbs")

    row_stats = {}
    for r in rows:
        ms = statistics.median([a.elapsed_time(b) for a, b in ev[r[0]]])
        row_stats[r[0]] = rate_stats(r, ms, hbm_peak, dadd_rate, fadd_rate)

    # per-row kernel times (profiled steps): the launch list is in issue
    # order, rows in turn
    per_row = {r[0]: {} for r in rows}
    pos = 0
    for _ in range(args.steps):
        for r in rows:
            cnt = row_launches[r[0]].pop(0)
            for name, ms in prof[pos:pos + cnt]:
                per_row[r[0]][name] = per_row[r[0]].get(name, 0.0) + ms / args.steps
            pos += cnt
    for r in rows:
        row_stats[r[0]]["kernels_ms"] = {k: round(v, 4) for k, v in per_row[r[0]].items()}

    # per-kernel launch list (profiled steps), and the dominant kernel's
    # launches in the timed region
    tot_k = sum(v[1] for v in kern.values()) or 1.0
    kernels = {k: {"launches": v[0], "ms_total": round(v[1], 3), "share": round(v[1] / tot_k, 4)}
               for k, v in sorted(kern.items(), key=lambda kv: -kv[1][1])}
    timed_top = {}
    for name, ms in prof_top:
        k = timed_top.setdefault(name, {"launches": 0, "ms_total": 0.0})
        k["launches"] += 1
        k["ms_total"] += ms
    # fp64 add peak from unit counts and clocks: GB300's nominal 1.25 TFLOP/s
    # fp64 (FMA = 2 flops) over 152 SMs at 2.07 GHz is 2 fp64 adds per clock
    # per SM (a warp-wide add every 16 clocks)
    props = torch.cuda.get_device_properties(dev)
    sm_max_mhz = clocks.get("sm_max_mhz") or 2070.0
    dadd_nominal = props.multi_processor_count * 2 * sm_max_mhz * 1e6
    roofline = dominant_roofline(timed_top or kernels, prof_top or prof, row_stats, dadd_rate,
                                 dadd_lat, hbm_peak, args.steps, dadd_nominal)

    extras = run_extras(args, scr, torch, dev, stream, run_row, dadd_rate, fadd_rate, hbm_peak)

    # ---- e2e through the public API with pinned host buffers
    e2e = run_e2e(args, scr, torch, dev, hin, rows, world, dist)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(seconds=args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": STEP_DTYPE,
            "data": "synthetic (seeded SplitMix64 families; no dataset)",
            "config": job_config(world),
            "rows": row_stats, "kernels": kernels, "roofline": roofline, "extras": extras,
            "peaks": {"hbm_gbs": hbm_peak, "dadd_per_s": dadd_rate, "dadd_latency_ns": dadd_lat,
                      "fadd_per_s": fadd_rate},
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
        }
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


L2_FLUSH_BYTES = 512 << 20  # more than the 126 MB L2
# the arithmetic type of the step's rows (both arms)
STEP_DTYPE = "mixed: f64 (every row but one), f32 (the 65536 x 4096 row reduce)"


def run_extras(args, scr, torch, dev, stream, run_row, dadd_rate, fadd_rate, hbm_peak):
    """Each extra row timed alone: W warm-up calls, then K calls bracketed by
    CUDA events on the launching stream (no per-launch events inside), then
    one call with libcr's per-launch events for the kernel breakdown. A row
    whose input is smaller than twice the L2 gets a 512 MB write between its
    calls (outside the events), so that every call starts from HBM."""
    out = {}
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for r in extra_rows():
        small = r[3] < 2 * L2_FLUSH_BYTES // 4
        for _ in range(args.warmup):
            run_row(r)
        torch.cuda.synchronize(dev)
        evs = []
        for _ in range(args.steps):
            if small:
                flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            run_row(r)
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize(dev)
        ms = statistics.median([a.elapsed_time(b) for a, b in evs])
        # kernel breakdown: one more call with every launch bracketed by
        # events (outside the timed calls)
        if small:
            flush.zero_()
        scr.profile_enable(True)
        run_row(r)
        torch.cuda.synchronize(dev)
        scr.profile_enable(False)
        prof = scr.profile_collect()
        kms = {}
        for name, t in prof:
            kms[name] = kms.get(name, 0.0) + t
        out[r[0]] = rate_stats(r, ms, hbm_peak, dadd_rate, fadd_rate)
        out[r[0]]["kernels_ms"] = {k: round(v, 4) for k, v in kms.items()}
        if small:
            out[r[0]]["l2"] = "flushed between calls"
    del flush
    return out


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return {"hbm_gbs": 6800.0, "note": "fallback"}


# DRAM bytes (read + written) per launch from one ncu capture of the kernel,
# scaled from the captured size to the benchmark's n = 2^28 by elements
# processed (traffic grows in proportion). Each figure holds only for the
# sources it was captured from: "sources" maps each file to the first 16 hex
# digits of its SHA-256 at capture time, and the figure reads as None once
# any of them differs (the kernel changed after the capture).
CSRC_DIR = os.path.join(ROOT, "scan_canonical_reduce_gb300", "csrc")
NCU_TRAFFIC = {
    # one-row iterated_pairwise scan, n = 2^25: 268.94 MB read + 263.24 MB
    # written, x 8
    "scan_onepass_kernel": {"bytes": (268.93568e6 + 263.244032e6) * 8,
                            "sources": {'cr_scan.cu': '35729d7c87f88a90', 'cr_scan.h': '13de311023332c6d', 'cr_device.cuh': 'b3f5f88a2d146302'}},
    # one-row reduce, n = 2^25, L = 16, level-0 pass: 268.47 MB read + 2.85 MB
    # written, x 8
    "lane_pass_kernel": {"bytes": (268.472576e6 + 2.846976e6) * 8,
                         "sources": {'cr_reduce.cu': 'fb65bc83a3c3da16', 'cr_plan.h': 'd781220e97c4b36f', 'cr_device.cuh': 'b3f5f88a2d146302'}},
}


def source_digest(name: str) -> str | None:
    import hashlib
    try:
        with open(os.path.join(CSRC_DIR, name), "rb") as f:
            return hashlib.sha256(f.read()).hexdigest()[:16]
    except OSError:
        return None


def ncu_traffic(kernel: str):
    """The recorded traffic of `kernel` per launch, or None when there is no
    capture or its sources have changed since."""
    t = NCU_TRAFFIC.get(kernel)
    if not t or not t["sources"]:
        return None
    if any(source_digest(f) != d for f, d in t["sources"].items()):
        return None
    return t["bytes"]


def dominant_roofline(kernels, prof, row_stats, dadd_rate, dadd_lat, hbm_peak, steps,
                      dadd_nominal):
    """Roofline of the kernel with the largest share of device time:
    achieved = algorithmic work per launch / its average launch duration
    (CUDA events recorded by libcr around each launch in the timed region).
    An fp64-add-bound kernel is rated against the add rate derived from the
    SM count and clock (dadd_nominal); the rate libcr's calibration kernel
    reaches on this GPU is reported beside it."""
    if not kernels:
        return None
    top = next(iter(kernels))
    launches = kernels[top]["launches"]
    avg_ms = kernels[top]["ms_total"] / max(1, launches)
    if top == "scan_onepass_kernel":
        # one launch = the whole iterated_pairwise scan of n = 2^28 fp64
        adds = row_stats["scan_iterated_pairwise"]["adds"]
        nbytes = row_stats["scan_iterated_pairwise"]["bytes"]
        achieved = adds / (avg_ms * 1e-3)
        return {"kernel": top, "bound": "alu", "achieved": achieved, "peak": dadd_nominal,
                "unit": "fp64 adds/s", "frac": round(achieved / dadd_nominal, 4),
                "traffic": ncu_traffic(top),
                "work_per_launch": {"adds": adds, "bytes": nbytes},
                "measured_peak": {"value": dadd_rate, "frac": round(achieved / dadd_rate, 4)},
                "hbm": {"achieved_gbs": round(nbytes / (avg_ms * 1e-3) / 1e9, 1),
                        "peak_gbs": hbm_peak,
                        "frac": round(nbytes / (avg_ms * 1e-3) / 1e9 / hbm_peak, 4)},
                "note": "peak = SMs x 2 fp64 adds a clock x max SM clock (GB300's nominal "
                        "1.25 TFLOP/s fp64); measured_peak = libcr's calibration kernel "
                        "(independent round-to-nearest adds on all SMs); traffic from an "
                        "ncu capture at n = 2^25 scaled by 8, null when the kernel's sources "
                        "changed after the capture"}
    if top == "lane_pass_kernel":
        r = row_stats["reduce_f64_L16"]
        achieved = r["bytes"] / (r["ms"] * 1e-3) / 1e9
        return {"kernel": top, "bound": "alu", "achieved": r["adds"] / (r["ms"] * 1e-3),
                "peak": dadd_nominal, "unit": "fp64 adds/s",
                "frac": round(r["adds"] / (r["ms"] * 1e-3) / dadd_nominal, 4),
                "measured_peak": {"value": dadd_rate,
                                  "frac": round(r["adds"] / (r["ms"] * 1e-3) / dadd_rate, 4)},
                "traffic": ncu_traffic(top),
                "hbm": {"achieved_gbs": round(achieved, 1), "peak_gbs": hbm_peak,
                        "frac": round(achieved / hbm_peak, 4)}}
    if top == "carry_chain_kernel":
        K = N // 16 - 1
        chains = [ms for nm, ms in prof if nm == top]
        ms = max(chains) if chains else avg_ms
        achieved = K / (ms * 1e-3)
        peak = 1e9 / dadd_lat
        return {"kernel": top, "bound": "alu", "achieved": achieved, "peak": peak,
                "unit": "dependent adds/s", "frac": round(achieved / peak, 4),
                "traffic": None}
    return {"kernel": top, "bound": "alu", "achieved": None, "peak": dadd_nominal,
            "unit": "fp64 adds/s", "frac": None, "traffic": None}


def run_e2e(args, scr, torch, dev, hin, rows, world, dist):
    """Same rows through the public API on pinned host tensors: each call
    copies its input in and its result out, inside the timed region."""
    h2 = torch.from_numpy(hin["f2"][:N]).pin_memory()
    h3 = torch.from_numpy(hin["f3"]).pin_memory()
    h4 = torch.from_numpy(hin["f4"]).pin_memory()
    h5 = torch.from_numpy(hin["f5"]).view(COLS_LEVELS, COLS_N).pin_memory()
    h2d = d2h = 0
    for r in rows:
        kind = r[1]
        if kind == "reduce":
            h2d += h2.numel() * 8
            d2h += 8
        elif kind == "scan":
            h2d += h3.numel() * 8
            d2h += h3.numel() * 8
        elif kind == "rows":
            h2d += h4.numel() * 4
            d2h += ROWS_R * 4
        else:
            h2d += h5.numel() * 8
            d2h += h5.numel() * 8

    def step():
        for r in rows:
            kind, p = r[1], r[2]
            if kind == "reduce":
                scr.reduce(h2, p["L"], 0.0)
            elif kind == "scan":
                scr.inclusive_scan(h3, p["policy"], p["B"])
            elif kind == "rows":
                scr.reduce_batched(h4, p["L"], 0.0, dim=-1)
            else:
                scr.inclusive_scan_batched(h5, p["policy"], p["B"], dim=0)

    for _ in range(max(1, args.warmup)):  # allocations, page-locked buffers, plans
        step()
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    steps = max(1, min(args.steps + 2, 7))
    step_ms = []
    t = time.perf_counter()
    for _ in range(steps):
        t1 = time.perf_counter()
        step()  # every call returns host data: the step ends synchronised
        step_ms.append(round((time.perf_counter() - t1) * 1e3, 2))
    torch.cuda.synchronize(dev)
    sec = max_over_ranks(time.perf_counter() - t, dist, dev)
    step_bytes = sum(r[3] for r in rows)
    # the host link of this pool stalls at random (plain 2 GB copies: ~10 %
    # of them 36-144 ms instead of 21 ms), so the value is taken at the
    # median step; the mean and every step's time are reported beside it
    med = max_over_ranks(sorted(step_ms)[len(step_ms) // 2] / 1e3, dist, dev)
    return {"value": round(job_gbs(step_bytes, 1, world, med), 2), "unit": "GB/s",
            "estimator": "median step",
            "mean_value": round(job_gbs(step_bytes, steps, world, sec), 2),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "step_ms": step_ms}


# ------------------------------------------------------- oracle (CPU) leg
def cpu_sample_rows(scale: int):
    """Bounded sample of every row for the oracle: same families, n / scale."""
    n = N // scale
    rs = []
    for L in (16, 128, 1024):
        rs.append(("reduce_f64_L%d" % L, "reduce", {"L": L}, 8 * n))
    rs.append(("scan_iterated_pairwise", "scan", {"policy": "iterated_pairwise", "B": 1}, 16 * n))
    for B in (16, 256):
        rs.append(("scan_block_dyadic_%d" % B, "scan", {"policy": "block_dyadic", "B": B}, 16 * n))
    rr = max(1, ROWS_R // scale)
    rs.append(("reduce_rows_f32_L128", "rows", {"L": 128, "rows": rr}, 4 * rr * ROWS_C))
    cc = max(1, COLS_N // scale)
    for pol, B in (("block_dyadic", 16), ("left_fold", 1)):
        rs.append(("colscan", "cols", {"policy": pol, "B": B, "cols": cc},
                   16 * COLS_LEVELS * cc))
    return n, rs


def sample_inputs(base: int, cache={}):
    """The oracle sample's inputs at 1/base of every row, generated once; a
    smaller sample is their prefix (the generators are counter-based)."""
    if base not in cache:
        cache.clear()
        cc = max(1, COLS_N // base)
        cache[base] = {
            "f2": W.family2(N // base), "f3": W.family3(N // base),
            "f4": W.family4(ROWS_R, ROWS_C, first_rows=max(1, ROWS_R // base)),
            "f5": W.family5(COLS_LEVELS, COLS_N).reshape(COLS_LEVELS, COLS_N)[:, :cc].copy(),
        }
    return cache[base]


def oracle_step(scale: int, base: int | None = None):
    """One pass of the oracle over every row at 1/scale of its size (inputs
    from the sample at 1/base, base dividing scale): (bytes, seconds, n)."""
    import oracle
    n, rs = cpu_sample_rows(scale)
    s0 = sample_inputs(base or scale)
    c = {"f2": s0["f2"][:n], "f3": s0["f3"][:n], "f4": s0["f4"][: max(1, ROWS_R // scale)],
         "f5": s0["f5"][:, : max(1, COLS_N // scale)].copy().reshape(-1)}
    t = time.perf_counter()
    for name, kind, p, _ in rs:
        if kind == "reduce":
            oracle.reduce(c["f2"], p["L"], 0.0)
        elif kind == "scan":
            oracle.scan(c["f3"], p["policy"], p["B"])
        elif kind == "rows":
            oracle.reduce_batched(c["f4"].reshape(-1), p["rows"], ROWS_C, 1, ROWS_C, p["L"],
                                  np.float32(0.0))
        else:
            oracle.scan_batched(c["f5"], p["cols"], COLS_LEVELS, p["cols"], 1, p["policy"], p["B"])
    sec = time.perf_counter() - t
    return sum(r[3] for r in rs), sec, n


def cpu_baseline(seconds: float = 15.0):
    """The oracle as it stands, single-threaded on this host, on a bounded
    sample of the same workload (every row at 1/scale of its size)."""
    # double the sample (1/64 of every row, then 1/32, ... up to 1/2) until
    # one measured pass takes at least 40 % of the budget
    scale = 64
    b, s, n = oracle_step(scale, base=2)
    while scale > 2 and s < 0.4 * seconds:
        scale //= 2
        b, s, n = oracle_step(scale, base=2)
    return {"value": round(b / s / 1e9, 4), "unit": "GB/s", "cores": 1,
            "host_cores_visible": len(os.sched_getaffinity(0)), "kind": "oracle",
            "seconds": round(s, 2),
            "sample": "every row at 1/%d of its size (1-D n = %d; row reduce %d rows; "
                      "column scans %d columns), same value families" %
                      (scale, n, max(1, ROWS_R // scale), max(1, COLS_N // scale))}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    scale = args.ref_scale
    oracle_step(scale)  # build + inputs, untimed
    for _ in range(args.warmup):
        oracle_step(scale)
    tot_b = tot_s = 0.0
    for _ in range(args.steps):
        b, s, n = oracle_step(scale)
        tot_b += b
        tot_s += s
    value = tot_b / tot_s / 1e9
    line = {
        "metric": METRIC, "impl": "reference", "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot_s / args.steps * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": STEP_DTYPE, "data": "synthetic",
        "config": job_config(world),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": "every row at 1/%d of its size (1-D n = %d; the oracle "
                                   "is single-threaded)" % (scale, n)},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ------------------------------------------------------- one row (profilers)
def run_one_row(args):
    """One hot-path row at a chosen size, called --warmup + --steps times and
    then synchronised, for a profiler (ncu) to capture; prints no JSON line.
    Inputs are the benchmark's seeded families."""
    import torch

    import scan_canonical_reduce_gb300 as scr

    dev = torch.device("cuda:0")
    f32 = args.dtype == "f32"
    if args.one_row == "reduce":
        x = torch.from_numpy(W.family2(args.n, np.float32 if f32 else np.float64)).to(dev)
        fn = lambda: scr.reduce(x, args.L, 0.0)  # noqa: E731
    elif args.one_row == "scan":
        x = torch.from_numpy(W.family3(args.n)).to(dev)
        if f32:
            x = x.float()
        y = torch.empty_like(x)
        fn = lambda: scr.inclusive_scan(x, args.policy, args.B, out=y)  # noqa: E731
    elif args.one_row == "rows":
        x = torch.from_numpy(W.family4(args.rows, args.cols)).to(dev)
        fn = lambda: scr.reduce_batched(x, args.L, 0.0, dim=-1)  # noqa: E731
    else:
        x = torch.from_numpy(W.family5(args.levels, args.cols)).to(dev).view(args.levels,
                                                                           args.cols)
        y = torch.empty_like(x)
        fn = lambda: scr.inclusive_scan_batched(x, args.policy, args.B, dim=0,  # noqa: E731
                                                out=y)
    for _ in range(args.warmup + args.steps):
        fn()
    torch.cuda.synchronize(dev)
    print("ok", args.one_row, args.n)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-scale", type=int, default=32)
    # --one-row: a single row for a profiler (no timing, no JSON line)
    ap.add_argument("--one-row", choices=["reduce", "scan", "rows", "cols"])
    ap.add_argument("--n", type=int, default=1 << 25)
    ap.add_argument("--L", type=int, default=16)
    ap.add_argument("--policy", default="iterated_pairwise")
    ap.add_argument("--B", type=int, default=1)
    ap.add_argument("--rows", type=int, default=8192)
    ap.add_argument("--cols", type=int, default=4096)
    ap.add_argument("--levels", type=int, default=90)
    ap.add_argument("--dtype", default="f64", choices=["f64", "f32"])
    args = ap.parse_args()
    if args.one_row:
        run_one_row(args)
        return
    if args.warmup < 3 and args.impl == "native":
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
