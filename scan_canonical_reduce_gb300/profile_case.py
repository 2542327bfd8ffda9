"""Runs one hot-path row at a chosen size, for profilers (ncu) to capture.

  python -m scan_canonical_reduce_gb300.profile_case --row reduce --n 33554432 --L 16
  python -m scan_canonical_reduce_gb300.profile_case --row scan --policy iterated_pairwise
  python -m scan_canonical_reduce_gb300.profile_case --row rows --rows 8192 --cols 4096

Inputs are the benchmark's seeded families; each call is repeated --reps
times after --warmup untimed calls, then the stream is synchronised.
"""
from __future__ import annotations

import argparse
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import workloads as W  # noqa: E402

import scan_canonical_reduce_gb300 as scr  # noqa: E402


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--row", required=True, choices=["reduce", "scan", "rows", "cols"])
    ap.add_argument("--n", type=int, default=1 << 25)
    ap.add_argument("--L", type=int, default=16)
    ap.add_argument("--policy", default="iterated_pairwise")
    ap.add_argument("--B", type=int, default=1)
    ap.add_argument("--rows", type=int, default=8192)
    ap.add_argument("--cols", type=int, default=4096)
    ap.add_argument("--levels", type=int, default=90)
    ap.add_argument("--dtype", default="f64", choices=["f64", "f32"])
    ap.add_argument("--warmup", type=int, default=1)
    ap.add_argument("--reps", type=int, default=2)
    a = ap.parse_args()
    dev = torch.device("cuda:0")
    if a.row == "reduce":
        import numpy as np
        x = torch.from_numpy(W.family2(a.n, np.float64 if a.dtype == "f64" else np.float32)).to(dev)
        fn = lambda: scr.reduce(x, a.L, 0.0)  # noqa: E731
    elif a.row == "scan":
        x = torch.from_numpy(W.family3(a.n)).to(dev)
        if a.dtype == "f32":
            x = x.float()
        y = torch.empty_like(x)
        fn = lambda: scr.inclusive_scan(x, a.policy, a.B, out=y)  # noqa: E731
    elif a.row == "rows":
        x = torch.from_numpy(W.family4(a.rows, a.cols)).to(dev)
        fn = lambda: scr.reduce_batched(x, a.L, 0.0, dim=-1)  # noqa: E731
    else:
        x = torch.from_numpy(W.family5(a.levels, a.cols)).to(dev).view(a.levels, a.cols)
        y = torch.empty_like(x)
        fn = lambda: scr.inclusive_scan_batched(x, a.policy, a.B, dim=0, out=y)  # noqa: E731
    for _ in range(a.warmup + a.reps):
        fn()
    torch.cuda.synchronize(dev)
    print("ok", a.row, a.n)


if __name__ == "__main__":
    main()
