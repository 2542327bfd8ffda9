"""The scans and reductions captured in a CUDA graph and replayed: every
kernel path (one pass, local + fused chain and fix-up, up/down, pairwise,
the left fold's fused chain, the reduce pyramid) with its workspace made
before the capture, then bit-equal to eager calls on new inputs copied into
the captured buffers."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

CALLS = [("scan", "iterated_pairwise", 1), ("scan", "pairwise", 1), ("scan", "left_fold", 1),
         ("scan", "block_dyadic", 16), ("scan", "block_dyadic", 256),
         ("scan", "block_dyadic", 4096), ("exclusive", "block_dyadic", 16),
         ("reduce", None, 16), ("reduce_policy", "block_dyadic", 16)]


@pytest.fixture(scope="module")
def scr():
    import scan_canonical_reduce_gb300 as m
    return m


def run(scr, kind, policy, B, x, out, stream):
    if kind == "scan":
        return scr.inclusive_scan(x, policy, B, out=out, stream=stream)
    if kind == "exclusive":
        return scr.exclusive_scan(x, policy, B, 0.5, out=out, stream=stream)
    if kind == "reduce":
        return scr.reduce(x, B, 0.25, out=out, stream=stream)
    return scr.reduce_policy(x, policy, B, out=out, stream=stream)


@pytest.mark.parametrize("kind,policy,B", CALLS)
def test_graph_replay(scr, kind, policy, B):
    n = 16 * 70000 + 5  # several chain tiles of 4096 carries at B = 16
    x = torch.from_numpy(W.family3(n)).to(DEV)
    out = torch.empty(1 if kind.startswith("reduce") else n, dtype=torch.float64, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run(scr, kind, policy, B, x, out, s)  # workspace and plans before the capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run(scr, kind, policy, B, x, out, s)
    for seed in (3, 4):
        x.copy_(torch.from_numpy(W.signed_pow2(n, W.seed_for(36, seed), np.float64, -20, 20)))
        g.replay()
        torch.cuda.synchronize()
        got = out.cpu().numpy().copy()
        want = run(scr, kind, policy, B, x, torch.empty_like(out), None).cpu().numpy()
        assert got.tobytes() == want.tobytes(), (kind, policy, B, seed)
