"""Calls from several host threads at once, each thread on a stream of its own
(and so with a workspace of its own): every result has the bits that the same
call returns when it runs alone. This covers the library's host state that
threads share (launch bookkeeping, the lock around the host-copy streams, the
fused carry pass's per-device grid limit, filled by whichever call comes
first) and cooperative launches of the fused carry pass beside other kernels
on other streams."""
import threading

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
THREADS = 4
ROUNDS = 3


@pytest.fixture(scope="module")
def scr():
    import scan_canonical_reduce_gb300 as m
    return m


def cases(scr):
    """(name, call) pairs; each call takes its inputs from the closure and
    returns a tensor (device or host)."""
    n = (1 << 22) + 37
    x = torch.from_numpy(W.family3(n)).to(DEV)
    xf = torch.from_numpy(W.family2(n, np.float32)).to(DEV)
    xh = torch.from_numpy(W.family3((1 << 21) + 5)).pin_memory()
    cols = torch.from_numpy(W.family5(90, 20000)).to(DEV).view(90, 20000)
    torch.cuda.synchronize()
    return [
        ("reduce_L16", lambda: scr.reduce(x, 16, 0.5)),
        ("reduce_f32_L1024", lambda: scr.reduce(xf, 1024, 0.0)),
        ("iterated_pairwise", lambda: scr.inclusive_scan(x, "iterated_pairwise", 1)),
        ("pairwise", lambda: scr.inclusive_scan(x, "pairwise", 1)),
        ("block_dyadic16", lambda: scr.inclusive_scan(x, "block_dyadic", 16)),  # fused pass
        ("block_dyadic256", lambda: scr.inclusive_scan(x, "block_dyadic", 256)),
        ("left_fold", lambda: scr.inclusive_scan(x, "left_fold", 1)),
        ("block_dyadic16_f32", lambda: scr.inclusive_scan(xf, "block_dyadic", 16)),
        ("exclusive_pairwise", lambda: scr.exclusive_scan(x, "pairwise", 1, 0.25)),
        ("colscan_bd16", lambda: scr.inclusive_scan_batched(cols, "block_dyadic", 16, dim=0)),
        ("host_scan_bd16", lambda: scr.inclusive_scan(xh, "block_dyadic", 16)),
        ("host_reduce", lambda: scr.reduce(xh, 128, 0.0)),
    ]


def as_bytes(t):
    return t.cpu().numpy().tobytes()


def test_concurrent_threads_same_bits(scr):
    calls = cases(scr)
    want = {}
    for name, fn in calls:
        want[name] = as_bytes(fn())
    torch.cuda.synchronize()
    launched = scr.launch_count()

    got = [dict() for _ in range(THREADS)]
    errors = []
    start = threading.Barrier(THREADS)

    def worker(k):
        try:
            s = torch.cuda.Stream(device=DEV)
            order = calls[k:] + calls[:k]  # every thread in another order
            start.wait()
            for r in range(ROUNDS):
                with torch.cuda.stream(s):
                    outs = [(name, fn()) for name, fn in order]
                scr.sync_status(stream=s)  # no wait of this thread's calls timed out
                for name, o in outs:
                    got[k][name, r] = as_bytes(o)
        except Exception as e:  # reported by the main thread
            errors.append((k, repr(e)))

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(THREADS)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert scr.launch_count() > launched
    differ = [(k, key) for k in range(THREADS) for key, b in got[k].items()
              if b != want[key[0]]]
    assert not differ, differ
    assert all(len(g) == len(calls) * ROUNDS for g in got)
