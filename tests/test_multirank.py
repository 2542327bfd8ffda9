"""The replica path of bench.py on two gloo ranks (CPU, no GPU): the job's
time is its slowest rank's, and its throughput counts every rank's bytes.
bench.py runs one independent replica per GPU (the rows do not exchange
data), so these reductions are its only cross-rank steps."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        slowest = bench.max_over_ranks(times[rank], dist, "cpu")
        dist.barrier()
        value = bench.job_gbs(4 * 10**9, 5, world, slowest)
        q.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def _run(times):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, len(times), port, times, q))
          for r in range(len(times))]
    for p in ps:
        p.start()
    out = {}
    for _ in ps:
        r, slowest, value = q.get(timeout=120)
        out[r] = (slowest, value)
    for p in ps:
        p.join(60)
        assert p.exitcode == 0
    return out


def test_two_ranks_take_the_slowest_time():
    out = _run([2.0, 2.5])
    assert out[0] == out[1]
    slowest, value = out[0]
    assert slowest == 2.5
    assert value == pytest.approx(4 * 5 * 2 / 2.5)  # both ranks' bytes over the max time


def test_single_process_passes_through():
    import bench
    assert bench.max_over_ranks(1.25, None, "cpu") == 1.25
    assert bench.job_gbs(10**9, 4, 1, 2.0) == pytest.approx(2.0)
