"""Host logic of the benchmark's multi-rank path, on CPU with two gloo ranks:
the whole-job rate is every rank's tokens over the slowest rank's step time
(replicas of the layer, weak scaling, no exchange on the data path)."""
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import sys
    import torch
    import torch.distributed as dist
    sys.path.insert(0, os.path.join(os.path.dirname(__file__), ".."))
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took (r + 1) ms per step for 8 tokens per step
        value, ms = bench.job_rate(torch, float(rank + 1), 8, world, torch.device("cpu"))
        q.put((rank, value, ms))
    finally:
        dist.destroy_process_group()


def test_job_rate_takes_the_slowest_rank_and_all_tokens():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, value, ms in got:
        assert ms == 2.0                       # max over ranks
        assert value == pytest.approx(8 * 2 / 2e-3)  # both ranks' tokens / slowest step


def test_job_rate_single_rank():
    torch = pytest.importorskip("torch")
    import sys
    sys.path.insert(0, os.path.join(os.path.dirname(__file__), ".."))
    import bench
    value, ms = bench.job_rate(torch, 4.0, 2, 1, torch.device("cpu"))
    assert ms == 4.0 and value == pytest.approx(2 / 4e-3)
