"""bench.py's multi-rank path on the CPU: two gloo ranks on 127.0.0.1 reduce their
timings to the slowest rank's and report the whole-job (weak-scaling) value."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        total = 10.0 + 5.0 * rank                 # rank 1 is the slow one
        segs = [1.0 + rank, 7.0 - 3 * rank, 2.0]
        tot, seg = bench.max_over_ranks(total, segs, dist, "cpu")
        value = bench.whole_job_tflops(world, 4, 1e12, tot)
        out[rank] = torch.tensor([tot] + seg + [value], dtype=torch.float64)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        tot, s0, s1, s2, value = out[r].tolist()
        assert (tot, s0, s1, s2) == (15.0, 2.0, 7.0, 2.0)
        assert value == pytest.approx(2 * 4 * 1e12 / 15e-3 / 1e12)


def test_single_process_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.0, [1.0, 2.0], None, "cpu") == (3.0, [1.0, 2.0])
    assert bench.whole_job_tflops(1, 2, 1e12, 1000.0) == pytest.approx(2.0)
