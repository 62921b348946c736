"""Multi-rank plumbing of bench.py on CPU: two gloo ranks on 127.0.0.1.

The timed path shards by sequence with no data exchange; the only
collective is the max over ranks of the measured time (whole-job throughput
= all ranks' work over the slowest rank's time).  These tests run that
plumbing with world size 2 and no GPU."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    # rank r took (r + 1) seconds for 4 steps of 1e12 flops each
    value, ms = bench.aggregate(1e12, float(rank + 1), 4, w)
    mx = bench.max_over_ranks(float(rank * 10), w)
    # the reference arm does its work on rank 0 only; other ranks return at once
    ret = bench.run_reference(None, w, r) if r != 0 else 0
    out[rank] = (value, ms, mx, ret)
    dist.destroy_process_group()


def test_two_rank_aggregate_takes_slowest_rank():
    world, port = 2, _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        value, ms, mx, ret = out[r]
        # slowest rank: 2 s for 4 steps; whole job: 2 ranks x 4 steps x 1e12 flops
        assert ms == pytest.approx(500.0)
        assert value == pytest.approx(2 * 4 * 1e12 / 2.0 / 1e12)
        assert mx == pytest.approx(10.0)
        assert ret == 0
