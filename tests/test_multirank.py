"""Host-side multi-rank logic of bench.py on CPU (gloo, world size 2).

With N GPUs every rank runs an independent replica of the step; the job's
time is the max over ranks and the value counts every rank's parameters.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mproc


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    seconds = 1.0 + rank  # rank 1 is the slow one
    mx = bench.max_over_ranks(seconds, w, torch.device("cpu"))
    val = bench.whole_job_value(1000, w, 10, mx)
    q.put((rank, mx, val))
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_gloo():
    world = 2
    port = _free_port()
    ctx = mproc.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, val in out:
        assert mx == 2.0  # the slowest rank sets the time
        assert val == pytest.approx(1000 * 2 * 10 / 2.0 / 1e9)
