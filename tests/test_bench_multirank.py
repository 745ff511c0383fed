"""bench.py's multi-GPU arithmetic on CPU: independent replicas, the job's
step time is the slowest rank's and its throughput counts every rank's batch
(weak scaling).  Two gloo ranks stand in for two GPUs."""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [0.040, 0.052][rank]              # rank 1 is the slower replica
        out[rank] = bench.job_step_and_throughput(ms, world, batch=8, device="cpu")
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_sum_batches():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        for r in range(2):
            ms, value = out[r]
            assert ms == pytest.approx(0.052)
            assert value == pytest.approx(2 * 8 / 0.052e-3)


def test_single_replica_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    ms, value = bench.job_step_and_throughput(0.040, 1, batch=4)
    assert ms == 0.040 and value == pytest.approx(4 / 0.040e-3)
