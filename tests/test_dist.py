"""The multi-replica bench logic on two gloo ranks (CPU): the step time is the slowest rank's and the
whole-job value counts every rank's FLOPs (weak scaling, no collective on the data path)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.reduce_max(1.0 + rank, world, torch.device("cpu"))   # rank 1 is the slow replica
    value = bench.weak_scaling_tflops(2.0e12, ms, world)
    dist.barrier()
    q.put((rank, ms, value))
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in out:
        assert ms == pytest.approx(2.0)                      # max over ranks
        assert value == pytest.approx(2 * 2.0e12 / 2.0e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.reduce_max(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.weak_scaling_tflops(1.0e12, 1.0, 1) == pytest.approx(1.0e3)
