"""Data parallelism on two gloo ranks (CPU): the bench's step time is the slowest rank's and the whole-job value
counts every rank's FLOPs (weak scaling); token shards tile the batch, and the weight-gradient all-reduce of the
shards gives the whole batch's dW1 and dW2 (checked against the oracle)."""
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


def _dp_worker(rank, world, port, q):
    """One data-parallel rank on the CPU: its token shard through the oracle, then the weight-gradient all-reduce."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from fine_grained_mixture_gb300 import dp, synth
        from oracle import moe_oracle as orc

        w = synth.custom(T=97, d=16, n=8, E=5, K=2)      # 97 tokens: the two shards differ in size
        inp = synth.make_inputs(w, 3)
        X, W1, W2, dO = (inp[k].double().numpy() for k in ("X", "W1", "W2", "dO"))
        z = inp["logits"].numpy()
        a, b = dp.token_shard(w.T, rank, world)
        ref = orc.route(z[a:b], w.K, "tc")
        fwd, bwd = orc.layer(X[a:b], W1, W2, dO[a:b], ref)
        dW1 = torch.from_numpy(bwd["dW1"].copy())
        dW2 = torch.from_numpy(bwd["dW2"].copy())
        dp.allreduce_weight_grads(dW1, dW2)
        q.put((rank, a, b, dW1.numpy(), dW2.numpy(), fwd["O"], bwd["dX"]))
    finally:
        dist.destroy_process_group()


def test_data_parallel_weight_gradients_equal_the_whole_batch():
    """Two gloo ranks each run their token shard and sum dW1/dW2 with the all-reduce: every rank then holds the
    weight gradients of the whole batch, and each shard's O and dX are the whole batch's rows (token choice routes
    each token on its own logits)."""
    import numpy as np

    from fine_grained_mixture_gb300 import synth
    from oracle import moe_oracle as orc

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_dp_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted((q.get(timeout=120) for _ in procs), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w = synth.custom(T=97, d=16, n=8, E=5, K=2)
    inp = synth.make_inputs(w, 3)
    X, W1, W2, dO = (inp[k].double().numpy() for k in ("X", "W1", "W2", "dO"))
    fwd, bwd = orc.layer(X, W1, W2, dO, orc.route(inp["logits"].numpy(), w.K, "tc"))
    assert [(a, b) for _, a, b, *_ in out] == [(0, 48), (48, 97)]
    for _, a, b, dW1, dW2, O, dX in out:
        np.testing.assert_allclose(dW1, bwd["dW1"], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(dW2, bwd["dW2"], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(O, fwd["O"][a:b], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(dX, bwd["dX"][a:b], rtol=1e-12, atol=1e-14)


def test_token_shards_tile_the_batch():
    from fine_grained_mixture_gb300 import dp
    for T in (0, 1, 7, 97, 24576):
        for world in (1, 2, 3, 8):
            bounds = [dp.token_shard(T, r, world) for r in range(world)]
            assert bounds[0][0] == 0 and bounds[-1][1] == T
            assert all(bounds[i][1] == bounds[i + 1][0] for i in range(world - 1))
            sizes = [b - a for a, b in bounds]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        dp.token_shard(10, 2, 2)


def test_allreduce_without_a_process_group_is_a_no_op():
    from fine_grained_mixture_gb300 import dp
    a, b = torch.ones(3), torch.full((2,), 2.0)
    assert dp.allreduce_weight_grads(a, b) is None
    assert dp.allreduce_weight_grads(a, b, async_op=True) == []
    assert a.tolist() == [1.0, 1.0, 1.0] and b.tolist() == [2.0, 2.0]
