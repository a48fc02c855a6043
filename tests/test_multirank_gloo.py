"""The multi-rank (torchrun) host logic of bench.py on CPU with the gloo
backend, world size 2: each rank routes its own tokens (distinct seeds)
against one shared gate weight, the job time is the max over ranks, throughput scales with the number of ranks
(weak scaling), and the load statistics are taken on the expert counts of all
ranks added up.  No GPU and no collective on the data path."""
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


def _rank_main(rank, world, port, q):
    import bench
    import moe_inputs as mi
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [10.0, 25.0][rank]                     # rank 1 is the slow one
        total = bench.max_over_ranks(local_ms, dist, "cpu")
        # the inputs bench.py gives each rank: its own tokens, the shared gate
        X, W, bias = mi.make_replica_inputs(mi.Workload("t", 64, 32, 8, 2, skew=True), rank)
        mine = (X.view(torch.int16).numpy().tobytes(), W.view(torch.int16).numpy().tobytes(),
                bias.numpy().tobytes())
        every = [None] * world
        dist.all_gather_object(every, mine)
        q.put((rank, total, bench.weak_scaling_tokens_per_s(world, 2048, 100, total), every))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_max_time_and_own_tokens():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, total, value, every in results:
        assert total == 25.0                              # max over ranks
        assert value == pytest.approx(2 * 2048 * 100 / 0.025)
        assert every[0][0] != every[1][0]                 # different tokens per rank
        assert every[0][1] == every[1][1]                 # one gate weight, bit for bit
        assert every[0][2] == every[1][2]                 # and one bias


def test_replica_inputs_of_rank_zero_are_the_workloads_own():
    import moe_inputs as mi
    w = mi.Workload("t", 48, 16, 8, 2)
    X0, W0, _ = mi.make_workload_inputs(w)
    X, W, _ = mi.make_replica_inputs(w, 0)
    assert torch.equal(X.view(torch.int16), X0.view(torch.int16))
    assert torch.equal(W.view(torch.int16), W0.view(torch.int16))
    X1, W1, _ = mi.make_replica_inputs(w, 1)
    assert torch.equal(W1.view(torch.int16), W0.view(torch.int16))
    assert not torch.equal(X1.view(torch.int16), X0.view(torch.int16))


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.weak_scaling_tokens_per_s(1, 2048, 10, 1.0) == pytest.approx(2048 * 10 / 1e-3)
    c = torch.tensor([3, 0, 5], dtype=torch.int32)
    assert bench.sum_over_ranks(c) is c


def _counts_main(rank, world, port, q):
    import numpy as np
    import bench
    import moe_inputs as mi
    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        X, W, _ = mi.make_route_inputs(256, 64, 16, seed=rank)
        idx, _ = oracle.route(mi.bf16_bits(X), mi.bf16_bits(W), None, 2)
        counts, _, _, _ = oracle.dispatch(idx, 16)
        job = bench.sum_over_ranks(torch.from_numpy(np.asarray(counts, dtype=np.int32)), dist)
        q.put((rank, np.asarray(counts).tolist(), job.tolist()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_add_up_their_expert_counts():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_counts_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    local = [r[1] for r in results]
    expect = [a + b for a, b in zip(*local)]
    for _, _, job in results:
        assert job == expect                              # every rank holds the job-wide histogram
    assert sum(expect) == world * 256 * 2                 # token conservation over the job
