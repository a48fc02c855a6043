"""The multi-rank (torchrun) host logic of bench.py on CPU with the gloo
backend, world size 2: each rank routes its own tokens (distinct seeds), the
job time is the max over ranks, throughput scales with the number of ranks
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
        X, _, _ = mi.make_route_inputs(64, 32, 8, seed=rank)  # the seed bench.py gives each rank
        digest = float(X.float().sum())
        digests = [None] * world
        dist.all_gather_object(digests, digest)
        q.put((rank, total, bench.weak_scaling_tokens_per_s(world, 2048, 100, total), digests))
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
    for rank, total, value, digests in results:
        assert total == 25.0                              # max over ranks
        assert value == pytest.approx(2 * 2048 * 100 / 0.025)
        assert digests[0] != digests[1]                   # different tokens per rank


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
