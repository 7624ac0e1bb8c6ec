"""The multi-rank logic of bench.py on two gloo ranks (CPU, no GPU).

Decode requests are independent, so under torchrun every rank processes its
own batch of the workload with no collective on the data path; the ranks
only meet at the timing barrier and the max-over-ranks reduction of the step
time, and the job's bandwidth is all ranks' bytes over the slowest rank.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    from workloads import make_inputs
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        bench.barrier(world)
        # per-rank step times: the job is as slow as its slowest rank
        local_ms = 1.0 + rank * 0.25
        ms = bench.max_over_ranks(local_ms, world, torch.device("cpu"))
        # each rank its own batch: same shapes, different values
        inp = make_inputs(0, seed=bench.rank_seed(0, rank))
        digest = float(inp["k"].float().sum())
        digests = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(digests, torch.tensor([digest], dtype=torch.float64))
        out[rank] = (ms, tuple(inp["k"].shape), [float(d) for d in digests])
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_and_shard():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert set(res) == {0, 1}
    # max over ranks
    assert res[0][0] == res[1][0] == pytest.approx(1.25)
    # same shapes, independent values per rank
    assert res[0][1] == res[1][1]
    d0, d1 = res[0][2]
    assert d0 != d1


def test_aggregate_bandwidth_is_weak_scaling():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    one = bench.aggregate_gbs(269_715_072, 1, 0.0430)
    two = bench.aggregate_gbs(269_715_072, 2, 0.0430)
    assert two == pytest.approx(2 * one)
    assert one == pytest.approx(269_715_072 / 43e-6 / 1e9)
    assert bench.rank_seed(1, 0) == 43 and bench.rank_seed(1, 1) != bench.rank_seed(1, 0)
