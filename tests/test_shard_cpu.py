"""Sequence sharding, host side: the shard bounds partition every request's
keys, and two gloo ranks exchange and merge their shards' states into the
unsharded result (FD++ §3 stage 2 across ranks).  The per-shard attention and
the merge are the fp64 oracle's here; the GPU tests run the library's."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from split_kv_flashdecoding_gb300 import shard

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("seed", range(4))
def test_shard_bounds_partition_each_request(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 20))
    lengths = rng.integers(0, 50, size=B)
    ip = np.concatenate([[0], np.cumsum(lengths)])
    for R in (1, 2, 3, 8):
        parts = [shard.shard_bounds(ip, R, i) for i in range(R)]
        for b in range(B):
            pieces = [(s[b], e[b]) for s, e in parts]
            assert pieces[0][0] == ip[b] and pieces[-1][1] == ip[b + 1]
            for (s0, e0), (s1, e1) in zip(pieces[:-1], pieces[1:]):
                assert e0 == s1 and s0 <= e0
            sizes = [e - s for s, e in pieces]
            assert max(sizes) - min(sizes) <= 1
        loc = shard.local_indptr(*parts[0])
        assert loc[0] == 0 and loc[-1] == sum(e - s for s, e in zip(*parts[0]))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import oracle
    from workloads import make_small
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        inp = make_small(3, 8, 2, 128, [50, 0, 7], seed=21)   # every rank the same step
        starts, ends = shard.shard_bounds(inp["kv_indptr"], world, rank)
        rows = np.concatenate([np.arange(s, e) for s, e in zip(starts, ends)]).astype(np.int64)
        k, v = inp["k"][rows], inp["v"][rows]
        o, lse = oracle.decode(inp["q"], k, v, shard.local_indptr(starts, ends), inp["scale"])
        o_all, lse_all = shard.gather_states(torch.from_numpy(o), torch.from_numpy(lse))
        # merge the gathered states: one segment of `world` states per row
        n_rows = lse.size
        acc = o_all.permute(1, 0, 2).reshape(-1, o.shape[1]).numpy()
        m = lse_all.permute(1, 0).reshape(-1).numpy()
        seg = np.arange(n_rows + 1, dtype=np.int64) * world
        finite = np.isfinite(m)
        m_safe = np.where(finite, m, -1e300)   # an empty shard's state weighs nothing
        om, lm = oracle.merge(acc, m_safe, np.where(finite, 1.0, 0.0), seg)
        o_ref, lse_ref = oracle.decode(inp["q"], inp["k"], inp["v"], inp["kv_indptr"], inp["scale"])
        out[rank] = (float(np.nanmax(np.abs(om - o_ref))),
                     float(np.nanmax(np.abs(lm[np.isfinite(lse_ref)] - lse_ref[np.isfinite(lse_ref)]))),
                     bool(np.all(np.isneginf(lse_ref) == (lm < -1e299))))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_exchange_and_merge():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert set(res) == {0, 1}
    for rank in (0, 1):
        max_o, max_lse, empty_ok = res[rank]
        assert max_o < 1e-12 and max_lse < 1e-12 and empty_ok
