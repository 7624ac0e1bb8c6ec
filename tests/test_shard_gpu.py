"""Sequence sharding on the GPU: fd_merge_states against the oracle's merge,
and R logical ranks on one GPU (each with its own K/V shard buffers, the
exchange a plain gather of the per-shard states) against the oracle on the
whole keys.  FD++ §3 stage 2 across ranks."""
import numpy as np
import pytest
import torch

import oracle
import split_kv_flashdecoding_gb300 as fd
from split_kv_flashdecoding_gb300 import shard
from tests.parity_util import assert_within, errors
from workloads import make_small

pytestmark = pytest.mark.gpu

TIGHT = dict(max_abs=1e-4, rel_l2=1e-5, lse_abs=2e-5)


def test_merge_states_matches_oracle_merge(cuda_device):
    rng = np.random.default_rng(3)
    S, rows, D = 5, 37, 128
    o = rng.standard_normal((S, rows, D)).astype(np.float32)
    lse = (rng.standard_normal((S, rows)) * 5).astype(np.float32)
    lse[1, :10] = -np.inf          # empty shards
    lse[:, 20] = -np.inf           # a row with no keys anywhere
    o[1, :10] = 0.0
    o[:, 20] = 0.0
    om, lm = fd.merge_states(torch.from_numpy(o).to(cuda_device), torch.from_numpy(lse).to(cuda_device))
    torch.cuda.synchronize()
    finite = np.isfinite(lse)
    acc = o.transpose(1, 0, 2).reshape(-1, D).astype(np.float64)
    m = np.where(finite, lse.astype(np.float64), -1e300).T.reshape(-1)
    l = np.where(finite, 1.0, 0.0).T.reshape(-1)
    seg = np.arange(rows + 1, dtype=np.int64) * S
    o_ref, lse_ref = oracle.merge(acc, m, l, seg)
    o_ref[20] = 0.0
    lse_ref[20] = -np.inf
    err = errors(om.cpu().numpy(), lm.cpu().numpy(), o_ref, lse_ref)
    assert_within(err, max_abs=1e-5, rel_l2=1e-6, lse_abs=1e-5)
    assert float(om[20].abs().max()) == 0.0 and torch.isneginf(lm[20])


CASES = [
    ("long_one", [9000]),
    ("ragged", [3000, 0, 17, 900, 2, 4100]),
]


@pytest.mark.parametrize("R", [2, 3, 4])
@pytest.mark.parametrize("name,lengths", CASES, ids=[c[0] for c in CASES])
def test_logical_ranks_on_one_gpu(cuda_device, R, name, lengths):
    B = len(lengths)
    inp = make_small(B, 32, 8, 128, lengths, seed=R * 7 + B)
    dev = cuda_device
    q = inp["q"].to(dev)
    os_, ls_ = [], []
    for rank in range(R):
        starts, ends = shard.shard_bounds(inp["kv_indptr"], R, rank)
        rows = np.concatenate([np.arange(s, e) for s, e in zip(starts, ends)]).astype(np.int64)
        loc = shard.local_indptr(starts, ends)
        k = inp["k"][rows].to(dev)   # this rank's own shard buffers
        v = inp["v"][rows].to(dev)
        o, lse = fd.decode(q, k, v, loc, torch.from_numpy(loc).to(dev), inp["scale"])
        os_.append(o)
        ls_.append(lse)
    o_all, lse_all = torch.stack(os_), torch.stack(ls_)   # the exchange
    o, lse = fd.merge_states(o_all, lse_all)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.decode(inp["q"], inp["k"], inp["v"], inp["kv_indptr"], inp["scale"])
    err = errors(o.cpu().numpy(), lse.cpu().numpy(), o_ref.reshape(o.shape), lse_ref.reshape(lse.shape))
    assert_within(err, **TIGHT, what=f"{name} over {R} ranks")


def _free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


SHARDED_LENGTHS = [9000, 1, 0, 3000, 64]   # request 1: rank 0's shard empty; request 2: no keys


def _gpu_rank_main(rank, world, port, out_dir):
    """One rank of the shipped sequence-sharded step: its own shard buffers on
    cuda:0, fd_decode, the gloo all-gather of the states, fd_merge_states."""
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        dev = torch.device("cuda:0")
        torch.cuda.set_device(dev)
        inp = make_small(len(SHARDED_LENGTHS), 32, 8, 128, SHARDED_LENGTHS, seed=77)
        starts, ends = shard.shard_bounds(inp["kv_indptr"], world, rank)
        rows = np.concatenate([np.arange(s, e) for s, e in zip(starts, ends)]).astype(np.int64)
        loc = shard.local_indptr(starts, ends)
        k = inp["k"][rows].to(dev)
        v = inp["v"][rows].to(dev)
        o, lse = shard.decode_sequence_sharded(inp["q"].to(dev), k, v, loc,
                                               torch.from_numpy(loc).to(dev), inp["scale"])
        torch.cuda.synchronize()
        np.save(os.path.join(out_dir, f"o{rank}.npy"), o.cpu().numpy())
        np.save(os.path.join(out_dir, f"lse{rank}.npy"), lse.cpu().numpy())
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_sequence_sharded_step_two_processes(cuda_device, tmp_path):
    """shard.decode_sequence_sharded as shipped: two processes on one GPU, each
    holding half of every request's keys, exchange their states through a gloo
    all-gather (host copies; no peer memory) and merge them with
    fd_merge_states.  Both ranks get the same result, and every row matches the
    oracle on the unsharded keys (an empty shard and an empty request
    included)."""
    import torch.multiprocessing as mp
    world = 2
    mp.spawn(_gpu_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    outs = [(np.load(tmp_path / f"o{r}.npy"), np.load(tmp_path / f"lse{r}.npy")) for r in range(world)]
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
    inp = make_small(len(SHARDED_LENGTHS), 32, 8, 128, SHARDED_LENGTHS, seed=77)
    o_ref, lse_ref = oracle.decode(inp["q"], inp["k"], inp["v"], inp["kv_indptr"], inp["scale"])
    o, lse = outs[0]
    err = errors(o, lse, o_ref.reshape(o.shape), lse_ref.reshape(lse.shape))
    assert_within(err, **TIGHT, what="two processes")
    assert np.all(o[2] == 0) and np.all(np.isneginf(lse[2]))
