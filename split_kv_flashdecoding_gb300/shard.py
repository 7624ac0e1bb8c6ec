"""Sequence sharding of a decode step over ranks (one request's keys on
several GPUs).

"FlashDecoding++: sequence-dimension KV split parallelism for LLM serving"
(techknowgenie.com), §3 stage 2: the partial results of disjoint parts of the
keys merge exactly by their log-sum-exp.  Here the parts are ranks: each
request's keys [s_b, e_b) are cut into `num_shards` contiguous ranges of
nearly equal length, rank i holds the i-th range of K/V and runs fd_decode
on it, and the per-rank states (O, LSE: B * Hq * (D + 1) floats) are
all-gathered and merged with fd_merge_states.  That all-gather is the only
exchange; the attention itself never leaves a rank.
"""
from __future__ import annotations

import numpy as np

from . import decode, merge_states


def shard_bounds(kv_indptr, num_shards: int, shard: int):
    """Key rows [starts[b], ends[b]) of request b held by `shard` (int64 [B]):
    the shard-th of num_shards contiguous, nearly equal ranges of the
    request's keys (cut points s_b + L_b * i // num_shards)."""
    if not 0 <= shard < num_shards:
        raise ValueError("shard out of range")
    ip = np.asarray(kv_indptr, dtype=np.int64).reshape(-1)
    s, L = ip[:-1], ip[1:] - ip[:-1]
    return s + L * shard // num_shards, s + L * (shard + 1) // num_shards


def local_indptr(starts, ends) -> np.ndarray:
    """The shard's own ragged layout: int32 [B+1] prefix of its key counts
    (its K/V hold request b's shard at rows local[b] .. local[b+1]-1)."""
    out = np.zeros(len(starts) + 1, dtype=np.int64)
    out[1:] = np.cumsum(np.asarray(ends) - np.asarray(starts))
    return out.astype(np.int32)


def gather_states(o, lse, group=None):
    """All-gather every rank's (O, LSE) into [R, ...] tensors (rank order), on
    o's device.  NCCL gathers device tensors in place; a gloo group (CPU
    collectives) gets host copies and the result is copied back."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    staged = o.is_cuda and dist.get_backend(group) == "gloo"
    src_o = o.detach().cpu().contiguous() if staged else o.contiguous()
    src_l = lse.detach().cpu().contiguous() if staged else lse.contiguous()
    os_ = [torch.empty_like(src_o) for _ in range(world)]
    ls_ = [torch.empty_like(src_l) for _ in range(world)]
    dist.all_gather(os_, src_o, group=group)
    dist.all_gather(ls_, src_l, group=group)
    o_all, l_all = torch.stack(os_), torch.stack(ls_)
    if staged:
        o_all, l_all = o_all.to(o.device), l_all.to(lse.device)
    return o_all, l_all


def decode_sequence_sharded(q, k_shard, v_shard, local_indptr_host, local_indptr_dev, scale: float, *,
                            group=None, workspace=None, stream=None):
    """One decode step with the keys sharded over the ranks of `group`: fd_decode
    on this rank's shard, all-gather of the states, fd_merge_states.  Every
    rank passes the same q and returns the full (O, LSE)."""
    o, lse = decode(q, k_shard, v_shard, local_indptr_host, local_indptr_dev, scale,
                    workspace=workspace, stream=stream)
    o_all, lse_all = gather_states(o, lse, group)
    return merge_states(o_all, lse_all, stream=stream)
