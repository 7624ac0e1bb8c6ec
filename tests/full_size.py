"""The five full-size workloads and their fp64 oracle results, built once per
test session and shared by the GPU parity tests (bf16, FP8, INT4 and paged
K/V all read the same seeded keys).

The oracle runs on every (request, query head) row.  For FP8 and INT4 K/V it
dequantises a block of whole requests at a time (at most 131072 key rows, about
1 GB of fp64 per tensor) and decodes that block, so host memory stays bounded
on the largest workloads; each row's result depends only on its own request's
keys, so the blocks give the same numbers as one call over the whole batch.
"""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
from workloads import make_inputs, to_fp8, to_int4

_BLOCK_ROWS = 131072


@functools.lru_cache(maxsize=None)
def inputs(idx: int) -> dict:
    return make_inputs(idx)


@functools.lru_cache(maxsize=None)
def fp8_inputs(idx: int) -> dict:
    return to_fp8(inputs(idx))


@functools.lru_cache(maxsize=None)
def int4_inputs(idx: int) -> dict:
    return to_int4(inputs(idx))


@functools.lru_cache(maxsize=None)
def reference(idx: int):
    """Oracle (O [B*Hq, D], LSE [B*Hq]) of the bf16 workload, every row."""
    inp = inputs(idx)
    return oracle.decode(inp["q"], inp["k"], inp["v"], inp["kv_indptr"], inp["scale"])


def _request_blocks(kv_indptr):
    """[(b0, b1)] runs of whole requests holding at most _BLOCK_ROWS keys each
    (a longer request is a block of its own)."""
    ip = np.asarray(kv_indptr, dtype=np.int64)
    B = ip.size - 1
    blocks, b0 = [], 0
    while b0 < B:
        b1 = b0 + 1
        while b1 < B and ip[b1 + 1] - ip[b0] <= _BLOCK_ROWS:
            b1 += 1
        blocks.append((b0, b1))
        b0 = b1
    return blocks


def _blockwise(f, call):
    ip = np.asarray(f["kv_indptr"], dtype=np.int64)
    os_, ls_ = [], []
    for b0, b1 in _request_blocks(ip):
        r0, r1 = int(ip[b0]), int(ip[b1])
        o, lse = call(f["q"][b0:b1], r0, r1, ip[b0:b1 + 1] - r0)
        os_.append(o)
        ls_.append(lse)
    return np.concatenate(os_), np.concatenate(ls_)


@functools.lru_cache(maxsize=None)
def reference_fp8(idx: int):
    """Oracle on the exactly dequantised FP8 K/V, every row."""
    f = fp8_inputs(idx)
    return _blockwise(f, lambda q, r0, r1, ip: oracle.decode_fp8(
        q, f["k_fp8"][r0:r1], f["v_fp8"][r0:r1], f["k_scale"], f["v_scale"], ip, f["scale"]))


@functools.lru_cache(maxsize=None)
def reference_int4(idx: int):
    """Oracle on the exactly dequantised INT4 K/V, every row."""
    f = int4_inputs(idx)
    return _blockwise(f, lambda q, r0, r1, ip: oracle.decode_int4(
        q, f["k_int4"][r0:r1], f["v_int4"][r0:r1], f["k_scale_int4"][:, r0:r1],
        f["v_scale_int4"][:, r0:r1], ip, f["scale"]))


def as_rows(o: torch.Tensor, lse: torch.Tensor):
    """Device (O [B, Hq, D], LSE [B, Hq]) as host (O [B*Hq, D], LSE [B*Hq])."""
    return o.reshape(-1, o.shape[-1]).cpu().numpy(), lse.reshape(-1).cpu().numpy()
