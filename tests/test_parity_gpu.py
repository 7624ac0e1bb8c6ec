"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded bf16 inputs.

Method: "FlashDecoding++: sequence-dimension KV split parallelism for LLM
serving" (techknowgenie.com), §3 stage 1 (fd_decode_split), §3 stage 2
(fd_merge), and the whole step (fd_decode).
"""
import math
import zlib

import numpy as np
import pytest
import torch

import oracle
import split_kv_flashdecoding_gb300 as fd
from workloads import WORKLOADS, fp32_scale, make_small
from tests import full_size
from tests.parity_util import (assert_within, check_guards, errors, partial_segments,
                               to_device, two_stage)

pytestmark = pytest.mark.gpu

# tight bound for the small, well-conditioned cases (fp32 accumulation over <= a few
# thousand keys): a structural bug shows up far above it
TIGHT = dict(max_abs=1e-4, rel_l2=1e-5, lse_abs=2e-5)

SMALL_CASES = [
    # (name, B, Hq, Hkv, lengths)
    ("single_key", 1, 4, 4, [1]),
    ("one_tile_minus_one", 1, 8, 2, [31]),
    ("one_tile", 1, 8, 8, [32]),
    ("one_tile_plus_one", 2, 16, 2, [33, 5]),
    ("ragged_small", 4, 32, 8, [100, 1, 64, 257]),
    ("ragged_with_empty", 5, 16, 8, [0, 77, 0, 300, 1]),
    ("several_tiles", 2, 64, 8, [1000, 1537]),
    ("mha_long", 1, 8, 8, [4099]),
]


def _oracle(inp):
    return oracle.decode(inp["q"], inp["k"], inp["v"], inp["kv_indptr"], inp["scale"])


@pytest.mark.parametrize("name,B,Hq,Hkv,lengths", SMALL_CASES, ids=[c[0] for c in SMALL_CASES])
@pytest.mark.parametrize("chunk", [0, 32, 96, 1 << 20])
def test_two_stage_small(cuda_device, name, B, Hq, Hkv, lengths, chunk):
    inp = make_small(B, Hq, Hkv, 128, lengths, seed=zlib.crc32(name.encode()) % 1000 + chunk % 997)
    dev = to_device(inp, cuda_device)
    res = two_stage(dev, chunk=chunk, guard=2)
    torch.cuda.synchronize()
    assert fd.get_device_status(res["ws"]) == 0
    check_guards(res)
    o_ref, lse_ref = _oracle(inp)
    err = errors(res["o"].cpu().numpy(), res["lse"].cpu().numpy(), o_ref, lse_ref)
    assert_within(err, what=name)
    assert_within(err, **TIGHT, what=name + " (tight)")


@pytest.mark.parametrize("num_sms", [1, 3])
@pytest.mark.parametrize("name,B,Hq,Hkv,lengths", SMALL_CASES[4:7], ids=[c[0] for c in SMALL_CASES[4:7]])
def test_persistent_ctas_run_many_items(cuda_device, num_sms, name, B, Hq, Hkv, lengths):
    """A plan for 1 or 3 SMs launches 2 or 6 persistent CTAs, each running
    many items back to back (the stage ring and the item-descriptor ring wrap
    many times): the partials are bit-identical to the default grid's and the
    result matches the oracle."""
    inp = make_small(B, Hq, Hkv, 128, lengths, seed=zlib.crc32(name.encode()) % 1000 + num_sms)
    dev = to_device(inp, cuda_device)
    few = two_stage(dev, chunk=32, num_sms=num_sms, guard=2)
    full = two_stage(dev, chunk=32)
    torch.cuda.synchronize()
    assert fd.get_device_status(few["ws"]) == 0 and fd.get_device_status(full["ws"]) == 0
    check_guards(few)
    assert few["info"].num_work >= 8 * num_sms * few["info"].ctas_per_sm
    assert torch.equal(few["partial_o"], full["partial_o"])
    assert torch.equal(few["partial_lse"], full["partial_lse"])
    o_ref, lse_ref = _oracle(inp)
    err = errors(few["o"].cpu().numpy(), few["lse"].cpu().numpy(), o_ref, lse_ref)
    assert_within(err, **TIGHT, what=name)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("chunk", [32, 128, 0])
def test_split_partials_match_stage1_oracle(cuda_device, G, chunk):
    Hkv = 2
    inp = make_small(3, G * Hkv, Hkv, 128, [700, 33, 250], seed=40 + G)
    dev = to_device(inp, cuda_device)
    res = two_stage(dev, chunk=chunk)
    torch.cuda.synchronize()
    info = res["info"]
    items = fd.plan_work_items(info, inp["kv_indptr"])
    acc, m, l = oracle.split_partials(inp["q"], inp["k"], inp["v"], inp["kv_indptr"], inp["scale"],
                                      items[:, [0, 1, 3, 4]])
    On, Ln = oracle.normalised(acc, m, l)            # [n_items, G, D], [n_items, G]
    # place the oracle's partials at the documented row of (b, hq, split)
    seg = partial_segments(info, inp["kv_indptr"])
    Hq = G * Hkv
    ref_o = np.zeros((info.num_partial_rows, 128))
    ref_l = np.zeros(info.num_partial_rows)
    for i, (b, h, s, _, _) in enumerate(items):
        for g in range(G):
            row = seg[b * Hq + h * G + g] + s
            ref_o[row] = On[i, g]
            ref_l[row] = Ln[i, g]
    err = errors(res["partial_o"].cpu().numpy(), res["partial_lse"].cpu().numpy(), ref_o, ref_l)
    assert_within(err, what=f"partials G={G}")
    assert_within(err, **TIGHT, what=f"partials G={G} (tight)")


@pytest.mark.parametrize("G,lengths,chunk", [(4, [5000, 64, 3000], 64), (8, [1, 2000], 32),
                                             (1, [999] * 3, 128)])
def test_merge_matches_stage2_oracle(cuda_device, G, lengths, chunk):
    """fd_merge alone, on seeded synthetic partials (wide LSE spread)."""
    Hkv = 2
    B, Hq = len(lengths), G * Hkv
    ip = np.zeros(B + 1, dtype=np.int32)
    ip[1:] = np.cumsum(lengths)
    info = fd.plan(B, Hq, Hkv, 128, ip, chunk=chunk)
    gen = torch.Generator().manual_seed(77 + G)
    rows = info.num_partial_rows
    po = torch.randn((rows, 128), generator=gen, dtype=torch.float32)
    pl = torch.randn((rows,), generator=gen, dtype=torch.float32) * 8.0
    ip_dev = torch.from_numpy(ip).to(cuda_device)
    o = torch.empty((B, Hq, 128), dtype=torch.float32, device=cuda_device)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=cuda_device)
    ws = torch.zeros(256, dtype=torch.uint8, device=cuda_device)
    fd.merge(info, ip_dev, po.to(cuda_device), pl.to(cuda_device), o, lse, ws)
    torch.cuda.synchronize()
    seg = partial_segments(info, ip)
    o_ref, lse_ref = oracle.merge(po.numpy(), pl.numpy(), np.ones(rows), seg)
    err = errors(o.cpu().numpy(), lse.cpu().numpy(), o_ref.reshape(B, Hq, 128), lse_ref.reshape(B, Hq))
    assert_within(err, max_abs=1e-5, rel_l2=1e-6, lse_abs=1e-5, what="merge")


@pytest.mark.parametrize("idx", range(len(WORKLOADS)), ids=[w.name for w in WORKLOADS])
def test_workload_full_size(cuda_device, idx):
    """Full-size workloads in the benchmark's launch configuration (fd_decode,
    default plan): every (request, query head) row against the oracle, with
    rel-L2 over the whole O tensor; and O inside the convex hull of the
    request's V rows."""
    inp = full_size.inputs(idx)
    w = inp["workload"]
    dev = to_device(inp, cuda_device)
    B, Hq, D = w.batch, w.num_qo_heads, w.head_dim
    ws = torch.zeros(fd.workspace_bytes(B, Hq, w.num_kv_heads, D, inp["kv_indptr"]),
                     dtype=torch.uint8, device=cuda_device)
    o, lse = fd.decode(dev["q"], dev["k"], dev["v"], inp["kv_indptr"], dev["kv_indptr_dev"],
                       inp["scale"], workspace=ws)
    torch.cuda.synchronize()
    assert fd.get_device_status(ws) == 0
    o_ref, lse_ref = full_size.reference(idx)
    assert_within(errors(*full_size.as_rows(o, lse), o_ref, lse_ref), what=w.name)

    # every row: O is a convex combination of the request's V rows
    G = Hq // w.num_kv_heads
    ipl = inp["kv_indptr"].tolist()
    for b in range(B):
        vb = dev["v"][ipl[b]:ipl[b + 1]].float()             # [L, Hkv, D]
        lo = vb.amin(0).repeat_interleave(G, dim=0)            # [Hq, D]
        hi = vb.amax(0).repeat_interleave(G, dim=0)
        slack = 1e-5
        assert bool((o[b] >= lo - slack).all()) and bool((o[b] <= hi + slack).all()), b


def test_article_equivalence_check_on_gpu(cuda_device):
    """§5's setting (seed 42, B=1, H=32, D=128, S=8192, chunk 512, N(0,1)) with
    the inputs rounded to bf16: GPU split/merge vs fp64 unsplit < 1e-5."""
    g = torch.Generator().manual_seed(42)
    H, D, S = 32, 128, 8192
    q = torch.randn(1, H, D, generator=g).to(torch.bfloat16)
    k = torch.randn(S, H, D, generator=g).to(torch.bfloat16)
    v = torch.randn(S, H, D, generator=g).to(torch.bfloat16)
    inp = dict(q=q, k=k, v=v, kv_indptr=torch.tensor([0, S], dtype=torch.int32),
               scale=fp32_scale(D))
    res = two_stage(to_device(inp, cuda_device), chunk=512)
    torch.cuda.synchronize()
    o_ref, _ = _oracle(inp)
    assert np.abs(res["o"].reshape(H, D).cpu().numpy() - o_ref).max() < 1e-5


def test_stressed_outliers_small(cuda_device):
    """Score outliers (keys x16, q std 2, V uniform) on a size the oracle does
    in full: every row compared."""
    inp = make_small(4, 64, 8, 128, [2048, 300, 4096, 1], seed=5, q_std=2.0, v_dist="uniform")
    k = inp["k"].float()
    gen = torch.Generator().manual_seed(6)
    pos = torch.randperm(k.shape[0], generator=gen)[: k.shape[0] // 500]
    k[pos] *= 16
    inp["k"] = k.to(torch.bfloat16)
    res = two_stage(to_device(inp, cuda_device))
    torch.cuda.synchronize()
    o_ref, lse_ref = _oracle(inp)
    assert_within(errors(res["o"].cpu().numpy(), res["lse"].cpu().numpy(), o_ref, lse_ref),
                  what="stressed")


def test_empty_batch_and_empty_requests(cuda_device):
    inp = make_small(3, 8, 8, 128, [0, 0, 0], seed=1)
    res = two_stage(to_device(inp, cuda_device))
    torch.cuda.synchronize()
    assert res["info"].num_work == 0
    assert torch.all(res["o"] == 0) and torch.all(torch.isneginf(res["lse"]))
    # batch 0: nothing launched, nothing written
    info = fd.plan(0, 8, 8, 128, [0])
    ws = torch.zeros(256, dtype=torch.uint8, device=cuda_device)
    e = torch.empty(0, device=cuda_device)
    fd.merge(info, torch.zeros(1, dtype=torch.int32, device=cuda_device), e, e, e, e, ws)


def test_non_default_stream(cuda_device):
    inp = make_small(2, 32, 8, 128, [1500, 700], seed=9)
    dev = to_device(inp, cuda_device)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        o, lse = fd.decode(dev["q"], dev["k"], dev["v"], inp["kv_indptr"], dev["kv_indptr_dev"],
                           inp["scale"], stream=s)
    s.synchronize()
    o_ref, lse_ref = _oracle(inp)
    assert_within(errors(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref), **TIGHT)


def test_wait_timeout_reports_status_and_context_survives(cuda_device):
    """A plan whose waits give up at once: the kernel returns FD_ERR_TIMEOUT in
    the workspace status word (no trap, no hang), drains its copies, and the
    next normal call on the same context is correct."""
    inp = make_small(1, 8, 8, 128, [2000], seed=3)
    dev = to_device(inp, cuda_device)
    res = two_stage(dev, timeout_ns=0)
    assert fd.get_device_status(res["ws"]) == -5
    assert fd.get_device_status(res["ws"]) == 0      # read-and-clear
    res = two_stage(dev)
    assert fd.get_device_status(res["ws"]) == 0
    o_ref, lse_ref = _oracle(inp)
    assert_within(errors(res["o"].cpu().numpy(), res["lse"].cpu().numpy(), o_ref, lse_ref), **TIGHT)


def test_device_indptr_inconsistent_with_plan_is_flagged(cuda_device):
    """The kernels re-derive their key ranges from the device indptr; ranges or
    partial rows outside the plan are refused (status FD_ERR_DEVICE_BOUNDS) and
    nothing is written outside the buffers."""
    inp = make_small(1, 8, 8, 128, [100], seed=4)
    dev = to_device(inp, cuda_device)
    dev["kv_indptr_dev"] = torch.tensor([0, 200], dtype=torch.int32, device=cuda_device)
    res = two_stage(dev, chunk=32, guard=2)
    assert fd.get_device_status(res["ws"]) == -6
    check_guards(res)


FUSED_CASES = SMALL_CASES + [
    ("many_splits", 1, 32, 8, [5000]),
    ("ragged_many", 6, 16, 2, [3000, 0, 17, 900, 4100, 1]),
    ("g8_long", 2, 64, 8, [9000, 2500]),
]


@pytest.mark.parametrize("name,B,Hq,Hkv,lengths", FUSED_CASES, ids=[c[0] for c in FUSED_CASES])
def test_fused_decode_small(cuda_device, name, B, Hq, Hkv, lengths):
    """fd_decode (stage 2 fused into the split kernel: ticket merge, direct
    writes for single-split requests, zero rows for empty ones), called twice
    on one workspace with different values: the tickets reset themselves."""
    o_refs = []
    ws = None
    for rep in range(2):
        inp = make_small(B, Hq, Hkv, 128, lengths, seed=zlib.crc32(name.encode()) % 1000 + rep)
        dev = to_device(inp, cuda_device)
        if ws is None:
            ws = torch.zeros(fd.workspace_bytes(B, Hq, Hkv, 128, inp["kv_indptr"]),
                             dtype=torch.uint8, device=cuda_device)
        o, lse = fd.decode(dev["q"], dev["k"], dev["v"], inp["kv_indptr"], dev["kv_indptr_dev"],
                           inp["scale"], workspace=ws)
        torch.cuda.synchronize()
        assert fd.get_device_status(ws) == 0
        o_ref, lse_ref = _oracle(inp)
        err = errors(o.cpu().numpy(), lse.cpu().numpy(), o_ref.reshape(o.shape), lse_ref.reshape(lse.shape))
        assert_within(err, what=f"{name} rep {rep}")
        assert_within(err, **TIGHT, what=f"{name} rep {rep} (tight)")
        o_refs.append(o_ref)
    # the merge tickets are back to zero after each call
    assert torch.all(ws[256:256 + 4 * B * Hkv].view(torch.int32) == 0)


def test_fused_decode_after_timeout_with_rezeroed_workspace(cuda_device):
    """After a call reports an error status, zeroing the workspace makes the
    next fd_decode correct again (tickets and status start from zero)."""
    inp = make_small(1, 32, 8, 128, [6000], seed=8)
    dev = to_device(inp, cuda_device)
    res = two_stage(dev, timeout_ns=0)
    assert fd.get_device_status(res["ws"]) == -5
    ws = torch.zeros(fd.workspace_bytes(1, 32, 8, 128, inp["kv_indptr"]), dtype=torch.uint8,
                     device=cuda_device)
    o, lse = fd.decode(dev["q"], dev["k"], dev["v"], inp["kv_indptr"], dev["kv_indptr_dev"],
                       inp["scale"], workspace=ws)
    torch.cuda.synchronize()
    assert fd.get_device_status(ws) == 0
    o_ref, lse_ref = _oracle(inp)
    assert_within(errors(o.cpu().numpy(), lse.cpu().numpy(), o_ref.reshape(o.shape),
                         lse_ref.reshape(lse.shape)), **TIGHT)


def test_back_to_back_calls_match_isolated_calls(cuda_device):
    """Splits longer than the stage ring prefetch their first keys into L2 and
    let the next call launch before waiting for the previous one.  Calls on
    alternating inputs, queued back to back on one stream and sharing one
    workspace, give the bits of the same calls made one at a time."""
    B, Hq, Hkv = 1, 32, 8
    a = to_device(make_small(B, Hq, Hkv, 128, [16384], seed=91), cuda_device)
    b = to_device(make_small(B, Hq, Hkv, 128, [16384], seed=92), cuda_device)
    info = fd.plan(B, Hq, Hkv, 128, a["kv_indptr"])
    split_keys = 16384 // info.total_splits
    assert split_keys > 4 * 32, "the splits must be longer than the ring"
    ws = torch.zeros(info.workspace_bytes, dtype=torch.uint8, device=cuda_device)

    def call(x):
        return fd.decode(x["q"], x["k"], x["v"], x["kv_indptr"], x["kv_indptr_dev"], x["scale"],
                         workspace=ws)

    ref = []
    for x in (a, b):
        ref.append(call(x))
        torch.cuda.synchronize()
    outs = [call(a if i % 2 == 0 else b) for i in range(24)]
    torch.cuda.synchronize()
    assert fd.get_device_status(ws) == 0
    for i, (o, lse) in enumerate(outs):
        o_ref, lse_ref = ref[i % 2]
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref), f"call {i}"
