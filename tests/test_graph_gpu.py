"""fd_decode_graph on the GPU: the split plan derived on the device, captured
in a CUDA graph and replayed with new lengths, against the fp64 oracle.
FD++ §6 (decode steps run as CUDA graphs with a fixed batch)."""
import numpy as np
import pytest
import torch

import oracle
import split_kv_flashdecoding_gb300 as fd
from tests.parity_util import assert_within, errors
from workloads import make_small

pytestmark = pytest.mark.gpu

TIGHT = dict(max_abs=1e-4, rel_l2=1e-5, lse_abs=2e-5)
B, HQ, HKV, D, CAP = 6, 32, 8, 128, 24000


def _buffers(dev):
    return dict(q=torch.empty((B, HQ, D), dtype=torch.bfloat16, device=dev),
                k=torch.empty((CAP, HKV, D), dtype=torch.bfloat16, device=dev),
                v=torch.empty((CAP, HKV, D), dtype=torch.bfloat16, device=dev),
                ip=torch.zeros(B + 1, dtype=torch.int32, device=dev),
                o=torch.empty((B, HQ, D), dtype=torch.float32, device=dev),
                lse=torch.empty((B, HQ), dtype=torch.float32, device=dev))


def _load(buf, inp):
    T = int(inp["kv_indptr"][-1])
    buf["q"].copy_(inp["q"])
    buf["k"][:T].copy_(inp["k"])
    buf["v"][:T].copy_(inp["v"])
    buf["ip"].copy_(inp["kv_indptr"])


def _check(buf, inp, what):
    o_ref, lse_ref = oracle.decode(inp["q"], inp["k"], inp["v"], inp["kv_indptr"], inp["scale"])
    err = errors(buf["o"].cpu().numpy(), buf["lse"].cpu().numpy(), o_ref.reshape(B, HQ, D),
                 lse_ref.reshape(B, HQ))
    assert_within(err, **TIGHT, what=what)


LENGTHS = [
    [3000, 0, 17, 900, 4100, 1],        # ragged with an empty request
    [0, 0, 0, 0, 0, 0],                 # nothing at all: every row 0 / -inf
    [4000, 4000, 4000, 4000, 4000, 4000],   # the capacity exactly
    [129, 1, 23999 - 130, 0, 0, 0],      # one long request, most of the capacity
]


def test_device_plan_without_capture(cuda_device):
    info = fd.plan_graph(B, HQ, HKV, D, CAP)
    buf = _buffers(cuda_device)
    ws = torch.zeros(info.workspace_bytes, dtype=torch.uint8, device=cuda_device)
    for i, lengths in enumerate(LENGTHS):
        inp = make_small(B, HQ, HKV, D, lengths, seed=100 + i)
        _load(buf, inp)
        fd.decode_graph(info, buf["q"], buf["k"], buf["v"], buf["ip"], inp["scale"], buf["o"],
                        buf["lse"], ws)
        torch.cuda.synchronize()
        assert fd.get_device_status(ws) == 0
        _check(buf, inp, f"lengths {lengths}")


def test_captured_graph_replays_with_new_lengths(cuda_device):
    info = fd.plan_graph(B, HQ, HKV, D, CAP)
    buf = _buffers(cuda_device)
    ws = torch.zeros(info.workspace_bytes, dtype=torch.uint8, device=cuda_device)
    scale = make_small(1, 1, 1, D, [1])["scale"]
    _load(buf, make_small(B, HQ, HKV, D, LENGTHS[0], seed=1))
    stream = torch.cuda.Stream(cuda_device)
    stream.wait_stream(torch.cuda.current_stream(cuda_device))
    with torch.cuda.stream(stream):   # one call before capture
        fd.decode_graph(info, buf["q"], buf["k"], buf["v"], buf["ip"], scale, buf["o"], buf["lse"],
                        ws, stream=stream)
    torch.cuda.current_stream(cuda_device).wait_stream(stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        fd.decode_graph(info, buf["q"], buf["k"], buf["v"], buf["ip"], scale, buf["o"], buf["lse"],
                        ws, stream=torch.cuda.current_stream(cuda_device))
    for i, lengths in enumerate(LENGTHS * 2):
        inp = make_small(B, HQ, HKV, D, lengths, seed=200 + i)
        _load(buf, inp)
        graph.replay()
        torch.cuda.synchronize()
        assert fd.get_device_status(ws) == 0
        _check(buf, inp, f"replay {i}, lengths {lengths}")


def test_indptr_beyond_capacity_is_flagged(cuda_device):
    info = fd.plan_graph(2, 8, 8, D, 100)
    dev = cuda_device
    q = torch.zeros((2, 8, D), dtype=torch.bfloat16, device=dev)
    k = torch.zeros((100, 8, D), dtype=torch.bfloat16, device=dev)
    v = torch.zeros_like(k)
    ip = torch.tensor([0, 60, 160], dtype=torch.int32, device=dev)   # 160 > the 100 rows planned
    o = torch.empty((2, 8, D), dtype=torch.float32, device=dev)
    lse = torch.empty((2, 8), dtype=torch.float32, device=dev)
    ws = torch.zeros(info.workspace_bytes, dtype=torch.uint8, device=dev)
    fd.decode_graph(info, q, k, v, ip, 0.1, o, lse, ws)
    torch.cuda.synchronize()
    assert fd.get_device_status(ws) == -6


@pytest.mark.parametrize("lengths", [[1000, 0, 1999], [0, 0, 0], [3000, 0, 0], [1, 1, 1]])
def test_device_plan_in_one_wave(cuda_device, lengths):
    """A capacity whose plan fits one wave of CTAs runs the one-item-per-CTA
    kernel under the device-side plan (CTAs past the batch's items exit), also
    captured in a CUDA graph."""
    b, cap = 3, 3000
    info = fd.plan_graph(b, 16, 8, D, cap)
    assert info.num_work <= info.num_sms * info.ctas_per_sm, "the plan must fit one wave"
    dev = cuda_device
    inp = make_small(b, 16, 8, D, lengths, seed=sum(lengths) % 997)
    T = int(inp["kv_indptr"][-1])
    q = inp["q"].to(dev)
    k = torch.zeros((cap, 8, D), dtype=torch.bfloat16, device=dev)
    v = torch.zeros_like(k)
    k[:T].copy_(inp["k"])
    v[:T].copy_(inp["v"])
    ip = inp["kv_indptr"].to(dev)
    o = torch.empty((b, 16, D), dtype=torch.float32, device=dev)
    lse = torch.empty((b, 16), dtype=torch.float32, device=dev)
    ws = torch.zeros(info.workspace_bytes, dtype=torch.uint8, device=dev)
    o_ref, lse_ref = oracle.decode(inp["q"], inp["k"], inp["v"], inp["kv_indptr"], inp["scale"])
    fd.decode_graph(info, q, k, v, ip, inp["scale"], o, lse, ws)
    torch.cuda.synchronize()
    assert fd.get_device_status(ws) == 0
    err = errors(o.cpu().numpy(), lse.cpu().numpy(), o_ref.reshape(o.shape), lse_ref.reshape(lse.shape))
    assert_within(err, **TIGHT, what=f"{lengths}")
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    g = torch.cuda.CUDAGraph()
    o.fill_(7.0)
    with torch.cuda.graph(g, stream=s):
        fd.decode_graph(info, q, k, v, ip, inp["scale"], o, lse, ws,
                        stream=torch.cuda.current_stream(dev))
    g.replay()
    torch.cuda.synchronize()
    err = errors(o.cpu().numpy(), lse.cpu().numpy(), o_ref.reshape(o.shape), lse_ref.reshape(lse.shape))
    assert_within(err, **TIGHT, what=f"{lengths} (graph)")
