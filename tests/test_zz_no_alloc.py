"""fd_decode_static_workspace: decode attention for callers that cannot allocate.

Callers such as an inference-engine plugin in its enqueue step, or a runtime
whose device memory is planned up front and owned by someone else, must not
call cudaMalloc where they run attention.  This entry point keeps its scratch
in a fixed 16 MiB device array inside the library, so they pass only inputs
and outputs.  The test calls it through the C ABI twice in a row (the array
keeps the previous call's contents, which must not leak into the next) and
compares each result with fd_decode run on a caller-owned workspace, within
the parity tolerances of the other GPU tests.  It sits in a file of its own
that pytest collects last.
"""
import ctypes

import numpy as np
import pytest
import torch

import split_kv_flashdecoding_gb300 as fd
from tests.parity_util import assert_within, errors, to_device
from workloads import make_small

pytestmark = pytest.mark.gpu

CASES = [(3, 32, 8, [5000, 17, 2100]), (2, 64, 8, [9000, 300])]


def _static_call(dev, inp):
    """fd_decode_static_workspace straight through ctypes."""
    B, Hq, D = dev["q"].shape
    Hkv = dev["k"].shape[1]
    ip = np.ascontiguousarray(inp["kv_indptr"].numpy().astype(np.int32))
    o = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device=dev["q"].device)
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=dev["q"].device)
    P = ctypes.c_void_p
    rc = fd.lib().fd_decode_static_workspace(
        B, Hq, Hkv, D, ip.ctypes.data_as(P), P(dev["kv_indptr_dev"].data_ptr()),
        P(dev["q"].data_ptr()), P(dev["k"].data_ptr()), P(dev["v"].data_ptr()),
        ctypes.c_float(inp["scale"]), P(o.data_ptr()), P(lse.data_ptr()),
        P(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, fd.status_string(rc)
    return o, lse


def test_static_workspace_matches_fd_decode_twice_in_a_row(cuda_device):
    for rep, (B, Hq, Hkv, lengths) in enumerate(CASES):
        inp = make_small(B, Hq, Hkv, 128, lengths, seed=900 + rep)
        dev = to_device(inp, cuda_device)
        ws = torch.zeros(fd.workspace_bytes(B, Hq, Hkv, 128, inp["kv_indptr"]), dtype=torch.uint8,
                         device=cuda_device)
        o_ref, lse_ref = fd.decode(dev["q"], dev["k"], dev["v"], inp["kv_indptr"],
                                   dev["kv_indptr_dev"], inp["scale"], workspace=ws)
        o, lse = _static_call(dev, inp)
        torch.cuda.synchronize()
        err = errors(o.cpu().numpy(), lse.cpu().numpy(), o_ref.cpu().double().numpy(),
                     lse_ref.cpu().double().numpy())
        assert_within(err, what=f"call {rep}")


def test_static_workspace_rejects_plans_beyond_its_size(cuda_device):
    B, Hq, Hkv = 1024, 64, 8          # 65536 (request, head) rows of partials: ~33 MiB
    ip = np.zeros(B + 1, dtype=np.int32)
    ip[1:] = np.cumsum([2048] * B)
    need = fd.plan(B, Hq, Hkv, 128, ip).workspace_bytes
    assert need > 16 << 20
    P = ctypes.c_void_p
    rc = fd.lib().fd_decode_static_workspace(B, Hq, Hkv, 128, ip.ctypes.data_as(P), None, None,
                                             None, None, ctypes.c_float(0.1), None, None, None)
    assert rc == -3   # FD_ERR_WORKSPACE, returned before any device work
