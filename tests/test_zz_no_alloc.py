"""fd_decode_static_workspace: decode attention for callers that cannot allocate.

Callers such as an inference-engine plugin in its enqueue step, or a runtime
whose device memory is planned up front and owned by someone else, must not
call cudaMalloc where they run attention.  This entry point keeps its scratch
in a fixed 16 MiB device array inside the library, so they pass only inputs
and outputs.  The test calls it through the C ABI several times in a row and
compares every result with the fp64 oracle at the parity tolerances of the
other GPU tests.  The array keeps each call's contents: the pair of calls with
different batch shapes is chosen so that the second call's merge tickets lie
where the first call left partial log-sum-exp values, which only the entry
point's own clearing of the header and tickets turns back into zeros.  The file
sorts last, so pytest collects it after every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
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


def _check_against_oracle(dev, inp, what):
    o, lse = _static_call(dev, inp)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.decode(inp["q"], inp["k"], inp["v"], inp["kv_indptr"], inp["scale"])
    err = errors(o.cpu().numpy(), lse.cpu().numpy(), o_ref.reshape(o.shape), lse_ref.reshape(lse.shape))
    assert_within(err, what=what)


def test_static_workspace_matches_oracle_twice_in_a_row(cuda_device):
    for rep, (B, Hq, Hkv, lengths) in enumerate(CASES):
        inp = make_small(B, Hq, Hkv, 128, lengths, seed=900 + rep)
        _check_against_oracle(to_device(inp, cuda_device), inp, f"call {rep}")


def _regions(B, Hkv, lengths, Hq):
    """Byte ranges [tickets), [partial LSE) of a plan in the scratch layout
    fd_decode uses: 256-byte header, tickets, partial LSE, partial O."""
    ip = np.zeros(B + 1, dtype=np.int32)
    ip[1:] = np.cumsum(lengths)
    info = fd.plan(B, Hq, Hkv, 128, ip)
    t_end = 256 + -(-B * Hkv * 4 // 256) * 256
    return info, (256, 256 + B * Hkv * 4), (t_end, t_end + 4 * info.num_partial_rows)


def test_static_workspace_clears_tickets_left_dirty_by_a_previous_call(cuda_device):
    """Call 1 (2 requests, many splits) writes partial LSE values at the bytes
    where call 2 (64 requests, requests 10-17 split nine ways) keeps the
    tickets of those long requests.  Without the entry point's clearing, their
    merges would never run and their rows would keep the NaN the output starts
    with."""
    first = (2, 32, 8, [9000, 300])
    second_len = [300] * 64
    for b in range(10, 18):
        second_len[b] = 20000
    second = (64, 32, 8, second_len)
    _, _, lse1 = _regions(first[0], first[2], first[3], first[1])
    info2, _, _ = _regions(second[0], second[2], second[3], second[1])
    multi = [b for b in range(64) if -(-second_len[b] // info2.chunk) > 1]
    assert multi, "call 2 needs requests with several splits (merge tickets in use)"
    dirty = [256 + 4 * (b * 8 + h) for b in multi for h in range(8)
             if lse1[0] <= 256 + 4 * (b * 8 + h) < lse1[1]]
    assert dirty, "call 2's tickets must lie in call 1's partial LSE bytes"
    for rep, (B, Hq, Hkv, lengths) in enumerate([first, second, first]):
        inp = make_small(B, Hq, Hkv, 128, lengths, seed=950 + rep)
        _check_against_oracle(to_device(inp, cuda_device), inp, f"call {rep} (B={B})")


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
