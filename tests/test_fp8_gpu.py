"""FP8 (E4M3) KV on the GPU (fd_decode_fp8, fd_decode_paged_fp8) against the
fp64 oracle on the exactly dequantised K/V (oracle.decode_fp8).

FD++ §4 (quantisation-friendly fusion): the quantised K and V are read as they
are and dequantised in registers.  The reference result is attention over the
dequantised values; the tolerances are those of the bf16 path.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
import split_kv_flashdecoding_gb300 as fd
from tests import full_size
from tests.parity_util import assert_within, errors
from workloads import WORKLOADS, make_small, to_fp8, to_paged

pytestmark = pytest.mark.gpu

TIGHT = dict(max_abs=1e-4, rel_l2=1e-5, lse_abs=2e-5)

CASES = [
    # (name, B, Hq, Hkv, lengths)
    ("single_key", 1, 4, 4, [1]),
    ("one_tile_minus_one", 1, 8, 2, [31]),
    ("ragged_with_empty", 5, 16, 8, [0, 77, 0, 300, 1]),
    ("several_tiles_g8", 2, 64, 8, [1000, 1537]),
    ("mha_long", 1, 8, 8, [4099]),
    ("many_splits", 1, 32, 8, [5000]),          # one wave
    ("ragged_many", 6, 16, 2, [3000, 0, 17, 900, 4100, 1]),
    ("two_requests_g8", 2, 64, 8, [9000, 2500]),  # one wave on 152 SMs (296 items)
    # more items than one wave (600 on 152 SMs): the persistent kernel, in the
    # row form (G = 8) and the column form (G <= 4: keys and dims in the MMA rows)
    ("multi_wave_g8", 3, 64, 8, [16000, 16000, 3000]),
    ("multi_wave_g4", 3, 32, 8, [16000, 16000, 3000]),
    ("multi_wave_g2", 3, 16, 8, [16000, 16001, 2999]),
    ("multi_wave_g1", 3, 8, 8, [16001, 15999, 3000]),
]


def _run(f, dev, ws=None):
    d = {k: f[k].to(dev) for k in ("q", "k_fp8", "v_fp8", "k_scale", "v_scale")}
    ip_dev = f["kv_indptr"].to(dev)
    return fd.decode_fp8(d["q"], d["k_fp8"], d["v_fp8"], d["k_scale"], d["v_scale"], f["kv_indptr"],
                         ip_dev, f["scale"], workspace=ws)


@pytest.mark.parametrize("name,B,Hq,Hkv,lengths", CASES, ids=[c[0] for c in CASES])
def test_fp8_decode_matches_oracle(cuda_device, name, B, Hq, Hkv, lengths):
    f = to_fp8(make_small(B, Hq, Hkv, 128, lengths, seed=zlib.crc32(name.encode()) % 1000))
    ws = torch.zeros(fd.workspace_bytes(B, Hq, Hkv, 128, f["kv_indptr"]), dtype=torch.uint8,
                     device=cuda_device)
    for rep in range(2):   # the second call reuses the workspace (tickets, claim counter)
        o, lse = _run(f, cuda_device, ws)
        torch.cuda.synchronize()
        assert fd.get_device_status(ws) == 0
    o_ref, lse_ref = oracle.decode_fp8(f["q"], f["k_fp8"], f["v_fp8"], f["k_scale"], f["v_scale"],
                                       f["kv_indptr"], f["scale"])
    err = errors(o.cpu().numpy(), lse.cpu().numpy(), o_ref.reshape(o.shape), lse_ref.reshape(lse.shape))
    assert_within(err, what=name)
    assert_within(err, **TIGHT, what=name + " (tight)")


@pytest.mark.parametrize("q_mult,k_mult", [(2e4, 1e-4), (1e-6, 1e6), (0.0, 1.0)])
def test_fp8_q_of_any_magnitude(cuda_device, q_mult, k_mult):
    """q beyond f16's range (|q| up to ~8e4), below its normal range (~1e-6), or
    zero: each row is rescaled by a power of two before it becomes an f16 MMA
    operand.  The K scales are multiplied by the inverse so that the logits,
    and hence the conditioning of the softmax, stay those of N(0,1) inputs."""
    f = to_fp8(make_small(2, 16, 4, 128, [700, 130], seed=11))
    f["q"] = (f["q"].float() * q_mult).to(torch.bfloat16)
    f["k_scale"] = f["k_scale"] * k_mult
    o, lse = _run(f, cuda_device)
    o_ref, lse_ref = oracle.decode_fp8(f["q"], f["k_fp8"], f["v_fp8"], f["k_scale"], f["v_scale"],
                                       f["kv_indptr"], f["scale"])
    err = errors(o.cpu().numpy(), lse.cpu().numpy(), o_ref.reshape(o.shape), lse_ref.reshape(lse.shape))
    assert_within(err, what=f"q x {q_mult}")


@pytest.mark.parametrize("idx", range(len(WORKLOADS)), ids=[w.name for w in WORKLOADS])
def test_fp8_full_size(cuda_device, idx):
    """Full-size workloads quantised to FP8, in the launch configuration the
    benchmark uses: every row against the oracle, rel-L2 over the whole O."""
    f = full_size.fp8_inputs(idx)
    o, lse = _run(f, cuda_device)
    torch.cuda.synchronize()
    o_ref, lse_ref = full_size.reference_fp8(idx)
    assert_within(errors(*full_size.as_rows(o, lse), o_ref, lse_ref), what=WORKLOADS[idx].name)


@pytest.mark.parametrize("page_size", [16, 32, 48, 64])
def test_fp8_paged_matches_oracle_and_ragged(cuda_device, page_size):
    f = to_fp8(make_small(4, 32, 8, 128, [1000, 1, 0, 2500], seed=page_size))
    pf = to_paged({**f, "k": f["k_fp8"], "v": f["v_fp8"]}, page_size, seed=page_size + 1)
    dev = cuda_device
    d = {k: pf[k].to(dev) for k in ("q", "k_pages", "v_pages", "kv_page_indptr", "kv_page_indices",
                                      "kv_last_page_len")}
    ks, vs = f["k_scale"].to(dev), f["v_scale"].to(dev)
    o, lse = fd.decode_paged_fp8(d["q"], d["k_pages"], d["v_pages"], ks, vs, pf["kv_page_indptr"],
                                 pf["kv_last_page_len"], d["kv_page_indptr"], d["kv_last_page_len"],
                                 d["kv_page_indices"], f["scale"])
    o_r, lse_r = _run(f, dev)
    torch.cuda.synchronize()
    kq, vq, ip = oracle.gather_paged(pf["k_pages"], pf["v_pages"], pf["kv_page_indptr"],
                                     pf["kv_page_indices"], pf["kv_last_page_len"])
    o_ref, lse_ref = oracle.decode_fp8(f["q"], kq, vq, f["k_scale"], f["v_scale"], ip, f["scale"])
    err = errors(o.cpu().numpy(), lse.cpu().numpy(), o_ref.reshape(o.shape), lse_ref.reshape(lse.shape))
    assert_within(err, **TIGHT, what=f"paged fp8 P={page_size}")
    # the same keys through the ragged FP8 path: the same bits
    assert torch.equal(o, o_r) and torch.equal(lse, lse_r)
