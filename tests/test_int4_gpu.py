"""INT4 KV on the GPU (fd_decode_int4, fd_decode_paged_int4) against the fp64
oracle on the exactly dequantised K/V (oracle.decode_int4).

FD++ §4 (quantisation-friendly fusion): the packed codes are read as they are
and dequantised in registers.  The reference result is attention over the
dequantised values; the tolerances are those of the bf16 path.  Inputs are
both quantised bf16 (to_int4: codes -7..7, positive scales) and uniformly
random bytes with signed scales (random_int4: every code -8..7).
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
import split_kv_flashdecoding_gb300 as fd
from tests import full_size
from tests.parity_util import assert_within, errors
from workloads import WORKLOADS, make_small, random_int4, to_int4, to_paged_int4

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
    ("odd_offsets", 4, 8, 1, [5, 33, 63, 2049]),  # scale rows start at every offset mod 4
    ("two_requests_g8", 2, 64, 8, [9000, 2500]),  # one wave on 152 SMs (296 items)
    # more items than one wave (600 on 152 SMs): the persistent kernel, in the
    # row form (G = 8) and the column form (G <= 4: keys and dims in the MMA rows)
    ("multi_wave_g8", 3, 64, 8, [16000, 16000, 3000]),
    ("multi_wave_g4", 3, 32, 8, [16000, 16000, 3000]),
    ("multi_wave_g2", 3, 16, 8, [16000, 16001, 2999]),
    ("multi_wave_g1", 3, 8, 8, [16001, 15999, 3000]),
]

KINDS = {"quantised": lambda inp: to_int4(inp), "random": lambda inp: random_int4(inp, seed=21)}


def _run(f, dev, ws=None):
    d = {k: f[k].to(dev) for k in ("q", "k_int4", "v_int4", "k_scale_int4", "v_scale_int4")}
    ip_dev = f["kv_indptr"].to(dev)
    return fd.decode_int4(d["q"], d["k_int4"], d["v_int4"], d["k_scale_int4"], d["v_scale_int4"],
                          f["kv_indptr"], ip_dev, f["scale"], workspace=ws)


def _ref(f, rows=None):
    return oracle.decode_int4(f["q"], f["k_int4"], f["v_int4"], f["k_scale_int4"],
                              f["v_scale_int4"], f["kv_indptr"], f["scale"], rows=rows)


@pytest.mark.parametrize("kind", sorted(KINDS))
@pytest.mark.parametrize("name,B,Hq,Hkv,lengths", CASES, ids=[c[0] for c in CASES])
def test_int4_decode_matches_oracle(cuda_device, name, B, Hq, Hkv, lengths, kind):
    f = KINDS[kind](make_small(B, Hq, Hkv, 128, lengths, seed=zlib.crc32(name.encode()) % 1000))
    ws = torch.zeros(fd.workspace_bytes(B, Hq, Hkv, 128, f["kv_indptr"]), dtype=torch.uint8,
                     device=cuda_device)
    for rep in range(2):   # the second call reuses the workspace (tickets, claim counter)
        o, lse = _run(f, cuda_device, ws)
        torch.cuda.synchronize()
        assert fd.get_device_status(ws) == 0
    o_ref, lse_ref = _ref(f)
    err = errors(o.cpu().numpy(), lse.cpu().numpy(), o_ref.reshape(o.shape), lse_ref.reshape(lse.shape))
    assert_within(err, what=f"{name} {kind}")
    assert_within(err, **TIGHT, what=f"{name} {kind} (tight)")


@pytest.mark.parametrize("idx", range(len(WORKLOADS)), ids=[w.name for w in WORKLOADS])
def test_int4_full_size(cuda_device, idx):
    """Full-size workloads quantised to INT4, in the launch configuration the
    benchmark uses: every row against the oracle, rel-L2 over the whole O."""
    f = full_size.int4_inputs(idx)
    o, lse = _run(f, cuda_device)
    torch.cuda.synchronize()
    o_ref, lse_ref = full_size.reference_int4(idx)
    assert_within(errors(*full_size.as_rows(o, lse), o_ref, lse_ref), what=WORKLOADS[idx].name)


def _paged_call(pg, f, dev):
    d = {k: pg[k].to(dev) for k in ("q", "k_pages_int4", "v_pages_int4", "k_scale_pages",
                                      "v_scale_pages", "kv_page_indptr", "kv_page_indices",
                                      "kv_last_page_len")}
    return fd.decode_paged_int4(d["q"], d["k_pages_int4"], d["v_pages_int4"], d["k_scale_pages"],
                                d["v_scale_pages"], pg["kv_page_indptr"], pg["kv_last_page_len"],
                                d["kv_page_indptr"], d["kv_last_page_len"], d["kv_page_indices"],
                                f["scale"])


@pytest.mark.parametrize("page_size", [16, 32, 48, 64])
def test_int4_paged_matches_oracle_and_ragged(cuda_device, page_size):
    f = random_int4(make_small(4, 32, 8, 128, [1000, 1, 0, 2500], seed=page_size))
    pg = to_paged_int4(f, page_size, seed=page_size + 1)
    o, lse = _paged_call(pg, f, cuda_device)
    o_r, lse_r = _run(f, cuda_device)
    torch.cuda.synchronize()
    o_ref, lse_ref = _ref(f)
    err = errors(o.cpu().numpy(), lse.cpu().numpy(), o_ref.reshape(o.shape), lse_ref.reshape(lse.shape))
    assert_within(err, **TIGHT, what=f"paged int4 P={page_size}")
    # the same keys through the ragged INT4 path: the same bits
    assert torch.equal(o, o_r) and torch.equal(lse, lse_r)


def test_int4_unused_page_rows_do_not_leak(cuda_device):
    """Rows past a request's last key in its last page hold NaN scales and
    arbitrary codes: the result is that of zeroed rows."""
    f = random_int4(make_small(2, 16, 4, 128, [45, 70], seed=31))
    pg = to_paged_int4(f, 32, seed=5, spare_pages=0)
    o0, l0 = _paged_call(pg, f, cuda_device)
    bad = dict(pg)
    n, P = pg["k_pages_int4"].shape[:2]
    used = torch.zeros(n, P, dtype=torch.bool)
    ip, idx, last = pg["kv_page_indptr"], pg["kv_page_indices"], pg["kv_last_page_len"]
    for b in range(len(ip) - 1):
        for j in range(int(ip[b]), int(ip[b + 1])):
            cnt = int(last[b]) if j == int(ip[b + 1]) - 1 else P
            used[int(idx[j]), :cnt] = True
    for name in ("k", "v"):
        codes = pg[name + "_pages_int4"].clone()
        codes[~used] = 0x88
        bad[name + "_pages_int4"] = codes
        sc = pg[name + "_scale_pages"].clone().reshape(-1, n, P)
        sc[:, ~used] = float("nan")
        bad[name + "_scale_pages"] = sc.reshape(-1, n * P).contiguous()
    o1, l1 = _paged_call(bad, f, cuda_device)
    torch.cuda.synchronize()
    assert torch.isfinite(o1).all() and torch.isfinite(l1).all()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)


def test_int4_rejects_misaligned_scales(cuda_device):
    """A scale pointer that is not fp32-aligned is refused before any launch."""
    import ctypes
    f = random_int4(make_small(1, 8, 2, 128, [100], seed=2))
    dev = cuda_device
    d = {k: f[k].to(dev) for k in ("q", "k_int4", "v_int4", "k_scale_int4", "v_scale_int4")}
    ip = np.ascontiguousarray(f["kv_indptr"].numpy().astype(np.int32))
    ipd = f["kv_indptr"].to(dev)
    o = torch.empty((1, 8, 128), dtype=torch.float32, device=dev)
    lse = torch.empty((1, 8), dtype=torch.float32, device=dev)
    ws = torch.zeros(fd.workspace_bytes(1, 8, 2, 128, f["kv_indptr"]), dtype=torch.uint8, device=dev)
    P = ctypes.c_void_p
    rc = fd.lib().fd_decode_int4(1, 8, 2, 128, ip.ctypes.data_as(P), P(ipd.data_ptr()),
                                 P(d["q"].data_ptr()), P(d["k_int4"].data_ptr()),
                                 P(d["v_int4"].data_ptr()), P(d["k_scale_int4"].data_ptr() + 2),
                                 P(d["v_scale_int4"].data_ptr()), float(f["scale"]), P(o.data_ptr()),
                                 P(lse.data_ptr()), P(ws.data_ptr()), ws.numel(), None)
    assert rc == -1


@pytest.mark.parametrize("regime", ["tiny", "huge", "log_spread"])
def test_int4_v_scales_of_any_magnitude(cuda_device, regime):
    """P V runs on f16 tensor cores with the weights p * v_scale brought into
    [-1, 1] by a running power of two per warp, so V scales far below f16's
    normal range (1e-9) or far above its largest value (1e9), or spread over
    thirteen decades within a request, keep the path's relative accuracy:
    compared with the oracle relative to the output's own magnitude."""
    f = random_int4(make_small(3, 32, 8, 128, [2000, 333, 4096], seed=71), seed=72)
    g = torch.Generator().manual_seed(73)
    T = f["v_scale_int4"].shape[1]
    sign = torch.where(torch.rand(8, T, generator=g) < 0.5, -1.0, 1.0)
    if regime == "tiny":
        mag = 1e-9 * (1 + torch.rand(8, T, generator=g))
    elif regime == "huge":
        mag = 1e9 * (1 + torch.rand(8, T, generator=g))
    else:
        mag = 10.0 ** (torch.rand(8, T, generator=g) * 13 - 9)   # 1e-9 .. 1e4
    f["v_scale_int4"] = (sign * mag).float()
    o, lse = _run(f, cuda_device)
    torch.cuda.synchronize()
    o_ref, lse_ref = _ref(f)
    o_h = o.reshape(o_ref.shape).cpu().double().numpy()
    scale = np.abs(o_ref).max()
    assert np.isfinite(o_h).all()
    assert np.abs(o_h - o_ref).max() <= 1e-4 * scale, regime
    assert np.linalg.norm(o_h - o_ref) <= 1e-5 * np.linalg.norm(o_ref), regime
    assert np.abs(lse.reshape(-1).cpu().numpy() - lse_ref).max() <= 2e-5
