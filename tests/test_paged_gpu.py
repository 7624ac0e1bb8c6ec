"""Paged KV cache on the GPU (fd_decode_paged) against the fp64 oracle read
through the page table, and against fd_decode on the same keys laid out
ragged.

FD++ §6 (vLLM integration): the engine's page table maps each request's keys
onto fixed-size physical pages, and each split chunk streams the pages its
keys fall in.
"""
import numpy as np
import pytest
import torch

import oracle
import split_kv_flashdecoding_gb300 as fd
from tests import full_size
from tests.parity_util import assert_within, errors, to_device
from workloads import make_small, to_paged

pytestmark = pytest.mark.gpu

TIGHT = dict(max_abs=1e-4, rel_l2=1e-5, lse_abs=2e-5)

CASES = [
    ("ragged_gqa", 4, 32, 8, [1000, 1, 0, 2500]),
    ("mha", 2, 8, 8, [700, 4096]),
    ("g8_long", 2, 64, 8, [9000, 2500]),
    ("g2_tiny", 3, 4, 2, [17, 33, 64]),
]


def _paged_dev(pg, dev):
    return {k: pg[k].to(dev) for k in ("q", "k_pages", "v_pages", "kv_page_indptr",
                                       "kv_page_indices", "kv_last_page_len")}


def _decode_paged(pg, d, ws=None):
    return fd.decode_paged(d["q"], d["k_pages"], d["v_pages"], pg["kv_page_indptr"],
                           pg["kv_last_page_len"], d["kv_page_indptr"], d["kv_last_page_len"],
                           d["kv_page_indices"], pg["scale"], workspace=ws)


@pytest.mark.parametrize("page_size", [16, 32, 48, 64, 256])
@pytest.mark.parametrize("name,B,Hq,Hkv,lengths", CASES, ids=[c[0] for c in CASES])
def test_paged_matches_oracle_and_ragged(cuda_device, page_size, name, B, Hq, Hkv, lengths):
    inp = make_small(B, Hq, Hkv, 128, lengths, seed=len(name) * 31 + page_size)
    pg = to_paged(inp, page_size, seed=page_size + 1)
    d = _paged_dev(pg, cuda_device)
    info = fd.plan_paged(B, Hq, Hkv, 128, page_size, pg["kv_page_indptr"], pg["kv_last_page_len"])
    ws = torch.zeros(info.workspace_bytes, dtype=torch.uint8, device=cuda_device)
    o, lse = _decode_paged(pg, d, ws)
    torch.cuda.synchronize()
    assert fd.get_device_status(ws) == 0
    K, V, ip = oracle.gather_paged(pg["k_pages"], pg["v_pages"], pg["kv_page_indptr"],
                                   pg["kv_page_indices"], pg["kv_last_page_len"])
    o_ref, lse_ref = oracle.decode(inp["q"], K, V, ip, inp["scale"])
    err = errors(o.cpu().numpy(), lse.cpu().numpy(), o_ref.reshape(o.shape), lse_ref.reshape(lse.shape))
    assert_within(err, what=f"{name} P={page_size}")
    assert_within(err, **TIGHT, what=f"{name} P={page_size} (tight)")
    # the same keys laid out ragged go through the same splits: identical bits
    r = to_device(inp, cuda_device)
    o_r, lse_r = fd.decode(r["q"], r["k"], r["v"], inp["kv_indptr"], r["kv_indptr_dev"], inp["scale"])
    torch.cuda.synchronize()
    assert torch.equal(o, o_r) and torch.equal(lse, lse_r)


@pytest.mark.parametrize("page_size", [16, 64])
def test_paged_full_size_64k(cuda_device, page_size):
    """The 64k-context GQA workload (B=1, Hq=32, Hkv=8) in 16- and 64-key
    pages: all 32 rows against the oracle."""
    inp = full_size.inputs(1)
    pg = to_paged(inp, page_size, seed=11)
    d = _paged_dev(pg, cuda_device)
    o, lse = _decode_paged(pg, d)
    torch.cuda.synchronize()
    o_ref, lse_ref = full_size.reference(1)
    assert_within(errors(*full_size.as_rows(o, lse), o_ref, lse_ref), what=f"64k P={page_size}")


def test_page_index_outside_pool_is_flagged(cuda_device):
    """A page index past the pool sets FD_ERR_DEVICE_BOUNDS; the page is not read."""
    inp = make_small(1, 8, 8, 128, [200], seed=5)
    pg = to_paged(inp, 32, seed=2)
    bad = pg["kv_page_indices"].clone()
    bad[2] = pg["k_pages"].shape[0] + 7
    d = _paged_dev(pg, cuda_device)
    d["kv_page_indices"] = bad.to(cuda_device)
    info = fd.plan_paged(1, 8, 8, 128, 32, pg["kv_page_indptr"], pg["kv_last_page_len"])
    ws = torch.zeros(info.workspace_bytes, dtype=torch.uint8, device=cuda_device)
    o, lse = _decode_paged(pg, d, ws)
    assert fd.get_device_status(ws) == -6
    assert torch.isfinite(o).all()


def _unused_rows(pg):
    """[num_pages, page_size] mask of the pool rows no request's key occupies."""
    n, P = pg["k_pages"].shape[:2]
    used = torch.zeros(n, P, dtype=torch.bool)
    ip, idx, last = pg["kv_page_indptr"], pg["kv_page_indices"], pg["kv_last_page_len"]
    for b in range(len(ip) - 1):
        for j in range(int(ip[b]), int(ip[b + 1])):
            used[int(idx[j]), : int(last[b]) if j == int(ip[b + 1]) - 1 else P] = True
    return ~used


@pytest.mark.parametrize("page_size", [16, 64])
def test_nan_in_unused_page_rows_does_not_leak(cuda_device, page_size):
    """The rows past a request's last key in its last page are read with the
    page but must not touch the result: filled with NaN, they leave O and LSE
    bit-identical to zero-filled ones (bf16 and FP8 pools)."""
    from workloads import to_fp8
    inp = make_small(3, 16, 4, 128, [45, 70, 129], seed=page_size)
    pg = to_paged(inp, page_size, seed=5, spare_pages=0)
    unused = _unused_rows(pg)
    bad = dict(pg)
    for name in ("k_pages", "v_pages"):
        t = pg[name].clone()
        t[unused] = float("nan")
        bad[name] = t
    o0, l0 = _decode_paged(pg, _paged_dev(pg, cuda_device))
    o1, l1 = _decode_paged(bad, _paged_dev(bad, cuda_device))
    torch.cuda.synchronize()
    assert torch.isfinite(o1).all() and torch.isfinite(l1).all()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    # FP8: byte 0x7F is E4M3 NaN
    f = to_fp8(inp)
    pf = to_paged({**f, "k": f["k_fp8"], "v": f["v_fp8"]}, page_size, seed=5, spare_pages=0)
    dev = cuda_device
    ks, vs = f["k_scale"].to(dev), f["v_scale"].to(dev)
    outs = []
    for nan in (False, True):
        kp, vp = pf["k_pages"].clone(), pf["v_pages"].clone()
        if nan:
            kp[unused] = 0x7F
            vp[unused] = 0x7F
        d = {k: pf[k].to(dev) for k in ("q", "kv_page_indptr", "kv_page_indices", "kv_last_page_len")}
        outs.append(fd.decode_paged_fp8(d["q"], kp.to(dev), vp.to(dev), ks, vs, pf["kv_page_indptr"],
                                        pf["kv_last_page_len"], d["kv_page_indptr"],
                                        d["kv_last_page_len"], d["kv_page_indices"], f["scale"]))
    torch.cuda.synchronize()
    assert torch.isfinite(outs[1][0]).all() and torch.isfinite(outs[1][1]).all()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_back_to_back_paged_calls_with_page_tables_rewritten_in_stream(cuda_device):
    """Long paged splits read the page list through L2 and prefetch their first
    pages before waiting for the preceding grid.  Here every call is preceded,
    in the same stream and with no synchronisation, by kernels that rewrite the
    page list and the page contents between two layouts (different keys and a
    different page order): a page id read early may be stale, which may only
    misdirect a prefetch.  The queued calls must give the bits of the same
    calls made one at a time, with device status 0."""
    B, Hq, Hkv, P = 1, 32, 8, 16
    layouts = []
    for seed in (93, 94):
        inp = make_small(B, Hq, Hkv, 128, [16384], seed=seed)
        layouts.append(to_paged(inp, P, seed=seed + 10))
    info = fd.plan_paged(B, Hq, Hkv, 128, P, layouts[0]["kv_page_indptr"],
                         layouts[0]["kv_last_page_len"])
    split_keys = 16384 // info.total_splits
    assert split_keys > 4 * 32, "the splits must be longer than the ring"
    src = [_paged_dev(pg, cuda_device) for pg in layouts]
    for name in ("kv_page_indptr", "kv_last_page_len"):
        assert torch.equal(src[0][name], src[1][name])
    live = {k: src[0][k].clone() for k in src[0]}
    ws = torch.zeros(info.workspace_bytes, dtype=torch.uint8, device=cuda_device)

    def load(x):   # elementwise kernels writing the live page list and pools
        torch.add(src[x]["kv_page_indices"], 0, out=live["kv_page_indices"])
        torch.mul(src[x]["k_pages"], 1, out=live["k_pages"])
        torch.mul(src[x]["v_pages"], 1, out=live["v_pages"])
        torch.mul(src[x]["q"], 1, out=live["q"])

    ref = []
    for x in (0, 1):
        load(x)
        torch.cuda.synchronize()
        o, lse = _decode_paged(layouts[x], live, ws)
        torch.cuda.synchronize()
        ref.append((o.clone(), lse.clone()))
    assert not torch.equal(ref[0][0], ref[1][0])
    outs = []
    for i in range(24):
        load(i % 2)
        outs.append(_decode_paged(layouts[i % 2], live, ws))
    torch.cuda.synchronize()
    assert fd.get_device_status(ws) == 0
    for i, (o, lse) in enumerate(outs):
        o_ref, lse_ref = ref[i % 2]
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref), f"call {i}"
