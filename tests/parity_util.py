"""Shared helpers of the GPU parity tests: run the library through its C ABI and
compare with the oracle under the tolerances the decode path is held to."""
from __future__ import annotations

import numpy as np
import torch

import split_kv_flashdecoding_gb300 as fd

# Tolerances on fp32 outputs against the fp64 oracle (same seeded bf16 inputs):
# max |O - O_ref| <= 2e-3, ||O - O_ref||_2 / ||O_ref||_2 <= 1e-3, max |LSE - LSE_ref| <= 1e-4.
MAX_ABS = 2e-3
REL_L2 = 1e-3
LSE_ABS = 1e-4
SENTINEL = 12345.0


def errors(o, lse, o_ref, lse_ref) -> dict:
    o = np.asarray(o, dtype=np.float64).reshape(o_ref.shape)
    lse = np.asarray(lse, dtype=np.float64).reshape(lse_ref.shape)
    both_inf = np.isneginf(lse) & np.isneginf(lse_ref)
    finite = ~both_inf
    lse_err = float(np.abs(lse[finite] - lse_ref[finite]).max()) if finite.any() else 0.0
    if np.any(np.isneginf(lse) != np.isneginf(lse_ref)):
        lse_err = float("inf")
    diff = o - o_ref
    ref_norm = float(np.linalg.norm(o_ref))
    return dict(
        max_abs=float(np.abs(diff).max()) if diff.size else 0.0,
        rel_l2=float(np.linalg.norm(diff) / ref_norm) if ref_norm > 0 else float(np.linalg.norm(diff)),
        lse_abs=lse_err,
        finite=bool(np.all(np.isfinite(o))),
    )


def assert_within(err: dict, max_abs=MAX_ABS, rel_l2=REL_L2, lse_abs=LSE_ABS, what=""):
    assert err["finite"], f"{what}: non-finite output {err}"
    assert err["max_abs"] <= max_abs, f"{what}: max-abs {err}"
    assert err["rel_l2"] <= rel_l2, f"{what}: rel-L2 {err}"
    assert err["lse_abs"] <= lse_abs, f"{what}: LSE {err}"


def to_device(inp: dict, device) -> dict:
    out = dict(inp)
    for key in ("q", "k", "v"):
        out[key] = inp[key].to(device)
    out["kv_indptr_dev"] = inp["kv_indptr"].to(device)
    return out


def two_stage(dev_inp: dict, *, chunk=0, ctas_per_sm=0, num_sms=0, guard=0, stream=None,
              timeout_ns=None):
    """Plan + fd_decode_split + fd_merge through the C ABI.

    With guard > 0 every output buffer sits inside a larger one whose extra
    elements hold a sentinel; check_guards() verifies nothing wrote there.
    """
    q, k = dev_inp["q"], dev_inp["k"]
    B, Hq, D = q.shape
    Hkv = k.shape[1]
    info = fd.plan(B, Hq, Hkv, D, dev_inp["kv_indptr"], chunk=chunk, ctas_per_sm=ctas_per_sm,
                   num_sms=num_sms, timeout_ns=timeout_ns)
    dev = q.device
    rows = info.num_partial_rows
    g = guard * 128   # whole rows of 128 floats keep interior pointers 16-byte aligned

    def guarded(n):
        full = torch.full((n + 2 * g,), SENTINEL, dtype=torch.float32, device=dev)
        return full, full[g:g + n]

    po_full, po = guarded(rows * D)
    pl_full, pl = guarded(rows)
    o_full, o = guarded(B * Hq * D)
    l_full, lse = guarded(B * Hq)
    ws = torch.zeros(fd.WORKSPACE_HEADER_BYTES, dtype=torch.uint8, device=dev)
    fd.decode_split(info, q, k, dev_inp["v"], dev_inp["kv_indptr_dev"], dev_inp["scale"], po, pl,
                    ws, stream=stream)
    fd.merge(info, dev_inp["kv_indptr_dev"], po, pl, o, lse, ws, stream=stream)
    return dict(info=info, partial_o=po.view(rows, D), partial_lse=pl, o=o.view(B, Hq, D),
                lse=lse.view(B, Hq), ws=ws,
                guards=[(po_full, g, rows * D), (pl_full, g, rows), (o_full, g, B * Hq * D),
                        (l_full, g, B * Hq)])


def check_guards(res: dict):
    for full, g, n in res["guards"]:
        if g:
            assert torch.all(full[:g] == SENTINEL), "write before the buffer"
            assert torch.all(full[g + n:] == SENTINEL), "write past the buffer"


def partial_segments(info, kv_indptr) -> np.ndarray:
    """seg_indptr over partial rows per output row b*Hq + hq (documented layout:
    row = split_prefix[b]*Hq + hq*splits_b + s)."""
    ip = np.asarray(kv_indptr, dtype=np.int64)
    B, Hq = info.batch, info.num_qo_heads
    seg = np.zeros(B * Hq + 1, dtype=np.int64)
    prefix = 0
    for b in range(B):
        L = int(ip[b + 1] - ip[b])
        n = -(-L // info.chunk) if L > 0 else 0
        for hq in range(Hq):
            start = prefix * Hq + hq * n
            seg[b * Hq + hq] = start
            seg[b * Hq + hq + 1] = start + n
        prefix += n
    return seg
