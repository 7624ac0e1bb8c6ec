"""Seeded synthetic decode-attention inputs.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both the CUDA path's tests/bench and the CPU oracle take
their inputs from here, so the two sides see bit-identical bf16 tensors.

Layout (the ragged "packed" KV cache used throughout the library):
  q          bf16 [B, Hq, D]
  k, v       bf16 [T, Hkv, D]     T = kv_indptr[B]; request b owns rows
                                   kv_indptr[b] .. kv_indptr[b+1]-1
  kv_indptr  int32 [B+1]          kv_indptr[0] = 0, non-decreasing
  scale      Python float holding an fp32 value (1/sqrt(D) rounded to fp32)

Recipe (one torch CPU generator per workload, seed = 42 + index, draws in this
order; every draw is fp32 and then rounded to bf16 with round-to-nearest-even):
  1. per-request lengths (ragged workload only): integers uniform in [lo, hi]
  2. q
  3. K  (drawn in blocks of 65536 tokens, in token order)
  4. outlier positions (stressed workload only): for each (request b, kv head h)
     round(0.001 * L_b) distinct token positions, taken from a seeded
     permutation; K[pos, h, :] *= 16 before the bf16 rounding
  5. V  (same blocking as K)
The seed base 42 is the seed of the equivalence check printed on the
FlashDecoding++ sequence-split article (techknowgenie.com), section 5.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

_BLOCK_TOKENS = 65536


@dataclass(frozen=True)
class Workload:
    """One synthetic decode workload: shapes plus value distributions."""
    name: str
    index: int
    batch: int
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    kv_len: int | None            # fixed length, or None when ragged
    ragged: tuple | None = None   # (lo, hi) inclusive, when ragged
    q_std: float = 1.0
    v_dist: str = "normal"        # "normal" (N(0,1)) or "uniform" (U(-1,1))
    k_outlier_frac: float = 0.0   # fraction of positions per (request, head) scaled
    k_outlier_mult: float = 16.0
    description: str = field(default="", compare=False)


# The five decode workloads the benchmark and the full-size parity tests use.
WORKLOADS = [
    Workload("tiny_mha_b1_h8_l2048", 0, 1, 8, 8, 128, 2048,
             description="tiny MHA decode, B=1, Hq=Hkv=8, D=128, L=2048, N(0,1)"),
    Workload("gqa_b1_h32x8_l65536", 1, 1, 32, 8, 128, 65536,
             description="Llama-3-8B-shaped GQA decode, B=1, Hq=32, Hkv=8, L=65536, N(0,1)"),
    Workload("gqa_b1_h32x8_l131072", 2, 1, 32, 8, 128, 131072,
             description="GQA decode at 128k context, B=1, Hq=32, Hkv=8, L=131072, N(0,1)"),
    Workload("ragged_b64_h32x8_l512to16384", 3, 64, 32, 8, 128, None, ragged=(512, 16384),
             description="ragged batch, B=64, Hq=32, Hkv=8, L~U[512,16384], N(0,1)"),
    Workload("stressed_b16_h64x8_l32768", 4, 16, 64, 8, 128, 32768,
             q_std=2.0, v_dist="uniform", k_outlier_frac=0.001,
             description="stressed GQA, B=16, Hq=64, Hkv=8, L=32768, K N(0,1) with 0.1% "
                         "of positions per head x16, q std 2, V U(-1,1)"),
]


def workload(key) -> Workload:
    """Look a workload up by index or by name."""
    if isinstance(key, int):
        return WORKLOADS[key]
    for w in WORKLOADS:
        if w.name == key:
            return w
    raise KeyError(key)


def fp32_scale(head_dim: int) -> float:
    """1/sqrt(D) rounded to fp32 (the same fp32 value is given to every side)."""
    return float(np.float32(1.0 / math.sqrt(head_dim)))


def _lengths(w: Workload, g: torch.Generator) -> list[int]:
    if w.ragged is None:
        return [w.kv_len] * w.batch
    lo, hi = w.ragged
    return torch.randint(lo, hi + 1, (w.batch,), generator=g, dtype=torch.int64).tolist()


def _blocked_draw(shape_tail, rows, g, kind):
    """Draw a [rows, *shape_tail] fp32 array block by block, return bf16."""
    out = torch.empty((rows, *shape_tail), dtype=torch.bfloat16)
    for r0 in range(0, rows, _BLOCK_TOKENS):
        r1 = min(rows, r0 + _BLOCK_TOKENS)
        if kind == "normal":
            blk = torch.randn((r1 - r0, *shape_tail), generator=g, dtype=torch.float32)
        else:
            blk = torch.rand((r1 - r0, *shape_tail), generator=g, dtype=torch.float32) * 2.0 - 1.0
        out[r0:r1] = blk.to(torch.bfloat16)
    return out


def make_inputs(key, *, seed: int | None = None) -> dict:
    """Build one workload's inputs on the CPU (torch tensors, bf16 / int32)."""
    w = workload(key)
    g = torch.Generator(device="cpu")
    g.manual_seed(42 + w.index if seed is None else seed)
    lengths = _lengths(w, g)
    indptr = np.zeros(w.batch + 1, dtype=np.int64)
    indptr[1:] = np.cumsum(lengths)
    total = int(indptr[-1])
    assert total < 2**31, "token count must fit int32"
    D, Hq, Hkv = w.head_dim, w.num_qo_heads, w.num_kv_heads

    q = (torch.randn((w.batch, Hq, D), generator=g, dtype=torch.float32) * w.q_std).to(torch.bfloat16)

    if w.k_outlier_frac > 0.0:
        # Draw K in fp32, apply the outlier multiplier, then round to bf16.
        k32 = torch.empty((total, Hkv, D), dtype=torch.float32)
        for r0 in range(0, total, _BLOCK_TOKENS):
            r1 = min(total, r0 + _BLOCK_TOKENS)
            k32[r0:r1] = torch.randn((r1 - r0, Hkv, D), generator=g, dtype=torch.float32)
        for b in range(w.batch):
            L = lengths[b]
            n = int(round(w.k_outlier_frac * L))
            for h in range(Hkv):
                pos = torch.randperm(L, generator=g)[:n] + int(indptr[b])
                k32[pos, h, :] *= w.k_outlier_mult
        k = k32.to(torch.bfloat16)
        del k32
    else:
        k = _blocked_draw((Hkv, D), total, g, "normal")

    v = _blocked_draw((Hkv, D), total, g, w.v_dist)
    return dict(
        workload=w, q=q, k=k, v=v,
        kv_indptr=torch.from_numpy(indptr.astype(np.int32)),
        lengths=lengths, scale=fp32_scale(D),
    )


def make_small(batch: int, num_qo_heads: int, num_kv_heads: int, head_dim: int,
               lengths, *, seed: int = 0, q_std: float = 1.0, dtype=torch.bfloat16,
               v_dist: str = "normal") -> dict:
    """Small seeded inputs for parity and pin tests (same layout as make_inputs)."""
    assert len(lengths) == batch
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    indptr = np.zeros(batch + 1, dtype=np.int64)
    indptr[1:] = np.cumsum(lengths)
    total = int(indptr[-1])
    q = (torch.randn((batch, num_qo_heads, head_dim), generator=g) * q_std).to(dtype)
    k = torch.randn((total, num_kv_heads, head_dim), generator=g).to(dtype)
    if v_dist == "normal":
        v = torch.randn((total, num_kv_heads, head_dim), generator=g).to(dtype)
    else:
        v = (torch.rand((total, num_kv_heads, head_dim), generator=g) * 2.0 - 1.0).to(dtype)
    return dict(q=q, k=k, v=v, kv_indptr=torch.from_numpy(indptr.astype(np.int32)),
                lengths=list(lengths), scale=fp32_scale(head_dim))



def to_paged(inp: dict, page_size: int, *, seed: int = 7, spare_pages: int = 3) -> dict:
    """Lay a ragged input out as a paged KV cache (layout only, no arithmetic).

    Each request's keys fill ceil(L / page_size) pages in order; the pages are
    scattered over a pool of all used pages plus `spare_pages` unused ones in a
    seeded random order, so no request's pages are contiguous.  Returns the
    pools k_pages/v_pages [num_pages, page_size, Hkv, D] (unused rows zero),
    kv_page_indptr [B+1], kv_page_indices, kv_last_page_len [B] (int32).
    """
    k, v = inp["k"], inp["v"]
    ip = [int(x) for x in inp["kv_indptr"]]
    B = len(ip) - 1
    lens = [ip[b + 1] - ip[b] for b in range(B)]
    pages_per = [(L + page_size - 1) // page_size for L in lens]
    used = sum(pages_per)
    num_pages = used + spare_pages
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    perm = torch.randperm(num_pages, generator=g)[:used].tolist()
    Hkv, D = k.shape[1], k.shape[2]
    k_pages = torch.zeros((num_pages, page_size, Hkv, D), dtype=k.dtype)
    v_pages = torch.zeros((num_pages, page_size, Hkv, D), dtype=v.dtype)
    page_indptr = np.zeros(B + 1, dtype=np.int64)
    page_indptr[1:] = np.cumsum(pages_per)
    indices = np.array(perm, dtype=np.int32)
    last_len = np.zeros(B, dtype=np.int32)
    for b in range(B):
        for j in range(pages_per[b]):
            phys = perm[int(page_indptr[b]) + j]
            t0 = ip[b] + j * page_size
            t1 = min(t0 + page_size, ip[b + 1])
            k_pages[phys, : t1 - t0] = k[t0:t1]
            v_pages[phys, : t1 - t0] = v[t0:t1]
        if pages_per[b]:
            last_len[b] = lens[b] - (pages_per[b] - 1) * page_size
    out = dict(inp)
    out.update(k_pages=k_pages, v_pages=v_pages, page_size=page_size,
               kv_page_indptr=torch.from_numpy(page_indptr.astype(np.int32)),
               kv_page_indices=torch.from_numpy(indices),
               kv_last_page_len=torch.from_numpy(last_len))
    return out


def to_fp8(inp: dict) -> dict:
    """Quantise an input's K and V to FP8 E4M3 (storage layout only).

    Per tensor and KV head h: scale[h] = max |x[:, h, :]| / 448 in fp32 (1 for
    an all-zero head); codes = E4M3(x / scale[h]) rounded to nearest even,
    clamped to +-448 so nothing rounds to NaN.  Returns a copy of `inp` with
    k_fp8, v_fp8 (uint8 [T, Hkv, D]) and k_scale, v_scale (fp32 [Hkv]).
    """
    out = dict(inp)
    for name in ("k", "v"):
        x = inp[name].float()
        amax = x.abs().amax(dim=(0, 2)) if x.shape[0] else torch.zeros(x.shape[1])
        scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax)).float()
        q = (x / scale[None, :, None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
        out[name + "_fp8"] = q.view(torch.uint8).contiguous()
        out[name + "_scale"] = scale.contiguous()
    return out


def to_int4(inp: dict) -> dict:
    """Quantise an input's K and V to packed INT4 (storage layout only).

    Per tensor, key row t and KV head h: scale[h, t] = max |x[t, h, :]| / 7 in
    fp32 (1 for an all-zero row); codes = round-half-even(x / scale) clamped to
    -8..7, two per byte (element 2j in the low nibble of byte j, 2j + 1 in the
    high nibble, two's complement).  Returns a copy of `inp` with k_int4,
    v_int4 (uint8 [T, Hkv, D/2]) and k_scale_int4, v_scale_int4 (fp32
    [Hkv, T], head-major).
    """
    out = dict(inp)
    for name in ("k", "v"):
        x = inp[name].float()
        amax = x.abs().amax(dim=2) if x.shape[0] else torch.zeros(x.shape[:2])
        scale = torch.where(amax > 0, amax / 7.0, torch.ones_like(amax)).float()   # [T, Hkv]
        c = torch.round(x / scale[:, :, None]).clamp(-8, 7).to(torch.int16)
        u = (c & 0xF).to(torch.uint8)
        out[name + "_int4"] = (u[..., 0::2] | (u[..., 1::2] << 4)).contiguous()
        out[name + "_scale_int4"] = scale.t().contiguous()
    return out


def random_int4(inp: dict, *, seed: int = 11) -> dict:
    """Seeded uniformly random INT4 K/V for `inp`'s shapes: every byte (so
    every code -8..7 in both nibbles) equally likely, scales drawn from
    N(0, 0.5^2) (signs of both kinds).  Same keys as to_int4."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    out = dict(inp)
    T, Hkv, D = inp["k"].shape
    for name in ("k", "v"):
        out[name + "_int4"] = torch.randint(0, 256, (T, Hkv, D // 2), generator=g,
                                            dtype=torch.int32).to(torch.uint8)
        out[name + "_scale_int4"] = (torch.randn((Hkv, T), generator=g) * 0.5).float()
    return out


def to_paged_int4(inp: dict, page_size: int, *, seed: int = 7, spare_pages: int = 3) -> dict:
    """Lay an INT4 input (to_int4 / random_int4) out as a paged KV cache, with
    the same page order as to_paged(inp, page_size, seed=seed, spare_pages=...).

    Returns k_pages_int4 / v_pages_int4 [num_pages, page_size, Hkv, D/2]
    (unused rows zero), k_scale_pages / v_scale_pages fp32 [Hkv, num_pages *
    page_size] (entry h, p * page_size + r for row r of page p; unused zero),
    and the page table of to_paged.
    """
    codes = to_paged(dict(inp, k=inp["k_int4"], v=inp["v_int4"]), page_size, seed=seed,
                     spare_pages=spare_pages)
    # scales as [T, Hkv, 1] rows, paged the same way
    sc = to_paged(dict(inp, k=inp["k_scale_int4"].t()[:, :, None].contiguous(),
                       v=inp["v_scale_int4"].t()[:, :, None].contiguous()),
                  page_size, seed=seed, spare_pages=spare_pages)
    out = dict(codes)
    out["k"], out["v"] = inp["k"], inp["v"]
    out["k_pages_int4"], out["v_pages_int4"] = codes["k_pages"], codes["v_pages"]
    del out["k_pages"], out["v_pages"]
    n = sc["k_pages"].shape[0]
    Hkv = inp["k"].shape[1]
    for name in ("k", "v"):
        out[name + "_scale_pages"] = sc[name + "_pages"].reshape(n * page_size, Hkv).t().contiguous()
    return out
