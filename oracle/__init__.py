"""fp64 CPU oracle for split-KV decode attention -- TEST INFRASTRUCTURE ONLY.

Only tests/, the smoke check and the benchmark's CPU-baseline leg may import
this package.  The product library never loads it and shares no code with it.

Source of the method: "FlashDecoding++: sequence-dimension KV split
parallelism for LLM serving" (techknowgenie.com), §3 "Partial softmax and
two-stage global reduction".

  decode(...)             the plain definition (unsplit softmax attention)
  split_partials(...)     §3 stage 1: per-chunk (acc, local max m, local sum l)
  normalised(acc, m, l)   the same partial as (O_i, LSE_i) = (acc/l, m + ln l)
  merge(acc, m, l, seg)   §3 stage 2: rescale by exp(m_i - M) and reduce
  gather_paged(...)       a paged KV cache read through its page table into the
                          ragged layout decode() takes (§6: the engine's page
                          table maps each request's keys onto physical pages)
  e4m3_to_float(codes)    FP8 E4M3 byte codes -> fp64 values (the OCP format
                          definition; §4: K/V held in FP8 in HBM)
  dequant_fp8(codes, s)   K or V codes [T, Hkv, D] times a per-KV-head scale
  decode_fp8(...)         decode() on exactly dequantised FP8 K/V (§4: the
                          quantised cache is dequantised, then attended over)
  int4_codes(packed)      packed four-bit two's-complement codes -> integers
                          (§4 names INT4 K/V beside FP8)
  dequant_int4(codes, s)  K or V codes [rows, Hkv, D/2] times a per-(row, KV
                          head) scale [Hkv, rows]
  decode_int4(...)        decode() on exactly dequantised INT4 K/V

The arithmetic is in fd_oracle.c (fp64 throughout); this module only
marshals arrays.  build() compiles it with gcc.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fd_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libfd_oracle.so")
_lock = threading.Lock()
_lib = None

_DTYPE_CODES = {"bf16": 0, "f32": 1, "f64": 2}


def build(force: bool = False) -> str:
    """Compile fd_oracle.c into oracle/_build/libfd_oracle.so (gcc, -O2)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            lib.fdo_decode.argtypes = [I, P, P, P, P, I64, I64, I64, I64, ctypes.c_double,
                                       P, I64, P, P, I]
            lib.fdo_decode.restype = I
            lib.fdo_split_partials.argtypes = [I, P, P, P, P, I64, I64, I64, I64,
                                               ctypes.c_double, P, I64, P, P, P]
            lib.fdo_split_partials.restype = I
            lib.fdo_merge.argtypes = [P, P, P, P, I64, I64, P, P]
            lib.fdo_merge.restype = I
            _lib = lib
    return _lib


def _as_array(x):
    """(dtype code, contiguous numpy array) for q/K/V given as torch or numpy."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return 0, x.view(torch.int16).numpy().view(np.uint16)
            if x.dtype == torch.float32:
                return 1, x.numpy()
            if x.dtype == torch.float64:
                return 2, x.numpy()
            raise TypeError(f"unsupported dtype {x.dtype}")
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return 1, x
    if x.dtype == np.float64:
        return 2, x
    if x.dtype == np.uint16:
        return 0, x
    raise TypeError(f"unsupported dtype {x.dtype}")


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _indptr(kv_indptr):
    return np.ascontiguousarray(np.asarray(kv_indptr, dtype=np.int64).reshape(-1))


def decode(q, k, v, kv_indptr, scale, rows=None, threads: int | None = None):
    """Unsplit fp64 decode attention.

    q [B,Hq,D], k/v [T,Hkv,D] (bf16/fp32/fp64 torch or numpy), kv_indptr [B+1].
    rows: optional flat (b*Hq + hq) row indices; default all rows.
    Returns (O fp64 [nrows, D], LSE fp64 [nrows]).
    """
    cq, qa = _as_array(q)
    ck, ka = _as_array(k)
    cv, va = _as_array(v)
    if not (cq == ck == cv):
        raise TypeError("q, k, v must share one dtype")
    B, Hq, D = qa.shape
    Hkv = ka.shape[1]
    ip = _indptr(kv_indptr)
    if rows is None:
        rows_a, nrows = None, B * Hq
    else:
        rows_a = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        nrows = rows_a.size
    o = np.zeros((nrows, D), dtype=np.float64)
    lse = np.zeros(nrows, dtype=np.float64)
    nthreads = threads or max(1, len(os.sched_getaffinity(0)))
    rc = _load().fdo_decode(cq, _ptr(qa), _ptr(ka), _ptr(va), _ptr(ip), B, Hq, Hkv, D,
                            float(scale), None if rows_a is None else _ptr(rows_a), nrows,
                            _ptr(o), _ptr(lse), nthreads)
    if rc != 0:
        raise ValueError("fdo_decode rejected its arguments")
    return o, lse


def split_partials(q, k, v, kv_indptr, scale, items):
    """Stage 1 over explicit chunks.

    items: int array [n, 4] of (b, kvh, tok_begin, tok_end) absolute key rows.
    Returns (acc [n,G,D], m [n,G], l [n,G]) in fp64.
    """
    cq, qa = _as_array(q)
    ck, ka = _as_array(k)
    cv, va = _as_array(v)
    if not (cq == ck == cv):
        raise TypeError("q, k, v must share one dtype")
    B, Hq, D = qa.shape
    Hkv = ka.shape[1]
    G = Hq // Hkv
    it = np.ascontiguousarray(np.asarray(items, dtype=np.int64).reshape(-1, 4))
    n = it.shape[0]
    acc = np.zeros((n, G, D), dtype=np.float64)
    m = np.zeros((n, G), dtype=np.float64)
    l = np.zeros((n, G), dtype=np.float64)
    ip = _indptr(kv_indptr)
    rc = _load().fdo_split_partials(cq, _ptr(qa), _ptr(ka), _ptr(va), _ptr(ip), B, Hq, Hkv, D,
                                    float(scale), _ptr(it), n, _ptr(acc), _ptr(m), _ptr(l))
    if rc != 0:
        raise ValueError("fdo_split_partials rejected its arguments")
    return acc, m, l


def normalised(acc, m, l):
    """The stored-partial reading: (O_i, LSE_i) = (acc/l, m + ln l), fp64."""
    acc = np.asarray(acc, dtype=np.float64)
    m = np.asarray(m, dtype=np.float64)
    l = np.asarray(l, dtype=np.float64)
    return acc / l[..., None], m + np.log(l)


def merge(acc, m, l, seg_indptr):
    """Stage 2 global reduction.

    acc [n, D], m [n], l [n] fp64; seg_indptr [R+1] groups partials per output
    row.  A normalised partial (O_i, LSE_i) is passed as acc=O_i, m=LSE_i, l=1.
    Returns (O fp64 [R, D], LSE fp64 [R]).
    """
    acc = np.ascontiguousarray(np.asarray(acc, dtype=np.float64))
    D = acc.shape[-1]
    acc = acc.reshape(-1, D)
    m = np.ascontiguousarray(np.asarray(m, dtype=np.float64).reshape(-1))
    l = np.ascontiguousarray(np.asarray(l, dtype=np.float64).reshape(-1))
    seg = np.ascontiguousarray(np.asarray(seg_indptr, dtype=np.int64).reshape(-1))
    R = seg.size - 1
    o = np.zeros((R, D), dtype=np.float64)
    lse = np.zeros(R, dtype=np.float64)
    rc = _load().fdo_merge(_ptr(acc), _ptr(m), _ptr(l), _ptr(seg), R, D, _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError("fdo_merge rejected its arguments")
    return o, lse


def gather_paged(k_pages, v_pages, kv_page_indptr, kv_page_indices, kv_last_page_len):
    """Read a paged KV cache through its page table (plain indexing).

    Request b's keys are rows 0..page_size-1 of pages
    kv_page_indices[kv_page_indptr[b]:kv_page_indptr[b+1]] in that order, the
    last page holding kv_last_page_len[b] keys.  Returns (K, V, kv_indptr) in
    the ragged layout: K/V [T, Hkv, D] (same dtype), kv_indptr int64 [B+1].
    """
    import torch
    ip = [int(x) for x in np.asarray(kv_page_indptr).reshape(-1)]
    idx = [int(x) for x in np.asarray(kv_page_indices).reshape(-1)]
    last = [int(x) for x in np.asarray(kv_last_page_len).reshape(-1)]
    ks, vs, lens = [], [], []
    for b in range(len(ip) - 1):
        L = 0
        for j in range(ip[b], ip[b + 1]):
            n = last[b] if j == ip[b + 1] - 1 else k_pages.shape[1]
            ks.append(k_pages[idx[j], :n])
            vs.append(v_pages[idx[j], :n])
            L += n
        lens.append(L)
    indptr = np.zeros(len(lens) + 1, dtype=np.int64)
    indptr[1:] = np.cumsum(lens)
    if ks:
        return torch.cat(ks), torch.cat(vs), indptr
    shape = (0, k_pages.shape[2], k_pages.shape[3])
    return torch.zeros(shape, dtype=k_pages.dtype), torch.zeros(shape, dtype=v_pages.dtype), indptr


def e4m3_to_float(codes) -> np.ndarray:
    """FP8 E4M3 codes (uint8) -> fp64, from the format definition.

    The OCP 8-bit floating-point format E4M3: 1 sign bit, 4 exponent bits with
    bias 7, 3 mantissa bits, no infinities.  Exponent field 0 is subnormal,
    (m / 8) * 2^-6; otherwise (1 + m / 8) * 2^(e - 7).  S.1111.111 is NaN, so
    the largest finite magnitude is 1.75 * 2^8 = 448.
    """
    c = np.asarray(codes).astype(np.uint8)
    sign = (c >> 7) & 1
    e = ((c >> 3) & 0xF).astype(np.int64)
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


def dequant_fp8(codes, scale) -> np.ndarray:
    """K or V as E4M3 codes [T, Hkv, D] with one fp32 scale per KV head [Hkv]
    -> fp64 values code * scale[h] (exact: 4 significant bits times 24)."""
    try:
        import torch
        if isinstance(codes, torch.Tensor):
            codes = codes.detach().cpu().contiguous().view(torch.uint8).numpy()
        if isinstance(scale, torch.Tensor):
            scale = scale.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    vals = e4m3_to_float(codes)
    s = np.asarray(scale, dtype=np.float32).astype(np.float64).reshape(1, -1, 1)
    return vals * s


def _bf16_to_f64(q) -> np.ndarray:
    code, a = _as_array(q)
    if code == 0:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def decode_fp8(q, k_codes, v_codes, k_scale, v_scale, kv_indptr, scale, rows=None,
               threads: int | None = None):
    """decode() on FP8 K/V: both are dequantised exactly (dequant_fp8) and q
    is widened to fp64, then the same unsplit definition runs in fp64."""
    return decode(_bf16_to_f64(q), dequant_fp8(k_codes, k_scale), dequant_fp8(v_codes, v_scale),
                  kv_indptr, scale, rows=rows, threads=threads)


def int4_codes(packed) -> np.ndarray:
    """Packed four-bit two's-complement codes -> int64 values, two per byte.

    Byte j of a row holds element 2j in its low nibble and element 2j + 1 in
    its high nibble; a nibble n stands for n - 16 when n >= 8 (so -8..7).
    packed [..., D/2] uint8 -> [..., D].
    """
    try:
        import torch
        if isinstance(packed, torch.Tensor):
            packed = packed.detach().cpu().contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    b = np.asarray(packed).astype(np.int64)
    nib = np.stack([b & 0xF, (b >> 4) & 0xF], axis=-1).reshape(*b.shape[:-1], 2 * b.shape[-1])
    return np.where(nib >= 8, nib - 16, nib)


def dequant_int4(packed, scale) -> np.ndarray:
    """K or V as packed INT4 codes [rows, Hkv, D/2] with one fp32 scale per
    (row, KV head), stored head-major [Hkv, rows] -> fp64 values
    code * scale[h, row] [rows, Hkv, D] (exact: 4-bit codes times 24 bits)."""
    try:
        import torch
        if isinstance(scale, torch.Tensor):
            scale = scale.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    vals = int4_codes(packed).astype(np.float64)
    s = np.asarray(scale, dtype=np.float32).astype(np.float64)   # [Hkv, rows]
    return vals * s.T[:, :, None]


def decode_int4(q, k_packed, v_packed, k_scale, v_scale, kv_indptr, scale, rows=None,
                threads: int | None = None):
    """decode() on INT4 K/V: both are dequantised exactly (dequant_int4) and q
    is widened to fp64, then the same unsplit definition runs in fp64."""
    return decode(_bf16_to_f64(q), dequant_int4(k_packed, k_scale), dequant_int4(v_packed, v_scale),
                  kv_indptr, scale, rows=rows, threads=threads)
