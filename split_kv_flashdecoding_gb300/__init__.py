"""split_kv_flashdecoding_gb300 -- split-KV decode attention for GB300 (sm_103a).

A thin Python binding over the C ABI of libfd (include/fd.h).  Every step of
the computation runs in libfd's CUDA kernels; this module only marshals
pointers, sizes and the stream.  PyTorch supplies device memory and streams.

Entry points (same names as the C ABI, minus the ``fd_`` prefix):
  plan(...)          -> PlanInfo        host planner (chunk length, grid size)
  plan_work_items()  -> int32 [n, 5]    the plan's CTAs (b, kv_head, split, t0, t1)
  decode_split(...)                     stage 1: partial (O_i, LSE_i) per split
  merge(...)                            stage 2: LSE merge into O, LSE
  decode(...)        -> (O, LSE)        plan + stage 1 + stage 2
  decode_static_workspace(...)          the same for callers that cannot allocate
                                        (scratch in a fixed array in the library)
  plan_paged(...), decode_paged(...)    the same over a paged KV cache (page tables)
  decode_fp8(...), decode_paged_fp8()   FP8 (E4M3) K/V, one scale per KV head
  decode_int4(...), decode_paged_int4() INT4 K/V, one scale per key row and KV head
  plan_graph(...), decode_graph(...)    graph-capturable decode (device-side plan)
  merge_states(...)                     merge attention states (sequence shards)
  get_device_status(workspace)          read and clear the kernels' error word

There is no CPU fallback: if libfd.so cannot be loaded, importing the library
functions raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from ._build_lib import LIB as _LIB_PATH, build

TILE_TOKENS = 32
WORKSPACE_HEADER_BYTES = 256
DEFAULT_TIMEOUT_NS = 1_000_000_000

FD_OK = 0
STATUS_NAMES = {
    0: "FD_OK", -1: "FD_ERR_INVALID_ARG", -2: "FD_ERR_UNSUPPORTED", -3: "FD_ERR_WORKSPACE",
    -4: "FD_ERR_CUDA", -5: "FD_ERR_TIMEOUT", -6: "FD_ERR_DEVICE_BOUNDS",
}


class FdError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(code, code)} ({code})")
        self.code = code


class PlanInfo(ctypes.Structure):
    """Mirror of fd_plan_info (include/fd.h)."""
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("num_qo_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("group_size", ctypes.c_int32),
        ("chunk", ctypes.c_int32),
        ("total_splits", ctypes.c_int32),
        ("max_splits", ctypes.c_int32),
        ("num_work", ctypes.c_int32),
        ("num_partial_rows", ctypes.c_int32),
        ("num_sms", ctypes.c_int32),
        ("ctas_per_sm", ctypes.c_int32),
        ("total_tokens", ctypes.c_int64),
        ("workspace_bytes", ctypes.c_int64),
        ("timeout_ns", ctypes.c_int64),
    ]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


_lock = threading.Lock()
_lib = None

# Every symbol include/fd.h declares, with its ctypes signature.
_P, _I, _I64, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
_PI = ctypes.POINTER(PlanInfo)
SIGNATURES = {
    "fd_status_string": ([_I], ctypes.c_char_p),
    "fd_version": ([], _I),
    "fd_num_sms": ([_I, ctypes.POINTER(ctypes.c_int)], _I),
    "fd_plan": ([_I, _I, _I, _I, _P, _I, _I, _I, _PI], _I),
    "fd_plan_work_items": ([_PI, _P, _P, _I64], _I),
    "fd_decode_split": ([_PI, _P, _P, _P, _P, _F, _P, _P, _P, _I64, _P], _I),
    "fd_merge": ([_PI, _P, _P, _P, _P, _P, _P, _I64, _P], _I),
    "fd_decode": ([_I, _I, _I, _I, _P, _P, _P, _P, _P, _F, _P, _P, _P, _I64, _P], _I),
    "fd_get_device_status": ([_P, _P], _I),
    "fd_decode_static_workspace": ([_I, _I, _I, _I, _P, _P, _P, _P, _P, _F, _P, _P, _P], _I),
    "fd_plan_paged": ([_I, _I, _I, _I, _I, _P, _P, _I, _I, _I, _PI], _I),
    "fd_decode_paged": ([_I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _F, _P, _P,
                         _P, _I64, _P], _I),
    "fd_decode_fp8": ([_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _F, _P, _P, _P, _I64, _P], _I),
    "fd_plan_graph": ([_I, _I, _I, _I, _I64, _I, _I, _PI], _I),
    "fd_merge_states": ([_I, _I, _I, _P, _P, _P, _P, _P], _I),
    "fd_decode_graph": ([_PI, _P, _P, _P, _P, _F, _P, _P, _P, _I64, _P], _I),
    "fd_decode_paged_fp8": ([_I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _F,
                             _P, _P, _P, _I64, _P], _I),
    "fd_decode_int4": ([_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _F, _P, _P, _P, _I64, _P], _I),
    "fd_decode_paged_int4": ([_I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _F,
                              _P, _P, _P, _I64, _P], _I),
}


def lib(auto_build: bool = True):
    """Load libfd.so (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = build() if auto_build else _LIB_PATH
            if not os.path.exists(path):
                raise FdError(-4, f"libfd.so missing at {path}")
            handle = ctypes.CDLL(path)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.argtypes = args
                fn.restype = res
            _lib = handle
    return _lib


def _check(rc: int, what: str):
    if rc != FD_OK:
        raise FdError(rc, what)


def _host_indptr(kv_indptr) -> np.ndarray:
    try:
        import torch
        if isinstance(kv_indptr, torch.Tensor):
            kv_indptr = kv_indptr.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(np.asarray(kv_indptr, dtype=np.int32).reshape(-1))
    return a


def _ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def status_string(code: int) -> str:
    return lib().fd_status_string(code).decode()


def num_sms(device: int = -1) -> int:
    out = ctypes.c_int(0)
    _check(lib().fd_num_sms(device, ctypes.byref(out)), "fd_num_sms")
    return out.value


def plan(batch: int, num_qo_heads: int, num_kv_heads: int, head_dim: int, kv_indptr_host,
         *, num_sms: int = 0, ctas_per_sm: int = 0, chunk: int = 0,
         timeout_ns: int | None = None) -> PlanInfo:
    """fd_plan: choose the chunk length and size the split grid (host only)."""
    ip = _host_indptr(kv_indptr_host)
    if ip.size != batch + 1:
        raise FdError(-1, "kv_indptr must have batch+1 entries")
    info = PlanInfo()
    _check(lib().fd_plan(batch, num_qo_heads, num_kv_heads, head_dim,
                         ip.ctypes.data_as(ctypes.c_void_p), num_sms, ctas_per_sm, chunk,
                         ctypes.byref(info)), "fd_plan")
    if timeout_ns is not None:
        info.timeout_ns = timeout_ns
    return info


def plan_work_items(info: PlanInfo, kv_indptr_host) -> np.ndarray:
    """fd_plan_work_items: int32 [num_work, 5] = (b, kv_head, split, t0, t1)."""
    ip = _host_indptr(kv_indptr_host)
    items = np.zeros((max(info.num_work, 1), 5), dtype=np.int32)
    _check(lib().fd_plan_work_items(ctypes.byref(info), ip.ctypes.data_as(ctypes.c_void_p),
                                    items.ctypes.data_as(ctypes.c_void_p), info.num_work),
           "fd_plan_work_items")
    return items[: info.num_work]


def decode_split(info: PlanInfo, q, k, v, kv_indptr_dev, scale: float, partial_o, partial_lse,
                 workspace, stream=None):
    """fd_decode_split on torch CUDA tensors (stage 1; writes partial_o/partial_lse)."""
    _check(lib().fd_decode_split(ctypes.byref(info), _ptr(q), _ptr(k), _ptr(v),
                                 _ptr(kv_indptr_dev), float(scale), _ptr(partial_o),
                                 _ptr(partial_lse), _ptr(workspace), workspace.numel() *
                                 workspace.element_size(), _stream(stream)), "fd_decode_split")


def merge(info: PlanInfo, kv_indptr_dev, partial_o, partial_lse, o, lse, workspace, stream=None):
    """fd_merge on torch CUDA tensors (stage 2; writes o/lse)."""
    _check(lib().fd_merge(ctypes.byref(info), _ptr(kv_indptr_dev), _ptr(partial_o),
                          _ptr(partial_lse), _ptr(o), _ptr(lse), _ptr(workspace),
                          workspace.numel() * workspace.element_size(), _stream(stream)),
           "fd_merge")


def workspace_bytes(batch, num_qo_heads, num_kv_heads, head_dim, kv_indptr_host) -> int:
    """Workspace fd_decode needs for these arguments on the current device."""
    return plan(batch, num_qo_heads, num_kv_heads, head_dim, kv_indptr_host).workspace_bytes


def decode(q, k, v, kv_indptr_host, kv_indptr_dev, scale: float, *, o=None, lse=None,
           workspace=None, stream=None):
    """fd_decode: q [B,Hq,D], k/v [T,Hkv,D] bf16 CUDA tensors -> (O fp32, LSE fp32).

    kv_indptr_host: int32 [B+1] on the host (numpy or CPU tensor);
    kv_indptr_dev: the same values as an int32 CUDA tensor.
    """
    import torch
    B, Hq, D = q.shape
    Hkv = k.shape[1]
    ip = _host_indptr(kv_indptr_host)
    if o is None:
        o = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        need = plan(B, Hq, Hkv, D, ip).workspace_bytes
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    _check(lib().fd_decode(B, Hq, Hkv, D, ip.ctypes.data_as(ctypes.c_void_p), _ptr(kv_indptr_dev),
                           _ptr(q), _ptr(k), _ptr(v), float(scale), _ptr(o), _ptr(lse),
                           _ptr(workspace), workspace.numel() * workspace.element_size(),
                           _stream(stream)), "fd_decode")
    return o, lse


def decode_static_workspace(q, k, v, kv_indptr_host, kv_indptr_dev, scale: float, *, o=None,
                            lse=None, stream=None):
    """fd_decode_static_workspace: fd_decode for callers that cannot allocate.

    The library keeps the scratch in a fixed device array (16 MiB per GPU), so
    only inputs and outputs are passed; o/lse are allocated here only when not
    given.  Calls that can overlap on the GPU race (they share the array).
    """
    import torch
    B, Hq, D = q.shape
    Hkv = k.shape[1]
    ip = _host_indptr(kv_indptr_host)
    if o is None:
        o = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    _check(lib().fd_decode_static_workspace(B, Hq, Hkv, D, ip.ctypes.data_as(ctypes.c_void_p),
                                            _ptr(kv_indptr_dev), _ptr(q), _ptr(k), _ptr(v),
                                            float(scale), _ptr(o), _ptr(lse), _stream(stream)),
           "fd_decode_static_workspace")
    return o, lse


def plan_paged(batch: int, num_qo_heads: int, num_kv_heads: int, head_dim: int, page_size: int,
               kv_page_indptr_host, kv_last_page_len_host, *, num_sms: int = 0,
               ctas_per_sm: int = 0, chunk: int = 0) -> PlanInfo:
    """fd_plan_paged: the plan of a paged layout (host only)."""
    ip = _host_indptr(kv_page_indptr_host)
    ll = _host_indptr(kv_last_page_len_host)
    if ip.size != batch + 1 or ll.size != batch:
        raise FdError(-1, "kv_page_indptr must have batch+1 and kv_last_page_len batch entries")
    info = PlanInfo()
    _check(lib().fd_plan_paged(batch, num_qo_heads, num_kv_heads, head_dim, page_size,
                               ip.ctypes.data_as(ctypes.c_void_p), ll.ctypes.data_as(ctypes.c_void_p),
                               num_sms, ctas_per_sm, chunk, ctypes.byref(info)), "fd_plan_paged")
    return info


def decode_paged(q, k_pages, v_pages, kv_page_indptr_host, kv_last_page_len_host,
                 kv_page_indptr_dev, kv_last_page_len_dev, kv_page_indices_dev, scale: float, *,
                 o=None, lse=None, workspace=None, stream=None):
    """fd_decode_paged: q [B,Hq,D], page pools k/v [num_pages, page_size, Hkv, D] bf16.

    Page tables as in include/fd.h (host copies of indptr and last-page
    lengths for the plan, device copies plus the page indices for the kernels).
    """
    import torch
    B, Hq, D = q.shape
    num_pages, page_size, Hkv = k_pages.shape[0], k_pages.shape[1], k_pages.shape[2]
    ip = _host_indptr(kv_page_indptr_host)
    ll = _host_indptr(kv_last_page_len_host)
    if o is None:
        o = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        need = plan_paged(B, Hq, Hkv, D, page_size, ip, ll).workspace_bytes
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    _check(lib().fd_decode_paged(B, Hq, Hkv, D, page_size, num_pages,
                                 ip.ctypes.data_as(ctypes.c_void_p),
                                 ll.ctypes.data_as(ctypes.c_void_p), _ptr(kv_page_indptr_dev),
                                 _ptr(kv_last_page_len_dev), _ptr(kv_page_indices_dev), _ptr(q),
                                 _ptr(k_pages), _ptr(v_pages), float(scale), _ptr(o), _ptr(lse),
                                 _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream(stream)), "fd_decode_paged")
    return o, lse


def _fp8_bytes(x):
    """An FP8 K/V tensor as torch gives it (float8_e4m3fn) or as raw uint8."""
    import torch
    if x.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise FdError(-1, "FP8 K/V must be uint8 or float8_e4m3fn")
    return x


def decode_fp8(q, k_fp8, v_fp8, k_scale, v_scale, kv_indptr_host, kv_indptr_dev, scale: float, *,
               o=None, lse=None, workspace=None, stream=None):
    """fd_decode_fp8: q [B,Hq,D] bf16, k/v [T,Hkv,D] E4M3 bytes (uint8 or
    float8_e4m3fn), k_scale / v_scale fp32 [Hkv] CUDA tensors -> (O, LSE) fp32."""
    import torch
    B, Hq, D = q.shape
    Hkv = k_fp8.shape[1]
    ip = _host_indptr(kv_indptr_host)
    if o is None:
        o = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        need = plan(B, Hq, Hkv, D, ip).workspace_bytes
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    _check(lib().fd_decode_fp8(B, Hq, Hkv, D, ip.ctypes.data_as(ctypes.c_void_p), _ptr(kv_indptr_dev),
                               _ptr(q), _ptr(_fp8_bytes(k_fp8)), _ptr(_fp8_bytes(v_fp8)),
                               _ptr(k_scale), _ptr(v_scale), float(scale), _ptr(o), _ptr(lse),
                               _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _stream(stream)), "fd_decode_fp8")
    return o, lse


def decode_paged_fp8(q, k_pages_fp8, v_pages_fp8, k_scale, v_scale, kv_page_indptr_host,
                     kv_last_page_len_host, kv_page_indptr_dev, kv_last_page_len_dev,
                     kv_page_indices_dev, scale: float, *, o=None, lse=None, workspace=None,
                     stream=None):
    """fd_decode_paged_fp8: fd_decode_paged over E4M3 page pools with
    per-KV-head fp32 scales."""
    import torch
    B, Hq, D = q.shape
    num_pages, page_size, Hkv = k_pages_fp8.shape[0], k_pages_fp8.shape[1], k_pages_fp8.shape[2]
    ip = _host_indptr(kv_page_indptr_host)
    ll = _host_indptr(kv_last_page_len_host)
    if o is None:
        o = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        need = plan_paged(B, Hq, Hkv, D, page_size, ip, ll).workspace_bytes
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    _check(lib().fd_decode_paged_fp8(B, Hq, Hkv, D, page_size, num_pages,
                                     ip.ctypes.data_as(ctypes.c_void_p),
                                     ll.ctypes.data_as(ctypes.c_void_p), _ptr(kv_page_indptr_dev),
                                     _ptr(kv_last_page_len_dev), _ptr(kv_page_indices_dev), _ptr(q),
                                     _ptr(_fp8_bytes(k_pages_fp8)), _ptr(_fp8_bytes(v_pages_fp8)),
                                     _ptr(k_scale), _ptr(v_scale), float(scale), _ptr(o), _ptr(lse),
                                     _ptr(workspace), workspace.numel() * workspace.element_size(),
                                     _stream(stream)), "fd_decode_paged_fp8")
    return o, lse


def _int4_bytes(x, D: int):
    """Packed INT4 K/V: uint8 with D / 2 bytes per (row, KV head)."""
    import torch
    if x.dtype != torch.uint8 or x.shape[-1] != D // 2:
        raise FdError(-1, "INT4 K/V must be uint8 [..., Hkv, head_dim / 2]")
    return x


def decode_int4(q, k_int4, v_int4, k_scale, v_scale, kv_indptr_host, kv_indptr_dev, scale: float, *,
                o=None, lse=None, workspace=None, stream=None):
    """fd_decode_int4: q [B,Hq,D] bf16, k/v [T,Hkv,D/2] packed four-bit codes
    (uint8), k_scale / v_scale fp32 [Hkv, T] CUDA tensors -> (O, LSE) fp32."""
    import torch
    B, Hq, D = q.shape
    Hkv = k_int4.shape[1]
    ip = _host_indptr(kv_indptr_host)
    if o is None:
        o = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        need = plan(B, Hq, Hkv, D, ip).workspace_bytes
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    _check(lib().fd_decode_int4(B, Hq, Hkv, D, ip.ctypes.data_as(ctypes.c_void_p),
                                _ptr(kv_indptr_dev), _ptr(q), _ptr(_int4_bytes(k_int4, D)),
                                _ptr(_int4_bytes(v_int4, D)), _ptr(k_scale), _ptr(v_scale),
                                float(scale), _ptr(o), _ptr(lse), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream)),
           "fd_decode_int4")
    return o, lse


def decode_paged_int4(q, k_pages_int4, v_pages_int4, k_scale, v_scale, kv_page_indptr_host,
                      kv_last_page_len_host, kv_page_indptr_dev, kv_last_page_len_dev,
                      kv_page_indices_dev, scale: float, *, o=None, lse=None, workspace=None,
                      stream=None):
    """fd_decode_paged_int4: fd_decode_paged over packed INT4 page pools
    [num_pages, page_size, Hkv, D/2] with fp32 scales [Hkv, num_pages * page_size]."""
    import torch
    B, Hq, D = q.shape
    num_pages, page_size, Hkv = k_pages_int4.shape[0], k_pages_int4.shape[1], k_pages_int4.shape[2]
    ip = _host_indptr(kv_page_indptr_host)
    ll = _host_indptr(kv_last_page_len_host)
    if o is None:
        o = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        need = plan_paged(B, Hq, Hkv, D, page_size, ip, ll).workspace_bytes
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    _check(lib().fd_decode_paged_int4(B, Hq, Hkv, D, page_size, num_pages,
                                      ip.ctypes.data_as(ctypes.c_void_p),
                                      ll.ctypes.data_as(ctypes.c_void_p), _ptr(kv_page_indptr_dev),
                                      _ptr(kv_last_page_len_dev), _ptr(kv_page_indices_dev), _ptr(q),
                                      _ptr(_int4_bytes(k_pages_int4, D)),
                                      _ptr(_int4_bytes(v_pages_int4, D)), _ptr(k_scale),
                                      _ptr(v_scale), float(scale), _ptr(o), _ptr(lse),
                                      _ptr(workspace), workspace.numel() * workspace.element_size(),
                                      _stream(stream)), "fd_decode_paged_int4")
    return o, lse


def plan_graph(batch: int, num_qo_heads: int, num_kv_heads: int, head_dim: int,
               max_total_tokens: int, *, num_sms: int = 0, chunk: int = 0) -> PlanInfo:
    """fd_plan_graph: a plan for any kv_indptr of at most max_total_tokens keys
    (host only; fixes the chunk, sizes the workspace)."""
    info = PlanInfo()
    _check(lib().fd_plan_graph(batch, num_qo_heads, num_kv_heads, head_dim, int(max_total_tokens),
                               num_sms, chunk, ctypes.byref(info)), "fd_plan_graph")
    return info


def decode_graph(info: PlanInfo, q, k, v, kv_indptr_dev, scale: float, o, lse, workspace,
                 stream=None):
    """fd_decode_graph: device data only (capturable in a CUDA graph); o, lse
    and the workspace (info.workspace_bytes, zero-filled once) are given."""
    _check(lib().fd_decode_graph(ctypes.byref(info), _ptr(kv_indptr_dev), _ptr(q), _ptr(k), _ptr(v),
                                 float(scale), _ptr(o), _ptr(lse), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream)),
           "fd_decode_graph")


def merge_states(o_states, lse_states, *, o=None, lse=None, stream=None):
    """fd_merge_states: o_states fp32 [S, ..., D] and lse_states fp32 [S, ...]
    (S attention states over disjoint parts of the keys) -> merged (O, LSE)."""
    import torch
    S, D = o_states.shape[0], o_states.shape[-1]
    rows = lse_states[0].numel()
    if o is None:
        o = torch.empty(o_states.shape[1:], dtype=torch.float32, device=o_states.device)
    if lse is None:
        lse = torch.empty(lse_states.shape[1:], dtype=torch.float32, device=lse_states.device)
    _check(lib().fd_merge_states(S, rows, D, _ptr(o_states), _ptr(lse_states), _ptr(o), _ptr(lse),
                                 _stream(stream)), "fd_merge_states")
    return o, lse


def get_device_status(workspace, stream=None) -> int:
    """fd_get_device_status: synchronise, read and clear the kernels' status word."""
    return lib().fd_get_device_status(_ptr(workspace), _stream(stream))


__all__ = [
    "PlanInfo", "FdError", "lib", "build", "plan", "plan_work_items", "decode_split", "merge",
    "decode", "decode_static_workspace", "plan_paged", "decode_paged", "decode_fp8",
    "decode_paged_fp8", "decode_int4", "decode_paged_int4", "plan_graph", "decode_graph", "merge_states", "get_device_status",
    "workspace_bytes", "num_sms",
    "status_string",
    "TILE_TOKENS", "WORKSPACE_HEADER_BYTES", "DEFAULT_TIMEOUT_NS",
]
