"""The C-ABI library loads on a machine without a GPU, exports every symbol
include/fd.h declares, and rejects bad arguments on the host before any CUDA
call.  No compute call is made here."""
import ctypes
import os
import re
import subprocess

import pytest

import split_kv_flashdecoding_gb300 as fd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fd.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fd_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["fd_plan", "fd_decode_split", "fd_merge", "fd_decode",
                     "fd_get_device_status", "fd_status_string", "fd_plan_work_items"]:
        assert required in names


def test_library_exports_every_declared_symbol():
    lib = fd.lib()
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(fd.SIGNATURES)


def test_exports_are_c_symbols():
    out = subprocess.run(["nm", "-D", "--defined-only", fd.lib()._name], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (fd_[a-z0-9_]+)\b", out))
    assert set(declared_functions()) <= exported


def test_no_dynamic_cudart_dependency():
    out = subprocess.run(["ldd", fd.lib()._name], capture_output=True, text=True).stdout
    assert "libcudart" not in out


def test_status_strings():
    assert fd.status_string(0) == "FD_OK"
    assert fd.status_string(-5) == "FD_ERR_TIMEOUT"
    assert fd.status_string(-6) == "FD_ERR_DEVICE_BOUNDS"
    assert fd.status_string(123) == "FD_ERR_UNKNOWN"


def test_version():
    assert fd.lib().fd_version() >= 100


def _info():
    return fd.plan(1, 8, 8, 128, [0, 100], num_sms=4)


def test_decode_split_rejects_on_host():
    lib = fd.lib()
    info = _info()
    ws = ctypes.create_string_buffer(512)
    P = ctypes.c_void_p
    # null q
    assert lib.fd_decode_split(ctypes.byref(info), None, P(16), P(16), P(16), 0.1, P(16), P(16),
                               ctypes.cast(ws, P), 512, None) == -1
    # missing workspace
    assert lib.fd_decode_split(ctypes.byref(info), P(16), P(16), P(16), P(16), 0.1, P(16),
                               P(16), None, 0, None) == -3
    # misaligned k
    assert lib.fd_decode_split(ctypes.byref(info), P(16), P(18), P(16), P(16), 0.1, P(16),
                               P(16), ctypes.cast(ws, P), 512, None) == -1
    # inconsistent plan
    bad = _info()
    bad.num_work += 1
    assert lib.fd_decode_split(ctypes.byref(bad), P(16), P(16), P(16), P(16), 0.1, P(16),
                               P(16), ctypes.cast(ws, P), 512, None) == -1
    bad = _info()
    bad.group_size = 2
    assert lib.fd_decode_split(ctypes.byref(bad), P(16), P(16), P(16), P(16), 0.1, P(16),
                               P(16), ctypes.cast(ws, P), 512, None) == -1
    # NaN scale
    assert lib.fd_decode_split(ctypes.byref(info), P(16), P(16), P(16), P(16), float("nan"),
                               P(16), P(16), ctypes.cast(ws, P), 512, None) == -1


def test_merge_rejects_on_host():
    lib = fd.lib()
    info = _info()
    ws = ctypes.create_string_buffer(512)
    P = ctypes.c_void_p
    assert lib.fd_merge(ctypes.byref(info), None, P(16), P(16), P(16), P(16),
                        ctypes.cast(ws, P), 512, None) == -1
    assert lib.fd_merge(ctypes.byref(info), P(16), P(16), P(16), P(24), P(16),
                        ctypes.cast(ws, P), 512, None) == -1
    assert lib.fd_merge(ctypes.byref(info), P(16), P(16), P(16), P(16), P(16),
                        ctypes.cast(ws, P), 64, None) == -3


def test_decode_rejects_small_workspace_before_launch():
    lib = fd.lib()
    import numpy as np
    ip = np.array([0, 100], dtype=np.int32)
    P = ctypes.c_void_p
    rc = lib.fd_decode(1, 8, 8, 128, ip.ctypes.data_as(P), P(16), P(16), P(16), P(16), 0.1,
                       P(16), P(16), P(256), 16, None)
    # either the SM-count query fails (no GPU here) or the workspace check does
    assert rc in (-3, -4)


def test_plan_with_explicit_sms_needs_no_gpu():
    info = fd.plan(2, 32, 8, 128, [0, 1000, 3000], num_sms=152)
    assert info.num_sms == 152 and info.ctas_per_sm == 2
    assert info.timeout_ns == fd.DEFAULT_TIMEOUT_NS


def _prototypes():
    """name -> list of parameter declarations, parsed from include/fd.h."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    protos = {}
    for m in re.finditer(r"\b(fd_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", text):
        params = [p.strip() for p in m.group(2).split(",") if p.strip()]
        protos[m.group(1)] = [] if params == ["void"] else params
    return protos


def _kind(decl: str):
    if "*" in decl:
        return "ptr"
    if "int64_t" in decl or "size_t" in decl:
        return "i64"
    if "float" in decl:
        return "f32"
    return "i32"


def test_binding_signatures_match_the_header():
    """Every ctypes signature has the header's arity and parameter kinds, so a
    header change that the binding misses fails here rather than on a GPU."""
    to_kind = {ctypes.c_int: "i32", ctypes.c_int64: "i64", ctypes.c_float: "f32"}
    protos = _prototypes()
    assert set(protos) == set(fd.SIGNATURES)
    for name, params in protos.items():
        args, _ = fd.SIGNATURES[name]
        assert len(args) == len(params), f"{name}: {len(args)} ctypes args, header {len(params)}"
        for i, (a, decl) in enumerate(zip(args, params)):
            got = to_kind.get(a, "ptr")
            assert got == _kind(decl), f"{name} arg {i} ({decl}): binding {a}"
