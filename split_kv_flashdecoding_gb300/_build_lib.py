"""Build libfd.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

Each translation unit is compiled in parallel; the shared library links the
CUDA runtime statically, so it loads on a machine without a GPU (every CUDA
call then fails with FD_ERR_CUDA instead).
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libfd.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CUDA_SOURCES = ["split_kernel.cu", "split_kernel_fp8.cu", "split_kernel_int4.cu", "merge_kernel.cu",
                "fd_api.cu", "fd_static_ws.cu"]
HOST_SOURCES = ["plan.cpp"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: libfd needs the CUDA 13 toolkit to build")
    return cand


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "fd.h"))
    files.append(os.path.abspath(__file__))
    return files


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False, defines=(), out: str | None = None) -> str:
    """Compile csrc/ into _build/libfd.so if anything changed; return its path.

    defines/out build a variant (extra -D flags) into another file instead,
    e.g. to compare launch shapes.
    """
    if out is None and not force and not _stale():
        return LIB
    lib_path = out or LIB
    build_dir = os.path.dirname(lib_path) if out else BUILD
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", "-I", INCLUDE, "-I", CSRC, "-Xcompiler", "-fPIC",
              *[f"-D{d}" for d in defines]]
    jobs = []
    for src in CUDA_SOURCES:
        obj = os.path.join(build_dir, src + ".o")
        jobs.append([nvcc, *ARCH, "-lineinfo", *common, "-Xptxas", "-v" if verbose else "-O3",
                     "-c", os.path.join(CSRC, src), "-o", obj])
    for src in HOST_SOURCES:
        obj = os.path.join(build_dir, src + ".o")
        jobs.append([nvcc, *common, "-x", "c++", "-c", os.path.join(CSRC, src), "-o", obj])

    def run(cmd):
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"build failed: {' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
        return res.stderr

    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        logs = list(ex.map(run, jobs))
    if verbose:
        for log in logs:
            if log.strip():
                print(log)
    objs = [os.path.join(build_dir, s + ".o") for s in CUDA_SOURCES + HOST_SOURCES]
    tmp = lib_path + f".tmp{os.getpid()}"
    run([nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs, "-ldl", "-lpthread", "-lrt"])
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv))
