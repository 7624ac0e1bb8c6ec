"""Benchmark of one split-KV decode-attention step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl fd|reference] [--kv-dtype bf16|fp8|int4] [--page-size P]
                    [--graph] [--min-timed-ms MS] [--no-per-workload]

A step is the whole path: one fd_decode call through the C ABI, i.e. the host
plan (fd_plan), stage 1 (the split kernel) and stage 2 (fused into it), on one
batch of seeded synthetic inputs already resident in HBM.  The headline
workload is the Llama-3-8B-shaped GQA decode at 64k context (B=1, Hq=32,
Hkv=8, D=128, L=65536).  After W warm-up steps the K-step loop runs back to
back inside one pair of CUDA events, repeated until the timed region lasts at
least --min-timed-ms (200 ms); the K/V a step reads is at least twice the L2
size (small workloads rotate through copies of their inputs), so no step is
served from L2.  Stage 1 alone is also timed (back to back), and each step once
more one at a time after a 1 GiB L2 flush (that number includes launch latency
and event overhead).  Every other workload is then timed the same way, with
the same kind of step, into `per_workload`.

Prints one JSON line (rank 0).  `value` is achieved bandwidth in GB/s: the
algorithmic bytes of a step (q + K + V + O + LSE + the partials written and
read back) over the device time of the step; `ms_per_step` is that time.
`roofline` is that of the step's one kernel (the split kernel with stage 2
fused).  `--impl reference` times the fp64 CPU oracle on the host cores
instead (a bounded sample of the same workload, extrapolated to one step),
without loading the library.

Multi-GPU (torchrun): every rank runs its own copy of the workload (requests
are independent, no collective on the data path); value = all ranks' bytes /
the slowest rank's time ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import WORKLOADS, workload  # noqa: E402

METRIC = "decode-attention µs/step and achieved HBM GB/s vs ~8 TB/s GB300 peak"
DEFAULT_WORKLOAD = "gqa_b1_h32x8_l65536"
L2_FLUSH_BYTES = 1 << 30
GRAPH_STEPS = 8   # decode steps captured per CUDA graph with --graph
L2_BYTES = 129 * 1000 * 1000       # GB300 L2
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
SPLIT_SOURCES = ["split_kernel.cuh", "split_kernel.cu", "split_kernel_fp8.cu", "split_kernel_int4.cu",
                 "device_common.cuh", "plan_rule.h", "fd_api.cu"]


# ----------------------------------------------------------------- helpers

def kv_row_bytes(kv_dtype: str, D: int) -> int:
    """Bytes of one key row of one KV head in K (or V): bf16 2 per element,
    FP8 1 (its per-head scale is a few bytes per step), INT4 half a byte plus
    the row's fp32 scale."""
    return {"bf16": 2 * D, "fp8": D, "int4": D // 2 + 4}[kv_dtype]


def step_bytes(B, Hq, Hkv, D, T, rows, row_bytes=None) -> dict:
    """Algorithmic bytes of one step and of each kernel launch (K and V rows
    of row_bytes each per KV head; bf16 by default)."""
    q = B * Hq * D * 2
    kv = 2 * T * Hkv * (2 * D if row_bytes is None else row_bytes)
    out = B * Hq * (D + 1) * 4
    part = rows * (D + 1) * 4
    return dict(step=q + kv + out + 2 * part, split=q + kv + part, merge=part + out,
                kv=kv, q=q, out=out, partials=2 * part)


def measured_peaks() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def split_source_hash() -> str:
    h = hashlib.sha256()
    for name in SPLIT_SOURCES:
        with open(os.path.join(ROOT, "split_kv_flashdecoding_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload_name: str):
    """DRAM bytes per split-kernel launch from the committed ncu summary, if it
    was taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "split_kernel_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_hash") != split_source_hash():
        return None
    entry = rec.get("workloads", {}).get(workload_name)
    return None if entry is None else entry.get("dram_bytes_per_launch")


# ------------------------------------------------- partial rows of a plan

TILE_TOKENS = 32        # keys per pipeline stage (FD_TILE_TOKENS)
MIN_CHUNK = 128         # FD_MIN_CHUNK
CTA_OVERHEAD_TILES = 3  # the planner's fixed per-CTA cost, in tiles
CTAS_PER_SM = 2         # resident split-kernel CTAs per SM


def _splits(L, c):
    return -(-L // c) if L > 0 else 0


def _split_len(L, n):
    return -(-(-(-L // n)) // TILE_TOKENS) * TILE_TOKENS


def plan_chunk(lengths, num_kv_heads: int, num_sms: int) -> int:
    """The chunk length fd_plan picks (the rule include/fd.h documents): for
    grids of 1, 2, 4 and 8 waves of resident CTAs, the chunk that sizes the
    grid; keep the one whose dispatch, simulated in launch order onto the
    resident-CTA slots, ends first (the fewest waves on a tie).  Host
    bookkeeping only: the reference arm counts the partial bytes of the same
    plan without loading the library."""
    import heapq
    slots = num_sms * CTAS_PER_SM
    total = int(sum(lengths))

    def chunk_for(target):
        c = -(-(-(-total * num_kv_heads // target)) // TILE_TOKENS) * TILE_TOKENS
        return min(max(c, MIN_CHUNK), 1 << 30)

    def costs(c):
        for L in lengths:
            n = _splits(L, c)
            if n:
                sl = _split_len(L, n)
                for s_ in range(n):
                    keys = min(sl, L - s_ * sl)
                    yield -(-keys // TILE_TOKENS) + CTA_OVERHEAD_TILES

    best_c, best_t, last_c = chunk_for(slots), -1, -1
    for waves in (1, 2, 4, 8):
        c = chunk_for(slots * waves)
        if c == last_c:
            continue
        last_c = c
        cs = list(costs(c))
        ctas = len(cs) * num_kv_heads
        largest = max(cs, default=0)
        if ctas <= slots:
            t = largest
        else:
            lower = max(largest, -(-sum(cs) * num_kv_heads // slots))
            if best_t >= 0 and lower >= best_t:
                continue
            free = [0] * slots       # each CTA takes the earliest free slot
            heapq.heapify(free)
            for cost in cs:          # the KV heads of one split, in a row
                taken = []
                for _ in range(num_kv_heads):
                    if not free:         # more KV heads than slots: reuse the first ones
                        for x in taken:
                            heapq.heappush(free, x)
                        taken = []
                    taken.append(heapq.heappop(free) + cost)
                for x in taken:
                    heapq.heappush(free, x)
            t = max(free)
        if best_t < 0 or t < best_t:
            best_t, best_c = t, c
    return best_c


def plan_partial_rows(lengths, num_qo_heads: int, num_kv_heads: int, num_sms: int) -> int:
    c = plan_chunk(lengths, num_kv_heads, num_sms)
    return sum(_splits(L, c) for L in lengths) * num_qo_heads


def device_sm_count(default: int = 152) -> tuple[int, str]:
    """SM count of GPU 0 from the CUDA driver (no context is created), or the
    GB300's 152 when no driver answers."""
    import ctypes
    try:
        cu = ctypes.CDLL("libcuda.so.1")
        dev, n = ctypes.c_int(), ctypes.c_int()
        if cu.cuInit(0) == 0 and cu.cuDeviceGet(ctypes.byref(dev), 0) == 0 and \
                cu.cuDeviceGetAttribute(ctypes.byref(n), 16, dev) == 0 and n.value > 0:
            return n.value, "CUDA driver"    # 16: CU_DEVICE_ATTRIBUTE_MULTIPROCESSOR_COUNT
    except OSError:
        pass
    return default, "GB300 default"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed loop runs."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.device_index = device_index
        self.proc = None
        self.file = None

    def __enter__(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        self.t0 = time.time()
        time.sleep(0.2)
        return self

    def mark(self):
        self.t_start = time.time()
        self.t_end = None

    def stop(self):
        self.t_end = time.time()

    def __exit__(self, *exc):
        if getattr(self, "t_end", None) is None:
            self.t_end = time.time()
        if self.proc:
            time.sleep(0.1)
            self.proc.terminate()
            self.proc.wait(timeout=5)
        self.file.flush()
        self.file.close()

    def summary(self) -> dict:
        try:
            lines = open(self.file.name).read().strip().splitlines()
        except OSError:
            lines = []
        finally:
            try:
                os.unlink(self.file.name)
            except OSError:
                pass
        samples = []
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                samples.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        window = [s for s in samples if self.t_start - 0.05 <= s[0] <= self.t_end + 0.05] or samples
        if not window:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in window for i, v in enumerate(s[3]) if v == "Active"})
        return {"sm_mhz": float(np.median([s[1] for s in window])),
                "sm_max_mhz": max(s[2] for s in window), "reasons": reasons,
                "samples": len(window)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_seed(workload_index: int, rank: int) -> int:
    """Seed of the batch a rank processes: rank 0 gets the workload's own seed
    (42 + index), every other rank an independent batch of the same shape."""
    return 42 + workload_index + 1000 * rank


def aggregate_gbs(bytes_per_rank: int, world: int, max_ms_per_step: float) -> float:
    """Whole-job bandwidth: the bytes all ranks moved over the slowest rank's time."""
    return world * bytes_per_rank / (max_ms_per_step * 1e-3) / 1e9


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ fd arm

def build_case(w, args, dev, rank, fd):
    """One workload's inputs on the device and the step bench.py times: an
    fd_decode call (or its paged / FP8 / INT4 / graph form) through the C ABI.
    Returns a dict with the step, its bytes and everything the timings need."""
    import ctypes

    import torch

    from workloads import make_inputs, to_fp8, to_int4, to_paged, to_paged_int4

    inp = make_inputs(w.index, seed=rank_seed(w.index, rank))
    B, Hq, Hkv, D = w.batch, w.num_qo_heads, w.num_kv_heads, w.head_dim
    ip_host = np.ascontiguousarray(inp["kv_indptr"].numpy().astype(np.int32))
    T = int(ip_host[-1])
    scale = inp["scale"]
    ip_dev = inp["kv_indptr"].to(dev)

    # Steps run back to back.  K/V of one copy of the inputs must be at least
    # twice the L2 size, so no step finds the previous step's keys in L2;
    # small workloads rotate through enough copies of their inputs.
    fp8 = args.kv_dtype == "fp8"
    int4 = args.kv_dtype == "int4"
    quant = fp8 or int4
    row_bytes = kv_row_bytes(args.kv_dtype, D)
    kv_bytes = 2 * T * Hkv * row_bytes
    copies = max(1, -(-2 * L2_BYTES // max(kv_bytes, 1)))
    paged = args.page_size > 0
    if fp8:     # the same keys quantised to E4M3 with per-KV-head scales
        f = to_fp8(inp)
        inp = dict(inp, k=f["k_fp8"], v=f["v_fp8"], k_scale=f["k_scale"], v_scale=f["v_scale"])
        k_scale_dev, v_scale_dev = f["k_scale"].to(dev), f["v_scale"].to(dev)
        del f
    if int4:    # the same keys quantised to INT4 with one scale per key row and KV head
        f = to_int4(inp)
        if paged:
            pgi = to_paged_int4(f, args.page_size, seed=13)
            k_scale_dev, v_scale_dev = pgi["k_scale_pages"].to(dev), pgi["v_scale_pages"].to(dev)
            del pgi
        else:
            k_scale_dev, v_scale_dev = f["k_scale_int4"].to(dev), f["v_scale_int4"].to(dev)
        inp = dict(inp, k=f["k_int4"], v=f["v_int4"], k_scale=f["k_scale_int4"],
                   v_scale=f["v_scale_int4"], int4=True)
        del f
    pg_ip = pg_last = None
    if paged:   # the same keys in a paged KV cache (scattered pages)
        pg = to_paged(inp, args.page_size, seed=13)
        bufs = [tuple(pg[x].to(dev) for x in ("q", "k_pages", "v_pages")) for _ in range(copies)]
        pg_ip = np.ascontiguousarray(pg["kv_page_indptr"].numpy().astype(np.int32))
        pg_last = np.ascontiguousarray(pg["kv_last_page_len"].numpy().astype(np.int32))
        pg_ip_dev = pg["kv_page_indptr"].to(dev)
        pg_last_dev = pg["kv_last_page_len"].to(dev)
        pg_idx_dev = pg["kv_page_indices"].to(dev)
        num_pages = pg["k_pages"].shape[0]
        del pg
    else:
        bufs = [tuple(inp[x].to(dev) for x in ("q", "k", "v")) for _ in range(copies)]

    info0 = (fd.plan_paged(B, Hq, Hkv, D, args.page_size, pg_ip, pg_last) if paged
             else fd.plan(B, Hq, Hkv, D, ip_host))
    rows = info0.num_partial_rows
    nb = step_bytes(B, Hq, Hkv, D, T, rows, row_bytes)
    o = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    ws = torch.zeros(info0.workspace_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    lib = fd.lib()
    P = ctypes.c_void_p
    sp = P(stream.cuda_stream)
    ipp = ip_host.ctypes.data_as(P)

    # One step = fd_decode (or fd_decode_paged) through the C ABI: host plan +
    # the split kernel, which also runs stage 2 in the last CTA of each group.
    # Arguments are marshalled once so the host stays ahead of the GPU.
    scales = (P(k_scale_dev.data_ptr()), P(v_scale_dev.data_ptr())) if quant else ()
    if paged:
        step_args = [(B, Hq, Hkv, D, args.page_size, num_pages, pg_ip.ctypes.data_as(P),
                      pg_last.ctypes.data_as(P), P(pg_ip_dev.data_ptr()), P(pg_last_dev.data_ptr()),
                      P(pg_idx_dev.data_ptr()), P(qc.data_ptr()), P(kc.data_ptr()), P(vc.data_ptr()),
                      *scales, ctypes.c_float(scale), P(o.data_ptr()), P(lse.data_ptr()),
                      P(ws.data_ptr()), ws.numel(), sp) for qc, kc, vc in bufs]
        step_name = ("fd_decode_paged_fp8" if fp8 else "fd_decode_paged_int4" if int4
                     else "fd_decode_paged")
        step_fn = getattr(lib, step_name)
    elif quant:
        step_args = [(B, Hq, Hkv, D, ipp, P(ip_dev.data_ptr()), P(qc.data_ptr()), P(kc.data_ptr()),
                      P(vc.data_ptr()), *scales, ctypes.c_float(scale), P(o.data_ptr()),
                      P(lse.data_ptr()), P(ws.data_ptr()), ws.numel(), sp) for qc, kc, vc in bufs]
        step_name = "fd_decode_fp8" if fp8 else "fd_decode_int4"
        step_fn = getattr(lib, step_name)
    else:
        step_args = [(B, Hq, Hkv, D, ipp, P(ip_dev.data_ptr()), P(qc.data_ptr()), P(kc.data_ptr()),
                      P(vc.data_ptr()), ctypes.c_float(scale), P(o.data_ptr()), P(lse.data_ptr()),
                      P(ws.data_ptr()), ws.numel(), sp) for qc, kc, vc in bufs]
        step_fn, step_name = lib.fd_decode, "fd_decode"

    def step(i):
        rc = step_fn(*step_args[i % copies])
        if rc != 0:
            raise fd.FdError(rc, step_name)

    # stage 1 alone (fd_decode_split) on the same inputs: a diagnostic of the
    # ragged bf16 path (the other paths have no separate stage-1 entry point)
    split = None
    if not (paged or quant or args.graph):
        ws_split = torch.zeros(fd.WORKSPACE_HEADER_BYTES, dtype=torch.uint8, device=dev)
        po = torch.empty((rows, D), dtype=torch.float32, device=dev)
        pl = torch.empty((rows,), dtype=torch.float32, device=dev)
        split_args = [(ctypes.byref(info0), P(qc.data_ptr()), P(kc.data_ptr()), P(vc.data_ptr()),
                       P(ip_dev.data_ptr()), ctypes.c_float(scale), P(po.data_ptr()),
                       P(pl.data_ptr()), P(ws_split.data_ptr()), ws_split.numel(), sp)
                      for qc, kc, vc in bufs]

        def split(i):
            rc = lib.fd_decode_split(*split_args[i % copies])
            if rc != 0:
                raise fd.FdError(rc, "fd_decode_split")

    info_g = None
    step_calls = 1   # steps per step() call
    if args.graph:
        # GRAPH_STEPS fd_decode_graph steps per input copy captured in one CUDA
        # graph (device-side plan for a capacity of exactly this batch's keys),
        # as an engine captures a decode step's many attention calls; the
        # launches inside a graph keep their programmatic serialisation.
        if paged or quant:
            raise SystemExit("--graph times the ragged bf16 path")
        info_g = fd.plan_graph(B, Hq, Hkv, D, T)
        ws_g = torch.zeros(info_g.workspace_bytes, dtype=torch.uint8, device=dev)
        cap = torch.cuda.Stream(dev)
        graphs = []
        for qc, kc, vc in bufs:
            cap.wait_stream(stream)
            with torch.cuda.stream(cap):   # one call outside the capture
                fd.decode_graph(info_g, qc, kc, vc, ip_dev, scale, o, lse, ws_g, stream=cap)
            stream.wait_stream(cap)
            torch.cuda.synchronize(dev)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                for _ in range(GRAPH_STEPS):
                    fd.decode_graph(info_g, qc, kc, vc, ip_dev, scale, o, lse, ws_g,
                                    stream=torch.cuda.current_stream(dev))
            graphs.append(g)
        ws = ws_g
        step_name = "fd_decode_graph"
        step_calls = GRAPH_STEPS

        def step(i):   # GRAPH_STEPS steps
            graphs[i % copies].replay()

    # one item per CTA when the plan fits a wave of resident CTAs, else persistent
    work = info_g.num_work if args.graph else info0.num_work   # the graph plan's capacity
    persistent = work > info0.num_sms * info0.ctas_per_sm
    kernel = ("split_kv_persistent_kernel" if persistent else "split_kv_kernel") + \
        ("<fp8>" if fp8 else "<int4>" if int4 else "<bf16>")
    # stage 2 runs inside the split kernel; the merge kernel is launched only
    # when some request has no keys
    any_empty = bool(np.any(np.diff(ip_host) == 0))
    launches_per_step = int(info0.num_work > 0) + int(any_empty)
    # every device buffer the marshalled arguments point at stays referenced
    # here for as long as the case lives
    here = dict(locals())
    keep = [here[n] for n in ("k_scale_dev", "v_scale_dev", "pg_ip_dev", "pg_last_dev", "pg_idx_dev",
                              "ws_split", "po", "pl", "ws_g") if here.get(n) is not None]
    return dict(w=w, inp=inp, ip_host=ip_host, ip_dev=ip_dev, bufs=bufs, copies=copies, keep=keep,
                info=info0, nb=nb, o=o, lse=lse, ws=ws, stream=stream, step=step, split=split,
                step_name=step_name, step_calls=step_calls, kernel=kernel,
                launches_per_step=launches_per_step, paged=paged, fp8=fp8, int4=int4, T=T)


def measure_case(case, args, world, dev, flush, clocks=None, n_flushed=100) -> dict:
    """Time one workload's step: W warm-up steps; then the K-step loop, repeated
    back to back (one pair of CUDA events around all of it) until the timed
    region lasts at least --min-timed-ms; stage 1 alone; single steps after an
    L2 flush."""
    import torch

    import split_kv_flashdecoding_gb300 as fd

    stream, step, calls = case["stream"], case["step"], case["step_calls"]
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    if fd.get_device_status(case["ws"]) != 0:
        raise RuntimeError("device status set during warm-up")
    K = max(1, args.steps // calls) * calls
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    # how many back-to-back repeats of the K-step loop fill the timed region
    n_est = max(1, min(K, 50) // calls)
    torch.cuda._sleep(1_000_000)
    ev0.record(stream)
    for i in range(n_est):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    est_ms = ev0.elapsed_time(ev1) / (n_est * calls)
    rounds = max(1, math.ceil(args.min_timed_ms / max(K * est_ms, 1e-6)))
    rounds = int(max_over_ranks(float(rounds), world, dev))

    barrier(world)
    torch.cuda.synchronize(dev)
    if clocks is not None:
        clocks.mark()
    torch.cuda._sleep(2_000_000)        # lets the host queue steps ahead of the GPU
    t_wall0 = time.perf_counter()
    ev0.record(stream)
    for i in range(rounds * K // calls):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall0
    if clocks is not None:
        clocks.stop()
    barrier(world)
    status = fd.get_device_status(case["ws"])
    if status != 0:
        raise RuntimeError(f"device status {fd.status_string(status)}")
    timed_ms = ev0.elapsed_time(ev1)
    ms = max_over_ranks(timed_ms / (rounds * K), world, dev)

    # stage 1 alone, back to back on the same stream (ragged bf16 only)
    split_ms = None
    if case["split"] is not None:
        n_split = 500
        torch.cuda._sleep(2_000_000)
        ev0.record(stream)
        for i in range(n_split):
            case["split"](i)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        split_ms = ev0.elapsed_time(ev1) / n_split

    # The same step timed one at a time (each includes its launch latency and
    # about 2 us of event overhead) after two kinds of L2 flush: writing a
    # 1 GiB buffer (L2 left full of dirty lines, whose write-back to HBM then
    # shares the step's DRAM time), and reading one (L2 full of clean lines of
    # other data, as after a kernel that mostly reads, e.g. a GEMM).
    def single_steps(flush_op):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n_flushed)]
        for i in range(n_flushed):
            flush_op(i)
            evs[i][0].record(stream)
            step(0)
            evs[i][1].record(stream)
        torch.cuda.synchronize(dev)
        return np.array([a.elapsed_time(b) for a, b in evs]) / calls

    flushed_ms = single_steps(lambda i: flush.fill_(float(i)))
    clean_ms = single_steps(lambda i: flush.sum())
    status = fd.get_device_status(case["ws"])
    if status != 0:
        raise RuntimeError(f"device status {fd.status_string(status)} in the single steps")
    return dict(K=K, rounds=rounds, ms=ms, timed_ms=timed_ms, wall_s=t_wall, split_ms=split_ms,
                flushed_ms=flushed_ms, clean_ms=clean_ms,
                launches=rounds * K * case["launches_per_step"])


def workload_summary(case, m, world, peak) -> dict:
    """The per-workload entry of the JSON line."""
    nb, info = case["nb"], case["info"]
    gbs = aggregate_gbs(nb["step"], world, m["ms"])
    return {
        "us_per_step": round(m["ms"] * 1e3, 2),
        "gbs": round(gbs, 1),
        "frac_of_measured": round(gbs / world / peak, 4),
        "frac_of_nominal_8tbs": round(gbs / world / NOMINAL_HBM_GBS, 4),
        "split_only_us": None if m["split_ms"] is None else round(m["split_ms"] * 1e3, 2),
        "step_us_after_l2_flush_p50": round(float(np.percentile(m["flushed_ms"], 50)) * 1e3, 2),
        "step_us_after_l2_read_flush_p50": round(float(np.percentile(m["clean_ms"], 50)) * 1e3, 2),
        "timed_steps": m["rounds"] * m["K"],
        "timed_region_ms": round(m["timed_ms"], 1),
        "algorithmic_bytes_per_step": nb["step"],
        "total_tokens": case["T"], "chunk": info.chunk, "splits": info.total_splits,
        "ctas": info.num_work, "kernel": case["kernel"],
        # a CUDA-graph replay runs step_calls decode steps: the flushed figures
        # are one replay after one flush, divided by step_calls (only its first
        # step starts from the flushed L2)
        "flushed_steps_per_measure": case["step_calls"],
    }


def e2e_measure(case, args, world, dev, flush) -> dict:
    """End to end through the public API with host buffers: pinned H2D of the
    step's inputs, fd_decode, D2H of O and LSE, all inside the events."""
    import torch

    import split_kv_flashdecoding_gb300 as fd

    inp, w, info, stream = case["inp"], case["w"], case["info"], case["stream"]
    B, Hq, D = w.batch, w.num_qo_heads, w.head_dim
    q_h, k_h, v_h = (inp[x].pin_memory() for x in ("q", "k", "v"))
    ip_h = inp["kv_indptr"].pin_memory()
    o_h = torch.empty((B, Hq, D), dtype=torch.float32).pin_memory()
    l_h = torch.empty((B, Hq), dtype=torch.float32).pin_memory()
    wsd = torch.zeros(info.workspace_bytes, dtype=torch.uint8, device=dev)
    e2e_steps = max(3, min(args.steps, 20))
    q, k, v = case["bufs"][0]
    o, lse, ip_dev = case["o"], case["lse"], case["ip_dev"]
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(e2e_steps)]
    for i in range(e2e_steps + 2):
        flush.fill_(float(i))
        if i >= 2:
            evs[i - 2][0].record(stream)
        q.copy_(q_h, non_blocking=True)
        k.copy_(k_h, non_blocking=True)
        v.copy_(v_h, non_blocking=True)
        ip_dev.copy_(ip_h, non_blocking=True)
        fd.decode(q, k, v, case["ip_host"], ip_dev, inp["scale"], o=o, lse=lse, workspace=wsd,
                  stream=stream)
        o_h.copy_(o, non_blocking=True)
        l_h.copy_(lse, non_blocking=True)
        if i >= 2:
            evs[i - 2][1].record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in evs])), world, dev)
    h2d = sum(t.numel() * t.element_size() for t in (q_h, k_h, v_h, ip_h))
    d2h = sum(t.numel() * t.element_size() for t in (o_h, l_h))
    return {"value": round(world * case["nb"]["step"] / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


def run_fd(args, world, rank, local) -> dict | None:
    import torch

    import split_kv_flashdecoding_gb300 as fd

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    peak, peak_kind = measured_peaks()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    w = workload(args.workload)

    # the headline workload: timed step with clocks, e2e, the CPU baseline
    case = build_case(w, args, dev, rank, fd)
    with ClockSampler(local) as clocks:
        m = measure_case(case, args, world, dev, flush, clocks=clocks)
    summary = workload_summary(case, m, world, peak)
    e2e = None
    if not args.no_e2e and not (case["paged"] or case["fp8"] or case["int4"] or args.graph):
        e2e = e2e_measure(case, args, world, dev, flush)
    cpu = None
    if not args.no_cpu_baseline and world == 1 and rank == 0:
        cpu = cpu_baseline(w, case["inp"], case["nb"]["step"], budget_s=args.cpu_budget)
    info, nb, ms = case["info"], case["nb"], m["ms"]
    launches = m["launches"]
    del case
    torch.cuda.empty_cache()

    # every other workload, the same step kind, each timed the same way
    per_workload = {w.name: summary}
    if not args.no_per_workload:
        for other in WORKLOADS:
            if other.name == w.name:
                continue
            c = build_case(other, args, dev, rank, fd)
            mo = measure_case(c, args, world, dev, flush, n_flushed=50)
            per_workload[other.name] = workload_summary(c, mo, world, peak)
            del c
            torch.cuda.empty_cache()
    per_workload = {x.name: per_workload[x.name] for x in WORKLOADS if x.name in per_workload}

    if rank != 0:
        return None
    gbs = aggregate_gbs(nb["step"], world, ms)
    # The dominant kernel is the one the step launches (the split kernel, with
    # stage 2 fused): its launches are the timed steps, back to back.
    achieved = nb["step"] / (ms * 1e-3) / 1e9
    traffic = None
    if not (args.kv_dtype != "bf16" or args.page_size or args.graph):
        traffic = profiled_traffic(w.name)
    line = {
        "metric": METRIC,
        "value": round(gbs, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": m["K"],
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "us_per_step": round(ms * 1e3, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("bf16 q, fp8 e4m3 K/V widened to f16, fp32 accumulate/out" if args.kv_dtype == "fp8"
                  else "bf16 q, int4 K/V widened to bf16, fp32 scales/accumulate/out"
                  if args.kv_dtype == "int4" else "bf16 in, fp32 accumulate/out"),
        "data": "synthetic (seeded, see workloads/)",
        "config": {"workload": w.name, "description": w.description, "batch": w.batch,
                   "num_qo_heads": w.num_qo_heads, "num_kv_heads": w.num_kv_heads,
                   "head_dim": w.head_dim, "total_tokens": summary["total_tokens"],
                   "chunk": info.chunk, "splits": info.total_splits, "ctas": info.num_work,
                   "ctas_per_sm": info.ctas_per_sm, "num_sms": info.num_sms,
                   "l2": ("steps back to back; inputs larger than L2 (K/V of each step "
                          ">= 2x L2, input copies rotated when a workload is smaller)"),
                   "timed_rounds": m["rounds"],
                   "timed_steps": m["rounds"] * m["K"],
                   "timed_region_ms": round(m["timed_ms"], 1),
                   "timing": (f"the {m['K']}-step loop repeated {m['rounds']}x back to back "
                              "inside one pair of CUDA events, so the timed region lasts at "
                              f"least {args.min_timed_ms:g} ms"),
                   "algorithmic_bytes_per_step": nb["step"],
                   "frac_of_nominal_8tbs": round(gbs / world / NOMINAL_HBM_GBS, 4),
                   "split_only_us": summary["split_only_us"],
                   "step_us_after_l2_flush_p10_p50_p90": [
                       round(float(np.percentile(m["flushed_ms"], p)) * 1e3, 2) for p in (10, 50, 90)],
                   "step_us_after_l2_read_flush_p10_p50_p90": [
                       round(float(np.percentile(m["clean_ms"], p)) * 1e3, 2) for p in (10, 50, 90)],
                   "single_step_note": ("one step at a time after a 1 GiB L2 flush, launch latency and "
                                        "events included: a write flush leaves L2 full of dirty lines "
                                        "whose write-back shares the step's DRAM time; a read flush "
                                        "leaves it full of clean lines of other data"),
                   "wall_s": round(m["wall_s"], 3),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "kv_layout": (f"paged, page_size {args.page_size}, pages scattered in a pool"
                                 if args.page_size else "ragged packed"),
                   "kv_dtype": ("fp8 e4m3, one fp32 scale per KV head for K and for V"
                                if args.kv_dtype == "fp8" else
                                "int4 (two's complement, 2 per byte), one fp32 scale per key row "
                                "and KV head for K and for V" if args.kv_dtype == "int4" else "bf16"),
                   "launch": ("CUDA graph replay of fd_decode_graph (device-side plan)"
                              if args.graph else "C ABI call per step (host plan)")},
        "roofline": {"bound": "hbm", "kernel": summary["kernel"], "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
                     "algorithmic_bytes_per_launch": nb["step"],
                     "launch_us": round(ms * 1e3, 2),
                     "how": ("the step's one kernel (stage 1 with stage 2 fused): algorithmic "
                             "bytes per launch / its average launch time over the timed steps"),
                     "traffic": traffic,
                     "split_only": None if m["split_ms"] is None else {
                         "kernel": "fd_decode_split (stage 1 alone, diagnostic)",
                         "us": round(m["split_ms"] * 1e3, 2),
                         "achieved": round(nb["split"] / (m["split_ms"] * 1e-3) / 1e9, 1),
                         "frac": round(nb["split"] / (m["split_ms"] * 1e-3) / 1e9 / peak, 4)}},
        "per_workload": per_workload,
        "gpu_launches": launches,
        "clocks": clocks.summary(),
        "e2e": e2e,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    return line


# ------------------------------------------------------- oracle (CPU) timing

def _oracle_rows(inp, rows, threads) -> float:
    import oracle
    t0 = time.perf_counter()
    if inp.get("int4"):    # INT4 K/V: the oracle dequantises, then decodes
        oracle.decode_int4(inp["q"], inp["k"], inp["v"], inp["k_scale"], inp["v_scale"],
                           inp["kv_indptr"], inp["scale"], rows=rows, threads=threads)
    elif "k_scale" in inp:   # FP8 K/V: the oracle dequantises, then decodes
        oracle.decode_fp8(inp["q"], inp["k"], inp["v"], inp["k_scale"], inp["v_scale"],
                          inp["kv_indptr"], inp["scale"], rows=rows, threads=threads)
    else:
        oracle.decode(inp["q"], inp["k"], inp["v"], inp["kv_indptr"], inp["scale"], rows=rows,
                      threads=threads)
    return time.perf_counter() - t0


def _row_cost(w, inp, cores) -> float:
    """Core-seconds of oracle work per (request, query head) row."""
    rows = np.random.default_rng(1).permutation(w.batch * w.num_qo_heads)[:cores]
    return _oracle_rows(inp, rows, cores) / len(rows) * cores


def cpu_baseline(w, inp, step_bytes_total, budget_s=10.0) -> dict:
    """Time the fp64 oracle on the host cores over a bounded sample of the
    step's (request, query head) rows and extrapolate to one full step."""
    cores = max(1, len(os.sched_getaffinity(0)))
    all_rows = w.batch * w.num_qo_heads
    per_row = _row_cost(w, inp, cores)
    n = int(min(all_rows, max(min(cores, all_rows), budget_s * cores / max(per_row, 1e-9))))
    rows = np.random.default_rng(0).permutation(all_rows)[:n]
    # repeat a sample that finishes quickly so the timed span is at least ~1 s
    reps, t = 0, 0.0
    while reps == 0 or (t < min(1.0, budget_s) and reps < 100):
        t += _oracle_rows(inp, rows, cores)
        reps += 1
    t /= reps
    step_s = t * all_rows / n
    return {"value": round(step_bytes_total / step_s / 1e9, 4), "unit": "GB/s",
            "us_per_step": round(step_s * 1e6, 1), "cores": cores, "kind": "oracle",
            "sample": f"{n} of {all_rows} (request, query-head) rows of {w.name}, "
                      f"fp64 C oracle, {t:.3f} s wall per pass ({reps} passes) on {cores} "
                      f"threads, extrapolated to the full step"}


def run_reference(args, world, rank) -> dict | None:
    """The oracle arm: each timed step runs the fp64 oracle on a fixed sample
    of the step's rows on the host cores (sized so the whole run takes about a
    minute and a half) and is extrapolated to the full step."""
    if rank != 0:
        return None
    from workloads import make_inputs
    w = workload(args.workload)
    inp = make_inputs(w.index)
    B, Hq, Hkv, D = w.batch, w.num_qo_heads, w.num_kv_heads, w.head_dim
    T = int(inp["kv_indptr"][-1])
    # the fd arm's step bytes: the same plan's partials, counted on the host
    num_sms, sm_source = device_sm_count()
    rows_partial = plan_partial_rows(inp["lengths"], Hq, Hkv, num_sms)
    nb = step_bytes(B, Hq, Hkv, D, T, rows_partial)
    cores = max(1, len(os.sched_getaffinity(0)))
    all_rows = B * Hq
    per_row = _row_cost(w, inp, cores)
    per_step_budget = max(0.0, 90.0 / max(args.steps, 1))
    n = int(min(all_rows, max(1, per_step_budget * cores / max(per_row, 1e-9))))
    threads = min(cores, n)
    sample = np.random.default_rng(0).permutation(all_rows)[:n]
    for _ in range(args.warmup):
        _oracle_rows(inp, sample[:1], 1)
    times = [_oracle_rows(inp, sample, threads) for _ in range(args.steps)]
    step_s = float(np.mean(times)) * all_rows / n
    value = nb["step"] / step_s / 1e9
    return {
        "metric": METRIC, "impl": "reference", "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_s * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, see workloads/)",
        "config": {"workload": w.name, "description": w.description,
                   "algorithmic_bytes_per_step": nb["step"],
                   "bytes_counted_as": (f"the fd arm's step bytes (q + K + V + O + LSE + partials "
                                        f"of its plan for {num_sms} SMs, {sm_source})")},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"{n} of {all_rows} (request, query-head) rows of {w.name} "
                                   f"per step on {threads} threads, extrapolated to the full step"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=[x.name for x in WORKLOADS])
    ap.add_argument("--impl", default="fd", choices=["fd", "reference"])
    ap.add_argument("--graph", action="store_true",
                    help="time CUDA-graph replays of fd_decode_graph (device-side plan)")
    ap.add_argument("--kv-dtype", choices=["bf16", "fp8", "int4"], default="bf16",
                    help="fp8: the same keys quantised to E4M3 (fd_decode_fp8); int4: to packed "
                         "four-bit codes with per-row scales (fd_decode_int4)")
    ap.add_argument("--page-size", type=int, default=0,
                    help="time fd_decode_paged on the same keys laid out as a paged KV cache")
    ap.add_argument("--min-timed-ms", type=float, default=200.0,
                    help="the K-step loop is repeated back to back until the timed region "
                         "lasts at least this long")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="time only --workload (default: every workload, the same step kind)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle CPU work per timed sample")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        line = run_reference(args, world, rank)
    else:
        line = run_fd(args, world, rank, local)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and args.impl == "fd":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
