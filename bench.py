#!/usr/bin/env python
"""Benchmark of the fused residual-add + RMSNorm + FP4 quantization path.

One step = one call of fp4_add_rmsnorm_quant (the whole hot path: add,
RMSNorm, scales, codes, both writes) over one batch of the workload, inputs
resident in HBM.  The default workload is M=8192 x H=7168 bf16, MXFP4 with
tiled scales and 1% x50 outlier columns: 383.5 MB of algorithmic traffic per
call, three times the 129 MB L2, so no L2 flush is needed between steps.
Consecutive steps alternate between the input x and -x so the in-place
residual stays bounded (both copies are read the same way).

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "fused add+RMSNorm+FP4-quant HBM GB/s and % of GB300 HBM roofline (rows/s)"
DEFAULT_WORKLOAD = workloads.C3.name
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--rows", type=int, default=None,
                    help="override the workload's M (smaller cases for profiling)")
    ap.add_argument("--op", choices=["fused", "quantize", "gemm", "chain"], default="fused",
                    help="fused add+RMSNorm+quantize (default), the standalone quantize, "
                         "the NVFP4 GEMM that consumes them (--gemm picks the shape), or the "
                         "chain fused op -> GEMM on the rows of the GEMM's A operand")
    ap.add_argument("--gemm", default="G4_M8192_N7168_K7168",
                    help="GEMM workload for --op gemm")
    ap.add_argument("--gemm-format", choices=["nvfp4", "mxfp4"], default="nvfp4",
                    help="GEMM operand format (E4M3 per 16 or UE8M0 per 32 codes)")
    ap.add_argument("--gemm-variant", type=int, default=-1,
                    help="GEMM tile schedule: -1 automatic, 0/1 = one CTA per 128x128/128x256 "
                         "tile, 2/3 = persistent over 128x128/128x256 tiles, 4 = split K")
    ap.add_argument("--global-scale", type=float, default=None,
                    help="pass this global scale as a device scalar (E4M3 formats)")
    ap.add_argument("--format", default=None, help="override the workload's format")
    ap.add_argument("--y-out", action="store_true",
                    help="also write y (the normalised rows, input dtype): +2H bytes per row")
    ap.add_argument("--no-pdl", action="store_true",
                    help="launch the fused calls without programmatic dependent launch")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip timing the other large workloads after the headline")
    ap.add_argument("--config-steps", type=int, default=50,
                    help="timed calls per workload of the 'configs' list")
    ap.add_argument("--clock-seconds", type=float, default=1.0,
                    help="length of the sustained loop whose SM clocks the line reports")
    ap.add_argument("--cpu-cores", type=int, default=0,
                    help="host cores for the oracle baseline (0 = all)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# environment helpers
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# Sources each measured kernel is built from (its host launch code included):
# a committed ncu summary applies only while these files are unchanged.
KERNEL_SOURCES = {
    "fused": ("api.cu", "async_copy.cuh", "fp4q_device.cuh", "fp4q_launch.h", "fused_bf16.cu",
              "fused_common.cuh", "fused_direct.cuh", "fused_fp16.cu", "fused_launch.cuh",
              "fused_tma.cuh", "debug_checks.h"),
    "quantize": ("api.cu", "fp4q_device.cuh", "fp4q_launch.h", "quantize.cu"),
    "gemm": ("async_copy.cuh", "fp4q_device.cuh", "gemm_api.cu", "gemm_launch.h", "gemm_nvfp4.cu",
             "tcgen05.cuh"),
}


def kernel_source_sha(op: str = "fused") -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "rmsnorm_fp4_quant_gb300", "csrc")
    for name in sorted(KERNEL_SOURCES[op]):
        h.update(name.encode())
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()


def gemm_profile_key(workload_name: str, fmt: str, kernel: str, tile_n: int) -> str:
    """The `workload:` key of a GEMM capture: shape, operand format, kernel
    and output-tile width (the persistent kernel runs 128- or 256-wide)."""
    return f"{workload_name}_{fmt}_{kernel}_n{tile_n}"


def recorded_traffic(workload_name: str, op: str = "fused"):
    """dram bytes per launch from a committed ncu summary whose kernel-source
    hash matches the current sources; None otherwise."""
    sha = kernel_source_sha(op)
    for p in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        text = open(p).read()
        m_w = re.search(r"^workload:\s*(\S+)", text, re.M)
        m_s = re.search(r"^source_sha256:\s*([0-9a-f]{64})", text, re.M)
        m_t = re.search(r"^dram_bytes_per_launch:\s*([0-9]+)", text, re.M)
        if m_w and m_s and m_t and m_w.group(1) == workload_name and m_s.group(1) == sha:
            return int(m_t.group(1)), os.path.relpath(p, ROOT)
    return None, None


class ClockSampler:
    """nvidia-smi sampled every 100 ms in a background process; each line is
    stamped on arrival so samples can be matched to the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.samples = []
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if gpu_id:
            cmd += ["-i", gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        pad = max(0.0, 0.35 - (t1 - t0) / 2)
        sel = [p for (t, p) in self.samples if t0 - pad <= t <= t1 + pad]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[0]) for p in sel if num(p[0]) is not None]
        mx = [num(p[1]) for p in sel if num(p[1]) is not None]
        reasons = set()
        for p in sel:
            for name, val in zip(self.NAMES, p[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        pw = [num(p[2]) for p in sel if num(p[2]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sel),
                "power_w_max": max(pw) if pw else None}


def gpu_smi_id(torch, dev):
    try:
        u = torch.cuda.get_device_properties(dev).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        return None


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------
def oracle_rows_timing(wl, nrows: int, row0: int = 0):
    """Time the oracle (as it stands) on rows [row0, row0 + nrows) of `wl`."""
    import oracle
    x = workloads.make_rows(wl, "x", row0, row0 + nrows).float().numpy()
    r = workloads.make_rows(wl, "r", row0, row0 + nrows).float().numpy()
    w = workloads.make_weight(wl).float().numpy()
    t = time.perf_counter()
    oracle.add_rmsnorm_fp4_quant(x, r, w, wl.eps, wl.dtype, wl.fmt, wl.sf_layout)
    return time.perf_counter() - t


def cpu_rows_for(wl, seconds: float) -> int:
    oracle_rows_timing(wl, 8)                       # warm the allocator
    probe = min(wl.M, 32)
    dt = oracle_rows_timing(wl, probe)
    rows = int(probe * seconds / max(dt, 1e-6))
    return max(1, min(wl.M, rows))


def _oracle_worker(args):
    """One task of the row-partitioned oracle: draw its rows, wait for the
    other processes, time the oracle on them."""
    wl, row0, row1, barrier = args
    import oracle
    x = workloads.make_rows(wl, "x", row0, row1).float().numpy()
    r = workloads.make_rows(wl, "r", row0, row1).float().numpy()
    w = workloads.make_weight(wl).float().numpy()
    barrier.wait(600)
    t0 = time.time()
    oracle.add_rmsnorm_fp4_quant(x, r, w, wl.eps, wl.dtype, wl.fmt, wl.sf_layout)
    return t0, time.time()


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OraclePool:
    """The oracle row-partitioned over `cores` spawned processes, each
    single-threaded numpy on one row block.  Every call hands each process
    exactly one block (each task waits at a barrier of `cores` parties, so no
    process can take a second), and times from the first start to the last
    finish, inputs drawn beforehand."""

    def __init__(self, cores: int):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        self.cores = max(1, cores)
        keep = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS")}
        os.environ["OMP_NUM_THREADS"] = "1"
        os.environ["OPENBLAS_NUM_THREADS"] = "1"
        try:
            self.mgr = ctx.Manager()
            self.barrier = self.mgr.Barrier(self.cores)
            self.pool = ctx.Pool(self.cores)
        finally:
            for k, v in keep.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    def time_rows(self, wl, nrows: int, row0: int = 0) -> float:
        n = self.cores
        nrows = max(n, nrows)
        b = [row0 + nrows * i // n for i in range(n + 1)]
        spans = self.pool.map(_oracle_worker, [(wl, b[i], b[i + 1], self.barrier)
                                               for i in range(n)], chunksize=1)
        return max(t1 for _, t1 in spans) - min(t0 for t0, _ in spans)

    def close(self):
        self.pool.close()
        self.pool.join()
        self.mgr.shutdown()


def cpu_baseline(wl, seconds: float, cores: int = 0):
    """The oracle as it stands on this host: row-partitioned over all cores
    (the reported value), and single-threaded (a second field)."""
    rows = cpu_rows_for(wl, seconds)
    dt1 = oracle_rows_timing(wl, rows)
    single = {"value": round(wl.with_shape(rows).algorithmic_bytes() / dt1 / 1e9, 4),
              "unit": "GB/s", "cores": 1, "rows_per_s": round(rows / dt1, 2),
              "sample": f"first {rows} of {wl.M} rows of {wl.name}, numpy oracle, one process, "
                        f"{dt1:.1f} s"}
    n = min(cores or host_cores(), wl.M)
    # as many rows as the cores finish in about the same wall time
    prow = min(wl.M, max(n, int(rows * n)))
    pool = OraclePool(n)
    try:
        pool.time_rows(wl, n)                     # first task of each process: imports
        dtn = pool.time_rows(wl, prow)
    finally:
        pool.close()
    return {"value": round(wl.with_shape(prow).algorithmic_bytes() / dtn / 1e9, 4),
            "unit": "GB/s", "cores": n, "kind": "oracle",
            "sample": f"first {prow} of {wl.M} rows of {wl.name}, numpy oracle row-partitioned "
                      f"over {n} spawned processes (one per host core, single-threaded), "
                      f"{dtn:.2f} s wall from first start to last finish",
            "rows_per_s": round(prow / dtn, 2), "single_core": single}


def run_reference(args, wl):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    cores = min(args.cpu_cores or host_cores(), wl.M)
    # a step: the oracle on a row sample that the cores finish in about 2 s
    per_step = min(wl.M, max(cores, cpu_rows_for(wl, 2.0) * cores))
    pool = OraclePool(cores)
    try:
        for _ in range(max(1, min(args.warmup, 3))):
            pool.time_rows(wl, cores)
        times = [pool.time_rows(wl, per_step, row0=(i * per_step) % max(1, wl.M - per_step + 1))
                 for i in range(args.steps)]
    finally:
        pool.close()
    bytes_ = wl.with_shape(per_step).algorithmic_bytes()
    tot = sum(times)
    val = bytes_ * len(times) / tot / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot / len(times) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name, "M": wl.M, "H": wl.H, "format": wl.fmt,
                   "sf_layout": wl.sf_layout, "io_dtype": wl.dtype,
                   "sample_rows_per_step": per_step},
        "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"{per_step} of {wl.M} rows of {wl.name} per step, numpy "
                                   f"oracle row-partitioned over {cores} spawned processes"},
        "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "rows_per_s": round(per_step * len(times) / tot, 2),
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def run_ours(args, wl):
    import torch
    import torch.distributed as dist

    import rmsnorm_fp4_quant_gb300 as fq

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    L = fq.lib()
    fmt = {"nvfp4": fq.FP4_NVFP4, "mxfp4": fq.FP4_MXFP4, "e4m3b32": fq.FP4_E4M3_B32}[wl.fmt]
    lay = {"rowmajor": fq.FP4_SF_ROWMAJOR, "swizzled": fq.FP4_SF_SWIZZLED,
           "both": fq.FP4_SF_BOTH}[wl.sf_layout]
    dt = fq.FP4_DT_BF16 if wl.dtype == "bf16" else fq.FP4_DT_FP16

    # each rank owns an independent batch (weak scaling, no data exchange)
    import dataclasses
    wl_r = dataclasses.replace(wl, seed=wl.seed + 1000 * rank)
    x, r, w = workloads.make_inputs(wl_r, dev)
    xneg = -x
    M, H = wl.M, wl.H
    nb = H // wl.block
    packed = torch.empty(M, H // 2, dtype=torch.uint8, device=dev)
    sf = torch.empty(max(1, fq.fp4_sf_size_bytes(M, H, fmt, lay)), dtype=torch.uint8, device=dev)
    sf_rm = torch.empty(M * nb, dtype=torch.uint8, device=dev) if lay == fq.FP4_SF_BOTH else None
    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream
    ptrs = [x.data_ptr(), xneg.data_ptr()]
    rp, wp, pp, sp = r.data_ptr(), w.data_ptr(), packed.data_ptr(), sf.data_ptr()
    s2 = sf_rm.data_ptr() if sf_rm is not None else None
    eps = float(wl.eps)
    gs_t = None
    if args.global_scale is not None:
        gs_t = torch.tensor([args.global_scale], dtype=torch.float32, device=dev)
    gp = gs_t.data_ptr() if gs_t is not None else None
    y_t, yp = None, None
    # consecutive calls are programmatic dependents of the call before (the
    # way a serving stream chains its kernels): each launch is scheduled
    # during the previous call's last CTAs and waits for its results
    pdl_on = 0 if args.no_pdl else 1
    if args.op == "quantize":
        qcall = L.fp4_quantize

        def step(i, pdl=pdl_on):
            st = qcall(ptrs[i & 1], gp, M, H, dt, fmt, lay, pp, sp, s2, pdl, sh)
            if st != 0:
                raise fq.Fp4Error(st, "fp4_quantize")
    else:
        call = L.fp4_add_rmsnorm_quant_ex
        y_t = torch.empty(M, H, dtype=x.dtype, device=dev) if args.y_out else None
        yp = y_t.data_ptr() if y_t is not None else None

        def step(i, pdl=pdl_on):
            st = call(ptrs[i & 1], H, rp, H, wp, gp, eps, M, H, dt, fmt, lay, pp, sp, s2, yp,
                      None, pdl, sh)
            if st != 0:
                raise fq.Fp4Error(st, "fp4_add_rmsnorm_quant")

    # Workloads smaller than twice the L2 (C1, C2, short batches): rotate
    # through enough copies of the inputs and outputs that one pass touches
    # more than twice the L2, and replay the pass as a CUDA graph, so neither
    # warm caches nor host launch cost enter the number.  Each copy is called
    # with x and then -x in a pass, so its residual returns to where it was.
    alg_step = wl.algorithmic_bytes(args.op) + (2 * M * H if args.y_out and args.op == "fused"
                                                else 0)
    rot = 1 if alg_step >= 2 * L2_BYTES else min(256, -(-2 * L2_BYTES // alg_step))
    graph = None
    if rot > 1:
        copies = []
        for _ in range(rot):
            c = {"x": x.clone(), "xn": xneg.clone(), "r": r.clone(), "p": torch.empty_like(packed),
                 "s": torch.empty_like(sf),
                 "s2": torch.empty_like(sf_rm) if sf_rm is not None else None,
                 "y": torch.empty(M, H, dtype=x.dtype, device=dev) if args.y_out else None}
            copies.append(c)

        def step_copy(c, xs):
            s2p = c["s2"].data_ptr() if c["s2"] is not None else None
            if args.op == "quantize":
                st = L.fp4_quantize(xs.data_ptr(), gp, M, H, dt, fmt, lay, c["p"].data_ptr(),
                                    c["s"].data_ptr(), s2p, pdl_on, sh)
            else:
                st = L.fp4_add_rmsnorm_quant_ex(
                    xs.data_ptr(), H, c["r"].data_ptr(), H, wp, gp, eps, M, H, dt, fmt, lay,
                    c["p"].data_ptr(), c["s"].data_ptr(), s2p,
                    c["y"].data_ptr() if c["y"] is not None else None, None, pdl_on, sh)
            if st != 0:
                raise fq.Fp4Error(st, "graph step")

        def one_pass():
            for c in copies:
                step_copy(c, c["x"])
            for c in copies:
                step_copy(c, c["xn"])

        torch.cuda.synchronize(dev)       # the copies were made on the default stream
        with torch.cuda.stream(stream):
            one_pass()
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                one_pass()

    torch.cuda.synchronize(dev)
    sampler = ClockSampler(gpu_smi_id(torch, dev)) if rank == 0 else None
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            if graph is None:
                step(i)
        if graph is not None:
            for _ in range(3):
                graph.replay()
    stream.synchronize()

    # Timed region: K steps back to back on one stream between two events.  A
    # step is exactly one launch of the fused kernel, so the mean launch
    # duration is the region's time / K (per-launch events would add their own
    # gaps between launches).  Per-launch event pairs are taken afterwards on
    # a short separate loop for the spread.
    K = args.steps if graph is None else -(-args.steps // (2 * rot)) * 2 * rot
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    with torch.cuda.stream(stream):
        t_start.record(stream)
        if graph is None:
            for i in range(K):
                step(i)
        else:
            for _ in range(K // (2 * rot)):
                graph.replay()
        t_end.record(stream)
    stream.synchronize()
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    if world > 1:
        dist.barrier()
    total_ms = t_start.elapsed_time(t_end)
    n_ev = min(K, 200)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n_ev)]
    with torch.cuda.stream(stream):
        for i in range(n_ev):
            ev[i][0].record(stream)
            step(i)
            ev[i][1].record(stream)
    stream.synchronize()
    kern_ms = [a.elapsed_time(b) for a, b in ev]
    # the same K calls without programmatic dependent launch (reported beside)
    no_pdl_ms = None
    if graph is None and pdl_on:
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a0.record(stream)
            for i in range(K):
                step(i, 0)
            a1.record(stream)
        stream.synchronize()
        no_pdl_ms = a0.elapsed_time(a1) / K
    if world > 1:
        t = torch.tensor([total_ms], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    clocks = None
    if sampler and args.clock_seconds <= 0:
        clocks = sampler.summary(wall0, wall1)
        sampler.stop()
    elif sampler:
        # The timed region of a short run lasts a millisecond or so, shorter
        # than the sampling period; the clock record comes from a sustained
        # loop of the same calls right after it (outside the timed region).
        region = sampler.summary(wall0, wall1)
        per_call_s = total_ms * 1e-3 / K * (1 if graph is None else 2 * rot)
        n_loop = max(1, int(args.clock_seconds / max(per_call_s, 1e-6)))
        torch.cuda.synchronize(dev)
        c0 = time.time()
        with torch.cuda.stream(stream):
            for i in range(n_loop):
                if graph is None:
                    step(i)
                else:
                    graph.replay()
        stream.synchronize()
        c1 = time.time()
        clocks = sampler.summary(c0, c1)
        clocks["source"] = (f"sustained loop of {n_loop * (1 if graph is None else 2 * rot)} "
                            f"calls ({c1 - c0:.2f} s) right after the timed region, "
                            "nvidia-smi every 100 ms")
        clocks["timed_region"] = region
        sampler.stop()

    alg = wl.algorithmic_bytes(args.op) + (2 * M * H if args.y_out and args.op == "fused" else 0)
    ms_step = total_ms / K
    value = world * alg * K / (total_ms * 1e-3) / 1e9
    kern_mean = ms_step                       # one launch per step
    achieved = alg / (kern_mean * 1e-3) / 1e9
    peak, peak_src = measured_hbm_peak()
    if args.op == "quantize":
        shape = {"kernel": "quantize_kernel"}
    else:
        shape = fq.fp4_launch_shape(M, H, dt, fmt, lay)
    kernel_name = shape["kernel"]
    traffic, traffic_src = recorded_traffic(wl.name, args.op)

    # ---- end-to-end through the C ABI with host buffers --------------------
    # Every step copies its inputs from pinned host memory, calls the library
    # and copies all of its outputs back.  Steps are pipelined the way a
    # serving loop would run them: two device buffer sets, host-to-device
    # copies on one stream, the call on another, device-to-host copies on a
    # third, so step i+1's upload and step i-1's download overlap step i.
    e2e = None
    if rank == 0 and args.e2e_steps > 0:
        fused = args.op == "fused"
        hx = x.cpu().pin_memory()
        hr = r.cpu().pin_memory()
        hw = w.cpu().pin_memory()
        ho_r = torch.empty_like(hr).pin_memory()
        ho_p = torch.empty(packed.shape, dtype=torch.uint8).pin_memory()
        ho_s = torch.empty(sf.shape, dtype=torch.uint8).pin_memory()
        ho_s2 = torch.empty(sf_rm.shape, dtype=torch.uint8).pin_memory() if sf_rm is not None else None
        ho_y = torch.empty(M, H, dtype=x.dtype).pin_memory() if fused and args.y_out else None
        sets = []
        for _ in range(2):
            sets.append({
                "x": torch.empty_like(x), "r": torch.empty_like(r), "w": torch.empty_like(w),
                "p": torch.empty_like(packed), "s": torch.empty_like(sf),
                "s2": torch.empty_like(sf_rm) if sf_rm is not None else None,
                "y": torch.empty_like(y_t) if y_t is not None else None,
                "up": torch.cuda.Event(), "done": torch.cuda.Event(), "down": torch.cuda.Event()})
        h2d = hx.numel() * 2 + (hr.numel() * 2 + hw.numel() * 2 if fused else 0)
        d2h = (ho_r.numel() * 2 if fused else 0) + ho_p.numel() + ho_s.numel() + \
            (ho_s2.numel() if ho_s2 is not None else 0) + (ho_y.numel() * 2 if ho_y is not None else 0)
        s_up = torch.cuda.Stream(device=dev)
        s_down = torch.cuda.Stream(device=dev)

        def e2e_step(i):
            b = sets[i & 1]
            with torch.cuda.stream(s_up):
                if i >= 2:
                    s_up.wait_event(b["down"])        # step i-2 has read this set out
                b["x"].copy_(hx, non_blocking=True)
                if fused:
                    b["r"].copy_(hr, non_blocking=True)
                    b["w"].copy_(hw, non_blocking=True)
                b["up"].record(s_up)
            stream.wait_event(b["up"])
            s2p = b["s2"].data_ptr() if b["s2"] is not None else None
            if args.op == "quantize":
                st = L.fp4_quantize(b["x"].data_ptr(), gp, M, H, dt, fmt, lay, b["p"].data_ptr(),
                                    b["s"].data_ptr(), s2p, pdl_on, sh)
            else:
                st = L.fp4_add_rmsnorm_quant_ex(
                    b["x"].data_ptr(), H, b["r"].data_ptr(), H, b["w"].data_ptr(), gp, eps, M, H,
                    dt, fmt, lay, b["p"].data_ptr(), b["s"].data_ptr(), s2p,
                    b["y"].data_ptr() if b["y"] is not None else None, None, pdl_on, sh)
            if st != 0:
                raise fq.Fp4Error(st, "e2e step")
            b["done"].record(stream)
            with torch.cuda.stream(s_down):
                s_down.wait_event(b["done"])
                if fused:
                    ho_r.copy_(b["r"], non_blocking=True)
                ho_p.copy_(b["p"], non_blocking=True)
                ho_s.copy_(b["s"], non_blocking=True)
                if ho_s2 is not None:
                    ho_s2.copy_(b["s2"], non_blocking=True)
                if ho_y is not None:
                    ho_y.copy_(b["y"], non_blocking=True)
                b["down"].record(s_down)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        a.record(s_up)
        stream.wait_event(a)
        s_down.wait_event(a)
        for i in range(args.e2e_steps):
            e2e_step(i)
        e.record(s_down)                                # after the last download
        torch.cuda.synchronize(dev)
        e2e_ms = a.elapsed_time(e) / args.e2e_steps
        e2e = {"value": round(alg / (e2e_ms * 1e-3) / 1e9, 3), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(e2e_ms, 4), "steps": args.e2e_steps,
               "pipeline": "2 buffer sets; upload, call and download on 3 streams, "
                           "overlapped across steps"}

    # ---- the other large workloads, each timed the same way ----------------
    configs = None
    if rank == 0 and world == 1 and args.op == "fused" and not args.no_configs and \
            args.global_scale is None and not args.y_out:
        peak_gbs, _ = measured_hbm_peak()
        configs = []
        for other in large_workloads():
            if other.name == wl.name:
                continue
            configs.append(time_config(L, fq, other, dev, stream, args.config_steps, peak_gbs,
                                       pdl_on))

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.op == "fused":
        cpu = cpu_baseline(wl, args.cpu_seconds, args.cpu_cores)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": wl.name, "op": args.op, "global_scale": args.global_scale,
                       "y_out": bool(args.y_out), "pdl": bool(pdl_on),
                       "M": M, "H": H, "format": wl.fmt,
                       "sf_layout": wl.sf_layout, "io_dtype": wl.dtype, "eps": wl.eps,
                       "algorithmic_bytes_per_step": alg,
                       "l2": ("inputs larger than L2 (%.0f MB per step vs 129 MB), no flush"
                              % (alg / 1e6)) if rot == 1 else
                             ("%d input/output copies rotated (%.0f MB per pass vs 129 MB L2%s), "
                              "one pass of %d calls captured as a CUDA graph and replayed"
                              % (rot, 2 * rot * alg / 1e6,
                                 "" if 2 * rot * alg >= 2 * L2_BYTES else
                                 "; fewer bytes than L2: the number is L2-assisted",
                                 2 * rot)),
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "rows_per_s": round(world * M * K / (total_ms * 1e-3), 1),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                         if peak_src == "measured" else "fallback 6.8 TB/s",
                         "traffic": traffic, "traffic_source": traffic_src,
                         "kernel": kernel_name, "launch": shape,
                         "kernel_ms_mean": round(kern_mean, 5),
                         "kernel_ms_event_pairs_median": round(statistics.median(kern_ms), 5),
                         "no_pdl": None if no_pdl_ms is None else {
                             "kernel_ms_mean": round(no_pdl_ms, 5),
                             "achieved": round(alg / (no_pdl_ms * 1e-3) / 1e9, 1),
                             "frac": round(alg / (no_pdl_ms * 1e-3) / 1e9 / peak, 4)}},
            "clocks": clocks, "e2e": e2e, "gpu_launches": K, "cpu_baseline": cpu,
            "configs": configs,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def large_workloads():
    """The workloads graded against the HBM roofline: C3, C4 and every
    M = 32768 cell of the sweep (both formats, four widths)."""
    return [workloads.C3, workloads.C4] + [w for w in workloads.sweep() if w.M == 32768]


def time_config(L, fq, wl, dev, stream, steps: int, peak: float, pdl: int = 1):
    """One large workload: inputs drawn on the device, `steps` calls timed
    back to back between two events on `stream` after 5 warm-up calls
    (consecutive calls alternate x and -x, each a programmatic dependent of
    the one before when `pdl`), each call one launch; then the same without
    programmatic dependent launch.  Every one of these moves more than twice
    the L2 per call, so no flush is needed."""
    import torch
    M, H = wl.M, wl.H
    fmt = {"nvfp4": fq.FP4_NVFP4, "mxfp4": fq.FP4_MXFP4, "e4m3b32": fq.FP4_E4M3_B32}[wl.fmt]
    lay = {"rowmajor": fq.FP4_SF_ROWMAJOR, "swizzled": fq.FP4_SF_SWIZZLED,
           "both": fq.FP4_SF_BOTH}[wl.sf_layout]
    dt = fq.FP4_DT_BF16 if wl.dtype == "bf16" else fq.FP4_DT_FP16
    x, r, w = workloads.make_inputs(wl, dev)
    xs = (x, -x)
    nb = H // wl.block
    packed = torch.empty(M, H // 2, dtype=torch.uint8, device=dev)
    sf = torch.empty(max(1, fq.fp4_sf_size_bytes(M, H, fmt, lay)), dtype=torch.uint8, device=dev)
    sf_rm = torch.empty(M * nb, dtype=torch.uint8, device=dev) if lay == fq.FP4_SF_BOTH else None
    sh = stream.cuda_stream
    s2 = sf_rm.data_ptr() if sf_rm is not None else None

    def step(i, pdl_i):
        st = L.fp4_add_rmsnorm_quant_ex(xs[i & 1].data_ptr(), H, r.data_ptr(), H, w.data_ptr(),
                                        None, float(wl.eps), M, H, dt, fmt, lay,
                                        packed.data_ptr(), sf.data_ptr(), s2, None, None, pdl_i,
                                        sh)
        if st != 0:
            raise fq.Fp4Error(st, wl.name)

    def timed(pdl_i):
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for i in range(5):
                step(i, pdl_i)
            a.record(stream)
            for i in range(steps):
                step(i, pdl_i)
            b.record(stream)
        stream.synchronize()
        return a.elapsed_time(b) / steps

    ms = timed(pdl)
    ms_no_pdl = timed(0) if pdl else ms
    alg = wl.algorithmic_bytes()
    shape = fq.fp4_launch_shape(M, H, dt, fmt, lay)
    del x, r, w, xs, packed, sf, sf_rm
    torch.cuda.empty_cache()
    return {"workload": wl.name, "ms_per_step": round(ms, 5), "steps": steps, "pdl": bool(pdl),
            "algorithmic_bytes": alg, "gbs": round(alg / (ms * 1e-3) / 1e9, 1),
            "frac": round(alg / (ms * 1e-3) / 1e9 / peak, 4), "kernel": shape["kernel"],
            "launch": shape, "no_pdl": {"ms_per_step": round(ms_no_pdl, 5),
                                        "frac": round(alg / (ms_no_pdl * 1e-3) / 1e9 / peak, 4)}}


# ---------------------------------------------------------------------------
# the consumer GEMM
# ---------------------------------------------------------------------------
GEMM_METRIC = "NVFP4 GEMM TFLOP/s (bf16 out) and % of the GB300 FP4 tensor roofline"
FP4_PER_BF16 = 13.5 / 2.25     # nominal dense FP4 / bf16 tensor rates


def measured_fp4_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]) * FP4_PER_BF16, \
            "measured bf16 burst (MEASURED_PEAKS.json bf16_tflops) x 6, the nominal FP4/bf16 ratio"
    except Exception:
        return 1900.0 * FP4_PER_BF16, "fallback 1.9 PFLOP/s bf16 x 6"


def gemm_operands(gw, device, fmt="nvfp4"):
    K = gw.K
    a = workloads.random_bytes(gw.M * K // 2, gw.seed, 0, device=device).reshape(gw.M, K // 2)
    b = workloads.random_bytes(gw.N * K // 2, gw.seed, 1, device=device).reshape(gw.N, K // 2)
    # scale bytes: E4M3 2^-3..9 or UE8M0 2^-5..2^5; tiled buffers of 4-scale groups
    scales = list(range(0x20, 0x51)) if fmt == "nvfp4" else list(range(122, 133))
    group = 64 if fmt == "nvfp4" else 128
    nsa = ((gw.M + 127) // 128) * (K // group) * 512
    nsb = ((gw.N + 127) // 128) * (K // group) * 512
    sfa = workloads.random_bytes(nsa, gw.seed, 2, scales, device=device)
    sfb = workloads.random_bytes(nsb, gw.seed, 3, scales, device=device)
    return a, b, sfa, sfb


def gemm_cpu_baseline(gw, seconds: float):
    """The GEMM oracle on the first rows of the workload (the whole B operand
    is dequantised each time, as the oracle stands)."""
    import oracle
    a, b, sfa, sfb = gemm_operands(gw, "cpu")
    an, bn, san, sbn = a.numpy(), b.numpy(), sfa.numpy(), sfb.numpy()
    rows = 1
    while True:
        t = time.perf_counter()
        oracle.gemm_bf16(an, bn, san, sbn, gw.M, gw.N, gw.K, rows=np.arange(rows))
        dt = time.perf_counter() - t
        if dt > seconds / 4 or rows >= gw.M:
            break
        rows = min(gw.M, rows * 4)
    flops = 2 * rows * gw.N * gw.K
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": 1,
            "kind": "oracle",
            "sample": f"{rows} of {gw.M} rows of {gw.name} (B dequantised in full), numpy "
                      f"oracle, {dt:.1f} s"}


def run_gemm_reference(args):
    """The GEMM oracle as the reference arm: each step a bounded row sample."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    gw = workloads.GEMM_CONFIGS[args.gemm]
    steps = [gemm_cpu_baseline(gw, 2.0) for _ in range(max(1, args.steps))]
    val = statistics.median(s["value"] for s in steps)
    line = {"impl": "reference", "metric": GEMM_METRIC, "value": val, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": len(steps), "warmup": 0, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": gw.name, "op": "gemm", "M": gw.M, "N": gw.N, "K": gw.K},
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                             "sample": steps[0]["sample"]},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_gemm(args):
    import torch

    import rmsnorm_fp4_quant_gb300 as fq

    world, rank, local = dist_env()
    gw = workloads.GEMM_CONFIGS[args.gemm]
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    L = fq.lib()
    a, b, sfa, sfb = gemm_operands(gw, dev, args.gemm_format)
    gemm_call = L.fp4_gemm_nvfp4_bf16 if args.gemm_format == "nvfp4" else L.fp4_gemm_mxfp4_bf16
    out = torch.empty(gw.M, gw.N, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream
    op_ = out.data_ptr()

    alg = gw.algorithmic_bytes()
    # Operands smaller than L2: rotate through enough copies that one pass
    # touches more than twice the L2, and replay the pass as a CUDA graph (no
    # host launch cost: a decode step would be captured the same way).
    rot = 1 if alg >= 2 * L2_BYTES else -(-2 * L2_BYTES // alg)
    sets = [(a, b, sfa, sfb, out)]
    for j in range(1, rot):
        sets.append(tuple(t.clone() for t in (a, b, sfa, sfb)) + (torch.empty_like(out),))

    def launch(k):
        s_ = sets[k % rot]
        st = gemm_call(s_[0].data_ptr(), s_[1].data_ptr(), s_[2].data_ptr(), s_[3].data_ptr(),
                       1.0, None, None, gw.M, gw.N, gw.K, s_[4].data_ptr(), args.gemm_variant,
                       0, sh)
        if st != 0:
            raise fq.Fp4Error(st, "fp4_gemm_nvfp4_bf16")

    torch.cuda.synchronize(dev)           # operands and copies were made on the default stream
    sampler = ClockSampler(gpu_smi_id(torch, dev)) if rank == 0 else None
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, rot)):
            launch(i)
    stream.synchronize()
    graph = None
    if rot > 1:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                for i in range(rot):
                    launch(i)
            for _ in range(3):
                graph.replay()
        stream.synchronize()
    K = args.steps if rot == 1 else -(-args.steps // rot) * rot
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        if graph is None:
            for i in range(K):
                launch(i)
        else:
            for _ in range(K // rot):
                graph.replay()
        t1.record(stream)
    stream.synchronize()
    total_ms = t0.elapsed_time(t1)
    wall1 = time.time()
    clocks = sampler.summary(wall0, wall1) if sampler else None
    if sampler:
        sampler.stop()
    ms = total_ms / K
    tflops = gw.flops() / (ms * 1e-3) / 1e12
    gbs = alg / (ms * 1e-3) / 1e9
    fp4_peak, fp4_src = measured_fp4_peak()
    hbm_peak, hbm_src = measured_hbm_peak()
    tensor_bound = gw.flops() / alg > fp4_peak * 1e12 / (hbm_peak * 1e9)
    roof = ({"bound": "tensor", "achieved": round(tflops, 1), "peak": round(fp4_peak, 1),
             "unit": "TFLOP/s", "frac": round(tflops / fp4_peak, 4), "peak_source": fp4_src}
            if tensor_bound else
            {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak, "unit": "GB/s",
             "frac": round(gbs / hbm_peak, 4), "peak_source": f"{hbm_src} hbm_gbs"})
    sched = fq.fp4_gemm_variant(gw.M, gw.N, gw.K, 0 if args.gemm_format == "nvfp4" else 1,
                                False, args.gemm_variant)
    # a GEMM capture is keyed by shape, operand format, kernel and tile width
    traffic, traffic_src = recorded_traffic(gemm_profile_key(gw.name, args.gemm_format,
                                                             sched["kernel"], sched["tile_n"]),
                                            "gemm")
    roof.update({"traffic": traffic, "traffic_source": traffic_src,
                 "kernel": sched["kernel"], "schedule": sched, "kernel_ms_mean": round(ms, 5),
                 "algorithmic_bytes": alg, "flops": gw.flops()})

    e2e = None
    if rank == 0 and args.e2e_steps > 0:
        hs = [t.cpu().pin_memory() for t in (a, b, sfa, sfb)]
        ds = [torch.empty_like(t) for t in (a, b, sfa, sfb)]
        ho = torch.empty(out.shape, dtype=out.dtype).pin_memory()

        def e2e_step():
            for d, h in zip(ds, hs):
                d.copy_(h, non_blocking=True)
            st = gemm_call(ds[0].data_ptr(), ds[1].data_ptr(), ds[2].data_ptr(),
                           ds[3].data_ptr(), 1.0, None, None, gw.M, gw.N, gw.K, op_,
                           args.gemm_variant, 0, sh)
            if st != 0:
                raise fq.Fp4Error(st, "e2e gemm")
            ho.copy_(out, non_blocking=True)

        with torch.cuda.stream(stream):
            e2e_step()
            stream.synchronize()
            x0 = torch.cuda.Event(enable_timing=True)
            x1 = torch.cuda.Event(enable_timing=True)
            x0.record(stream)
            for _ in range(args.e2e_steps):
                e2e_step()
            x1.record(stream)
        stream.synchronize()
        e2e_ms = x0.elapsed_time(x1) / args.e2e_steps
        e2e = {"value": round(gw.flops() / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
               "h2d_bytes_per_step": sum(h.numel() for h in hs),
               "d2h_bytes_per_step": ho.numel() * 2, "ms_per_step": round(e2e_ms, 4),
               "steps": args.e2e_steps}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = gemm_cpu_baseline(gw, args.cpu_seconds)
    if rank == 0:
        line = {
            "metric": GEMM_METRIC.replace("NVFP4", args.gemm_format.upper()),
            "value": round(world * tflops, 2), "unit": "TFLOP/s",
            "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e2m1 x e2m1 -> f32 accumulate, bf16 out", "data": "synthetic",
            "config": {"workload": gw.name, "op": "gemm", "M": gw.M, "N": gw.N, "K": gw.K,
                       "variant": args.gemm_variant, "format": args.gemm_format,
                       "operands": "uniform random E2M1 bytes, scale bytes 2^-3..9 (E4M3) or "
                                   "2^-5..2^5 (UE8M0)",
                       "l2": ("%d operand copies rotated (%.0f MB per pass vs 129 MB L2), "
                              "one pass captured as a CUDA graph and replayed" % (rot, rot * alg / 1e6))
                             if rot > 1 else
                             "operands + output %.0f MB per launch vs 129 MB L2, no flush"
                             % (alg / 1e6),
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "roofline": roof, "clocks": clocks, "e2e": e2e, "gpu_launches": K,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# a decode step's chain: add + RMSNorm + NVFP4 quantization of M rows, then the
# projection that consumes the codes and tiled scales
# ---------------------------------------------------------------------------
CHAIN_METRIC = "fused add+RMSNorm+NVFP4 quant -> NVFP4 GEMM chain, us per step"


def run_chain(args):
    """One step = fp4_add_rmsnorm_quant_ex on M x K rows (bf16, NVFP4, tiled
    scales) followed by fp4_gemm_nvfp4_bf16 of its codes against an N x K
    NVFP4 weight, launched without programmatic dependent launch, with it
    (pdl = 1), and with it and the weights declared static (the GEMM's pdl =
    2: its B copies start before the dependency wait); enough copies of the inputs, weights and outputs rotate that one
    pass moves more than twice the L2, and a pass of steps is replayed as a
    CUDA graph (as a decode loop would run it)."""
    import torch

    import rmsnorm_fp4_quant_gb300 as fq

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    L = fq.lib()
    gw = workloads.GEMM_CONFIGS[args.gemm]
    M, N, K = gw.M, gw.N, gw.K
    wl = workloads.Workload("chain", M, K, "bf16", "nvfp4", "swizzled", 1e-6, seed=gw.seed)
    x, r, w = workloads.make_inputs(wl, dev)
    _, b, _, sfb = gemm_operands(gw, dev)
    sf_bytes = fq.fp4_sf_size_bytes(M, K, fq.FP4_NVFP4, fq.FP4_SF_SWIZZLED)
    per_step = wl.algorithmic_bytes() + gw.algorithmic_bytes()
    rot = max(1, -(-2 * L2_BYTES // per_step))
    sets = []
    for _ in range(rot):
        sets.append({"x": x.clone(), "xn": -x, "r": r.clone(), "b": b.clone(), "sfb": sfb.clone(),
                     "p": torch.empty(M, K // 2, dtype=torch.uint8, device=dev),
                     "s": torch.empty(sf_bytes, dtype=torch.uint8, device=dev),
                     "o": torch.empty(M, N, dtype=torch.bfloat16, device=dev)})
    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream
    torch.cuda.synchronize(dev)           # inputs and copies were made on the default stream

    def step(c, xs, mode):
        pdl = 1 if mode else 0          # the fused call: PDL on or off
        gemm_pdl = mode                 # the GEMM: 0, 1, or 2 (static weights)
        st = L.fp4_add_rmsnorm_quant_ex(xs.data_ptr(), K, c["r"].data_ptr(), K, w.data_ptr(),
                                        None, 1e-6, M, K, fq.FP4_DT_BF16, fq.FP4_NVFP4,
                                        fq.FP4_SF_SWIZZLED, c["p"].data_ptr(), c["s"].data_ptr(),
                                        None, None, None, pdl, sh)
        if st != 0:
            raise fq.Fp4Error(st, "chain: fused")
        st = L.fp4_gemm_nvfp4_bf16(c["p"].data_ptr(), c["b"].data_ptr(), c["s"].data_ptr(),
                                   c["sfb"].data_ptr(), 1.0, None, None, M, N, K,
                                   c["o"].data_ptr(), -1, gemm_pdl, sh)
        if st != 0:
            raise fq.Fp4Error(st, "chain: gemm")

    results = {}
    for mode in (0, 1, 2):
        def one_pass():
            for c in sets:
                step(c, c["x"], mode)
            for c in sets:
                step(c, c["xn"], mode)
        with torch.cuda.stream(stream):
            one_pass()
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                one_pass()
            for _ in range(max(3, args.warmup)):
                graph.replay()
        stream.synchronize()
        reps = max(1, -(-args.steps // (2 * rot)))
        a = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            for _ in range(reps):
                graph.replay()
            e.record(stream)
        stream.synchronize()
        results[mode] = a.elapsed_time(e) * 1e3 / (reps * 2 * rot)
    line = {"metric": CHAIN_METRIC, "value": round(results[2], 3), "unit": "us",
            "n_gpus": 1, "steps": reps * 2 * rot, "warmup": args.warmup,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16 in, e2m1 x e2m1 -> f32, bf16 out", "data": "synthetic",
            "config": {"workload": f"chain_{gw.name}", "M": M, "N": N, "K": K,
                       "l2": "%d copies of inputs, weights and outputs rotated (%.0f MB per "
                             "pass vs 129 MB L2), one pass captured as a CUDA graph"
                             % (rot, 2 * rot * per_step / 1e6),
                       "fused_kernel": fq.fp4_launch_shape(M, K, 0, 0, 1)["kernel"],
                       "gemm": fq.fp4_gemm_variant(M, N, K)},
            "us_per_step_without_pdl": round(results[0], 3),
            "us_per_step_with_pdl": round(results[1], 3),
            "us_per_step_with_pdl_static_weights": round(results[2], 3),
            "gpu_launches": 2 * reps * 2 * rot}
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.op == "chain":
        run_chain(args)
        return
    if args.op == "gemm":
        if args.impl == "reference":
            run_gemm_reference(args)
            return
        run_gemm(args)
        return
    wl = workloads.CONFIGS[args.workload]
    if args.rows is not None:
        wl = wl.with_shape(args.rows)
    if args.format is not None:
        import dataclasses
        wl = dataclasses.replace(wl, fmt=args.format)
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
