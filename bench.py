#!/usr/bin/env python3
"""Benchmark of the chunked AllGather x MatMul hot path on GB300.

A step is one fused AllGather-MatMul call (tgc_ag_matmul_ex, mode FUSED) on
the largest workload: 4 virtual ranks, a_shard bf16 (8192, 8192) each
(M = 32768), B bf16 (8192, 8192), comm_block_rows = 512, blocks released in a
seeded permutation with injected delays.  Inputs are resident in HBM when the
timed region starts; they are larger than L2, so L2 is not flushed.

The same JSON line also reports, each timed the same way:
  unfused   the library's TGATHER kernel then its GEMM kernel
  mm_only   the GEMM kernel alone on the gathered buffer (ceiling)
  no_delay  the fused path with the injected delays set to 0
  tgather   TGATHER GB/s on 8 x fp16 (2,1,1,1024,1024) and on the ragged
            int32 (1,1,1,1000,777) workload, rotating buffers (> 2 x L2)
  e2e       the fused call with its inputs copied from pinned host memory and
            C copied back inside the timed region
  cpu_baseline  the CPU oracle on a bounded row sample, host cores (also the
                TGATHER oracle and the whole square workload's oracle)

``--impl reference`` times the CPU oracle instead (rank 0 only).
Multi-GPU: the path does not shard; --gpus N runs N independent replicas
(weak scaling), with a barrier and max-over-ranks timing only.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused AG-MatMul TFLOP/s (% BF16 peak); TGATHER GB/s (% HBM peak)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = ["tile_gather_comm_gb300/csrc/gemm.cu", "tile_gather_comm_gb300/csrc/prims.cuh",
                  "tile_gather_comm_gb300/csrc/schedule.h", "tile_gather_comm_gb300/csrc/internal.h"]
TGATHER_SOURCES = ["tile_gather_comm_gb300/csrc/tgather.cu", "tile_gather_comm_gb300/csrc/prims.cuh",
                   "tile_gather_comm_gb300/csrc/internal.h"]


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="large_skewed", choices=["large_skewed", "mlp_up", "square", "tiny"])
    p.add_argument("--quick", action="store_true", help="main line only: skip extras, e2e and cpu baseline")
    p.add_argument("--only", choices=["all", "tgather", "gemm_vs_cublas"], default="all",
                   help="tgather: time only the TGATHER workloads (small footprint, for profiling); "
                        "gemm_vs_cublas: the plain GEMM and torch.matmul on the workload's gathered A, "
                        "two warm-up calls each then one call each (for an ncu capture of both)")
    p.add_argument("--clock-ms", type=int, default=20, help="nvidia-smi sampling period")
    p.add_argument("--pivot", default="auto", choices=["auto", "page", "shard", "none", "ready_queue"],
                   help="tile order of the headline call (auto: the library's choice, as tgc_ag_matmul)")
    p.add_argument("--tile-n", type=int, default=0, choices=[0, 256, 512],
                   help="GEMM tile width for the timed calls; 0 = the library's rule")
    p.add_argument("--band-n", type=int, default=0,
                   help="tile raster of the headline call: 0 = the library's choice, > 0 = bands of that many "
                        "tile columns, < 0 = the group raster")
    return p.parse_args(argv)


# ----------------------------------------------------------------------------- distributed plumbing


class Dist:
    """Rank bookkeeping: barrier and max-over-ranks reductions only (no data-path collective)."""

    def __init__(self, init: bool = True):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1 and init:
            import torch.distributed as dist
            backend = os.environ.get("TGC_BENCH_BACKEND", "gloo")
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if self.pg is None:
            return x
        import torch
        t = torch.tensor([float(x)], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def aggregate(per_rank_ms: float, units_per_rank: float, dist: Dist, scale: float = 1e-12):
    """Whole-job throughput: units processed by all ranks / max-over-ranks time (weak scaling)."""
    ms = dist.max(per_rank_ms)
    total_units = units_per_rank * dist.world
    return total_units / (ms * 1e-3) * scale, ms


# ----------------------------------------------------------------------------- measurement helpers


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def strip_comments(src: str) -> str:
    """C/C++/CUDA source without comments and blank lines, each line stripped: what the
    compiler sees of it (string and character literals are kept as written)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = (ln.strip() for ln in "".join(out).splitlines())
    return "\n".join(ln for ln in lines if ln)


def sources_sha(paths) -> str:
    """Hash of the kernel sources as compiled: comment and whitespace edits keep it."""
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), encoding="utf-8") as f:
            h.update(strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def profiled_traffic(key: str, sources):
    """DRAM bytes (read + write) per launch of one kernel on one workload, as an ncu capture
    recorded them in profiles/traffic.json, if the capture was taken on the current kernel
    sources (same comment-stripped hash); otherwise None."""
    try:
        with open(TRAFFIC_FILE, encoding="utf-8") as f:
            entry = json.load(f).get(key)
    except (OSError, ValueError):
        return None
    if not entry or entry.get("source_sha256_16") != sources_sha(sources):
        return None
    return float(entry["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed regions run."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="tgc_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 f"-lms={self.period}"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self, window: tuple | None = None):
        """Summary of the samples.  `window` = (t0, t1) in time.time() seconds: the
        region whose clocks `sm_mhz` reports (all samples under load if none fell in it).
        The raw lines stay in `self.lines` for summaries of other windows."""
        self.lines = []
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        with open(self.path) as f:
            self.lines = f.readlines()
        os.unlink(self.path)
        return clock_summary(self.lines, window)


def clock_summary(lines, window: tuple | None = None):
    """Summary of nvidia-smi CSV lines in ClockSampler.QUERY order: the median SM clock of
    the samples inside `window` (host time.time() seconds), else of the samples under load
    (power draw at least half the largest seen); the largest clocks and power; and every
    throttle reason seen active in those samples."""
    rows = []
    for line in lines:
        parts = [x.strip() for x in line.split(",")]
        if len(parts) < 10:
            continue
        try:
            ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            rows.append((float(parts[2]), float(parts[3]), float(parts[4]), parts[5], parts[6:10], ts))
        except ValueError:
            continue
    if not rows:
        return None
    pmax = max(r[2] for r in rows)
    loaded = [r for r in rows if r[2] >= 0.5 * pmax] or rows  # power draw marks the samples under load
    inside = [r for r in rows if window is not None and window[0] <= r[5] <= window[1]]
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = sorted({names[i] for r in loaded + inside for i, v in enumerate(r[4]) if v.lower() == "active"})
    return {"sm_mhz": statistics.median(r[0] for r in (inside or loaded)), "sm_max_mhz": max(r[1] for r in rows),
            "power_w_max": max(r[2] for r in rows), "samples": len(rows), "samples_under_load": len(loaded),
            "samples_in_value_region": len(inside),
            "sm_mhz_under_load_all_regions": statistics.median(r[0] for r in loaded),
            "reasons": reasons}


def check_device_status(ws, where: str):
    """The workspace's device status word after a timed region: a bounded wait that expired
    stops the kernels early, and the times of such calls are not measurements of the work."""
    import torch

    import tile_gather_comm_gb300 as tgc
    if ws.is_cuda:
        torch.cuda.synchronize()
    st = int(ws[:4].view(torch.int32)[0].item())
    if st != 0:
        raise RuntimeError(f"device status {st} ({tgc.tgc_status_string(st)}) after {where}; "
                           "the timings of that region are void")


def time_interleaved(variants: dict, steps: int, dist: Dist, stream, rounds: int = 6):
    """Median ms per call of each variant, timed in alternating rounds of ~steps/rounds calls."""
    import torch
    per = max(2, steps // rounds)
    names = list(variants)
    for n in names:
        for _ in range(2):
            variants[n]()
    torch.cuda.synchronize()
    times = {n: [] for n in names}
    for r in range(rounds):
        for n in (names if r % 2 == 0 else names[::-1]):
            dist.barrier()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(per):
                variants[n]()
            e1.record(stream)
            torch.cuda.synchronize()
            times[n].append(e0.elapsed_time(e1) / per)
    return {n: statistics.median(v) for n, v in times.items()}


def time_device(fn, steps: int, warmup: int, dist: Dist, stream, per_step: list | None = None,
                wall: list | None = None):
    """Barrier + sync, then CUDA events on `stream` around exactly `steps` calls.
    If `per_step` is a list, an event is also recorded after every call and the
    per-call times (ms) are appended to it.  If `wall` is a list, its two entries
    become the host times (time.time()) just before the first call and after the
    closing synchronize."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1 if per_step is not None else 2)]
    if wall is not None:
        wall[0] = time.time()
    ev[0].record(stream)
    for i in range(steps):
        fn()
        if per_step is not None:
            ev[i + 1].record(stream)
    ev[-1].record(stream)
    torch.cuda.synchronize()
    if wall is not None:
        wall[1] = time.time()
    dist.barrier()
    if per_step is not None:
        per_step.extend(ev[i].elapsed_time(ev[i + 1]) for i in range(steps))
    return ev[0].elapsed_time(ev[-1]) / steps


def percentiles(xs: list, qs=(10, 50, 90)) -> dict:
    """Nearest-rank percentiles of a list of numbers."""
    v = sorted(xs)
    if not v:
        return {}
    return {f"p{q}": round(v[min(len(v) - 1, max(0, -(-q * len(v) // 100) - 1))], 4) for q in qs}


# ----------------------------------------------------------------------------- our arm


def run_ours(args, dist: Dist):
    import numpy as np
    import torch

    import tile_gather_comm_gb300 as tgc
    from tile_gather_comm_gb300 import _build
    from tile_gather_comm_gb300.workloads import (AG_CONFIGS, TG_CONFIGS, make_ag_inputs,
                                                  make_release_schedule, make_tg_inputs)

    _build.build()
    tgc.lib()
    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    peaks, peaks_kind = load_peaks()
    if args.only == "gemm_vs_cublas":
        return gemm_vs_cublas(AG_CONFIGS[args.workload], dev, args)
    if args.only == "tgather":
        res = {"metric": METRIC, "unit": "GB/s", "n_gpus": dist.world, "steps": args.steps,
               "warmup": args.warmup, "note": "TGATHER only (profiling run)"}
        res["tgather"] = bench_tgather(TG_CONFIGS["bw_f16"], dev, stream, dist, peaks, peaks_kind, args)
        res["value"] = res["tgather"]["value"]
        res["tgather_ragged_i32"] = bench_tgather(TG_CONFIGS["ragged_i32"], dev, stream, dist, peaks,
                                                  peaks_kind, args)
        res["tgather_release"] = bench_tgather_release(TG_CONFIGS["bw_f16"], dev, dist, peaks, peaks_kind)
        res["tgather_strided"] = bench_tgather_strided(TG_CONFIGS["bw_f16"], dev, dist, peaks, peaks_kind)
        res["tgather_context_long"] = bench_tgather_context_long(dev, stream, dist, peaks, peaks_kind, args)
        return res
    cfg = AG_CONFIGS[args.workload]
    flops = float(cfg.flops)

    shards_h, B_h = make_ag_inputs(cfg, seed=0)
    shards = [s.to(dev) for s in shards_h]
    B = B_h.to(dev)
    C = torch.empty(cfg.M, cfg.N, dtype=torch.bfloat16, device=dev)
    a = torch.empty(cfg.M, cfg.K, dtype=torch.bfloat16, device=dev)
    progress = torch.zeros(cfg.nblocks, dtype=torch.int32, device=dev)
    ws = torch.zeros(tgc.tgc_ag_matmul_workspace_bytes(cfg.R, cfg.M, cfg.K, cfg.N, cfg.cb),
                     dtype=torch.uint8, device=dev)
    order = delay = None
    if cfg.skewed:
        o, d = make_release_schedule(cfg, rank=0, seed=0)
        order, delay = o.tolist(), d.tolist()
    epoch = [0]
    launches = [0]

    def call(mode="fused", delays=True, pivot=args.pivot, out=None, out_format="bf16", band_n=args.band_n,
             tile_n=args.tile_n):
        epoch[0] += 1
        tgc.tgc_ag_matmul_ex(shards, B, C if out is None else out, a, cfg.cb, mode=mode, progress=progress,
                             epoch=epoch[0], workspace=ws, order=order if mode == "fused" else None,
                             delay_ns=delay if (mode == "fused" and delays) else None, stream=stream,
                             pivot=pivot, out_format=out_format, band_n=band_n, tile_n=tile_n)
        launches[0] += 2 if mode == "unfused" else 1

    plan = tgc.tgc_ag_matmul_plan(shards, B, C, a, cfg.cb, progress=progress, workspace=ws, order=order,
                                  delay_ns=delay, pivot=args.pivot, band_n=args.band_n, tile_n=args.tile_n)

    sampler = ClockSampler(dist.local_rank, args.clock_ms)
    sampler.start()

    launches[0] = 0
    step_ms = []
    t_value = [0.0, 0.0]
    ms_fused = time_device(lambda: call("fused"), args.steps, args.warmup, dist, stream, per_step=step_ms,
                           wall=t_value)
    check_device_status(ws, "the value region")
    fused_launches_timed = args.steps  # one kernel per fused call
    value, ms_max = aggregate(ms_fused, flops, dist)
    kernel_tflops = flops / (ms_fused * 1e-3) * 1e-12
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {
            "workload": f"{cfg.name}: {cfg.R} virtual ranks x a_shard bf16 ({cfg.H},{cfg.K}) ~N(0,1), "
                        f"B bf16 ({cfg.N},{cfg.K}) ~N(0,{cfg.b_sigma}), comm_block_rows={cfg.cb}"
                        + (", seeded release permutation + delays U[0,20us]" if cfg.skewed else ""),
            "M": cfg.M, "N": cfg.N, "K": cfg.K, "R": cfg.R, "comm_block_rows": cfg.cb, "rank": 0,
            "pivot": args.pivot, "band_n": args.band_n,
            "plan": plan,
            "parallelism": f"replicas x{dist.world} (the path does not shard)",
            "l2": "inputs larger than L2 (shards 4x128 MiB + B 128 MiB); no flush",
            "timing": "CUDA events on the launching stream around exactly `steps` calls, max over ranks",
        },
        "gpu_launches": fused_launches_timed,
        "step_ms_percentiles": percentiles(step_ms),
    }
    prof = profiled_traffic(f"ag_gemm_fused/{cfg.name}", KERNEL_SOURCES)
    res["roofline"] = {"bound": "tensor", "achieved": round(kernel_tflops, 2), "peak": peaks["bf16_tflops"],
                       "unit": "TFLOP/s", "frac": round(kernel_tflops / peaks["bf16_tflops"], 4),
                       "traffic": prof, "peak_source": f"{peaks_kind} burst cuBLAS bf16",
                       "kernel": f"ag_gemm_kernel<fused, {plan['tile_n']}-column tiles>"}

    if not args.quick:
        # The comparison lines are timed interleaved (rounds of every variant, median per
        # variant), so that slow drifts of the power-capped clock do not bias their ratios.
        a_full = torch.cat(shards)

        def cublas():  # context only: the vendor library GEMM on the gathered A, same shapes
            torch.matmul(a_full, B.T, out=C)
        C8 = torch.empty(cfg.M, cfg.N, dtype=torch.uint8, device=dev)
        variants = {"fused": lambda: call("fused"), "unfused": lambda: call("unfused"),
                    "mm_only": lambda: call("mm_only"),
                    "ready_queue": lambda: call("fused", pivot="ready_queue"),
                    "page_group": lambda: call("fused", pivot="page", band_n=-1),
                    "fused_ce": lambda: call("fused_ce"),
                    "fused_fp8_out": lambda: call("fused", out=C8, out_format="f8e4m3"),
                    "cublas_gemm": cublas}
        if cfg.skewed:
            variants["no_delay"] = lambda: call("fused", delays=False)
        med = time_interleaved(variants, args.steps, dist, stream)
        check_device_status(ws, "the comparison lines")
        for k, v in med.items():
            res[k if k != "fused" else "fused_interleaved"] = {
                "value": round(aggregate(v, flops, dist)[0], 2), "unit": "TFLOP/s",
                "ms_per_step": round(dist.max(v), 4)}
        res["unfused"]["kernels_per_step"] = 2
        res["mm_only"]["frac_of_peak"] = round(flops / (med["mm_only"] * 1e-3) * 1e-12 / peaks["bf16_tflops"], 4)
        res["ready_queue"]["note"] = "same workload, READY_QUEUE tile order"
        res["page_group"]["note"] = "same workload, the page's rank pivot on the group raster (GROUP_SIZE_M swizzle)"
        res["cublas_gemm"]["note"] = ("context: torch.matmul (cuBLAS) on the already gathered A, "
                                      "same shapes; not part of this library")
        res["fused_ce"]["note"] = ("same workload, copy-engine producer: cudaMemcpyAsync per block on library "
                                   "side streams + a stream write of its flag; default release order, no delays")
        res["fused_fp8_out"]["note"] = "same workload and release schedule, C written as saturating float8 e4m3"
        del a_full, C8
        res["fused_over_unfused"] = round(med["unfused"] / med["fused"], 4)
        res["comparison_timing"] = "interleaved rounds (6), median per variant"
        res["tgather"] = bench_tgather(TG_CONFIGS["bw_f16"], dev, stream, dist, peaks, peaks_kind, args)
        res["tgather_ragged_i32"] = bench_tgather(TG_CONFIGS["ragged_i32"], dev, stream, dist, peaks,
                                                  peaks_kind, args)
        res["tgather_context_long"] = bench_tgather_context_long(dev, stream, dist, peaks, peaks_kind, args)
        res["tgather_strided"] = bench_tgather_strided(TG_CONFIGS["bw_f16"], dev, dist, peaks, peaks_kind)
        res["tgather_release"] = bench_tgather_release(TG_CONFIGS["bw_f16"], dev, dist, peaks, peaks_kind)
        # the same fused call over a region of at least a second: the GPU settles at its power
        # cap, so this is the figure to set against the sustained cuBLAS peak
        n_sus = max(args.steps, int(1.2e3 / max(ms_fused, 1e-3)) + 1)
        t_sus = [0.0, 0.0]
        ms_sus = time_device(lambda: call("fused"), n_sus, 3, dist, stream, wall=t_sus)
        check_device_status(ws, "the sustained region")
        v_sus, ms_sus_max = aggregate(ms_sus, flops, dist)
        k_sus = flops / (ms_sus * 1e-3) * 1e-12
        res["sustained"] = {
            "value": round(v_sus, 2), "unit": "TFLOP/s", "steps": n_sus, "ms_per_step": round(ms_sus_max, 4),
            "region_s": round(t_sus[1] - t_sus[0], 3),
            "frac_of_sustained_peak": round(k_sus / peaks["bf16_tflops_sustained"], 4),
            "frac_of_burst_peak": round(k_sus / peaks["bf16_tflops"], 4),
            "sustained_peak": peaks["bf16_tflops_sustained"],
            "peak_source": f"{peaks_kind} cuBLAS bf16 held for seconds under the power cap",
            "note": "the headline step (same call) timed over >= 1.2 s; `value` above is its first "
                    f"{args.steps} steps after {args.warmup} warm-up calls"}
        # context: cuBLAS's GEMM alone on the already gathered A, right after, over a region
        # as long, so that both figures are taken at the power cap
        a_full = torch.cat(shards)
        t_cb = [0.0, 0.0]
        ms_cb = time_device(lambda: torch.matmul(a_full, B.T, out=C), n_sus, 3, dist, stream, wall=t_cb)
        del a_full
        res["sustained"]["cublas_gemm"] = {
            "value": round(aggregate(ms_cb, flops, dist)[0], 2), "unit": "TFLOP/s", "steps": n_sus,
            "region_s": round(t_cb[1] - t_cb[0], 3),
            "note": "context: torch.matmul (cuBLAS) on the gathered A, same shapes, timed right after the "
                    "fused region; the fused figure includes the gather, this one does not"}
        res["sustained"]["fused_over_cublas_gemm"] = round(ms_cb / ms_sus, 4)
        # the other tile width over a region as long, so that each settles at its own clock
        other = 256 if plan["tile_n"] == 512 else 512
        t_ot = [0.0, 0.0]
        ms_ot = time_device(lambda: call("fused", tile_n=other), n_sus, 3, dist, stream, wall=t_ot)
        check_device_status(ws, f"the sustained {other}-column region")
        res["sustained"][f"tile_{other}"] = {
            "value": round(aggregate(ms_ot, flops, dist)[0], 2), "unit": "TFLOP/s", "steps": n_sus,
            "region_s": round(t_ot[1] - t_ot[0], 3),
            "note": f"the same fused call on {other}-column tiles, timed right after; the main figure uses "
                    f"{plan['tile_n']}-column tiles (tile_n = 0: the library's rule)"}
    res["clocks"] = sampler.stop(window=tuple(t_value))
    if "sustained" in res and sampler.lines:
        cs = clock_summary(sampler.lines, tuple(t_sus))
        if cs is not None:
            res["sustained"]["clocks"] = {"sm_mhz": cs["sm_mhz"], "samples": cs["samples_in_value_region"],
                                          "reasons": cs["reasons"]}
        cs = clock_summary(sampler.lines, tuple(t_cb))
        if cs is not None:
            res["sustained"]["cublas_gemm"]["clocks"] = {"sm_mhz": cs["sm_mhz"],
                                                         "samples": cs["samples_in_value_region"],
                                                         "reasons": cs["reasons"]}
        key = f"tile_{256 if plan['tile_n'] == 512 else 512}"
        cs = clock_summary(sampler.lines, tuple(t_ot))
        if cs is not None:
            res["sustained"][key]["clocks"] = {"sm_mhz": cs["sm_mhz"], "samples": cs["samples_in_value_region"],
                                               "reasons": cs["reasons"]}

    if not args.quick:
        res["other_workloads"] = bench_other_workloads(dev, stream, dist, args, peaks)
        res["e2e"] = bench_e2e(cfg, shards_h, B_h, a, progress, ws, order, delay, dev, stream, dist, args)
        if dist.rank == 0 and dist.world == 1:
            res["cpu_baseline"] = cpu_baseline(cfg, shards_h, B_h)
            res["cpu_baseline_tgather"] = cpu_baseline_tgather(TG_CONFIGS["bw_f16"])
            res["cpu_baseline_square"] = cpu_baseline_square()
    del shards, B, C, a
    torch.cuda.empty_cache()
    return res


def gemm_vs_cublas(cfg, dev, args):
    """The library's plain GEMM (MM_ONLY) and torch.matmul (cuBLAS) on the same gathered A and
    B: two calls of each, then one of each, so that an ncu capture skipping the first four
    launches sees one launch of each.  Prints their times for the record."""
    import torch

    import tile_gather_comm_gb300 as tgc
    from tile_gather_comm_gb300.workloads import make_ag_inputs

    sh, Bh = make_ag_inputs(cfg, seed=0)
    shards = [x.to(dev) for x in sh]
    B = Bh.to(dev)
    C = torch.empty(cfg.M, cfg.N, dtype=torch.bfloat16, device=dev)
    a = torch.cat(shards)
    progress = torch.zeros(max(1, cfg.nblocks), dtype=torch.int32, device=dev)

    def ours():
        tgc.tgc_ag_matmul_ex(shards, B, C, a, cfg.cb, mode="mm_only", progress=progress, epoch=1)

    def cublas():
        torch.matmul(a, B.T, out=C)
    ms = {}
    for name, f in (("mm_only", ours), ("mm_only", ours), ("cublas", cublas), ("cublas", cublas),
                    ("mm_only", ours), ("cublas", cublas)):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        f()
        e1.record()
        torch.cuda.synchronize()
        ms[name] = e0.elapsed_time(e1)
    return {"metric": METRIC, "unit": "ms", "workload": cfg.name, "note": "plain GEMM vs cuBLAS, one call each "
            "after two warm-up calls (profiling run)", "mm_only_ms": round(ms["mm_only"], 4),
            "cublas_ms": round(ms["cublas"], 4)}


def bench_other_workloads(dev, stream, dist, args, peaks):
    """The square and MLP-up AllGather-MatMul workloads: fused (page pivot), fused (ready
    queue), unfused and mm_only, TFLOP/s, timed interleaved.  Their inputs (up to 0.5 GB)
    also exceed L2."""
    import torch

    import tile_gather_comm_gb300 as tgc
    from tile_gather_comm_gb300.workloads import AG_CONFIGS, make_ag_inputs

    out = {}
    for name in ("square", "mlp_up"):
        cfg = AG_CONFIGS[name]
        sh, Bh = make_ag_inputs(cfg, seed=0)
        shards = [x.to(dev) for x in sh]
        B = Bh.to(dev)
        C = torch.empty(cfg.M, cfg.N, dtype=torch.bfloat16, device=dev)
        a = torch.empty(cfg.M, cfg.K, dtype=torch.bfloat16, device=dev)
        progress = torch.zeros(cfg.nblocks, dtype=torch.int32, device=dev)
        ws = torch.zeros(tgc.tgc_ag_matmul_workspace_bytes(cfg.R, cfg.M, cfg.K, cfg.N, cfg.cb),
                         dtype=torch.uint8, device=dev)
        ep = [0]

        def call(mode, pivot="page"):
            ep[0] += 1
            tgc.tgc_ag_matmul_ex(shards, B, C, a, cfg.cb, mode=mode, pivot=pivot, progress=progress,
                                 epoch=ep[0], workspace=ws, stream=stream)
        med = time_interleaved({"fused": lambda: call("fused", "auto"),
                                "fused_page": lambda: call("fused", "page"),
                                "fused_ready_queue": lambda: call("fused", "ready_queue"),
                                "unfused": lambda: call("unfused"), "mm_only": lambda: call("mm_only")},
                               max(args.steps, 300), dist, stream, rounds=10)
        check_device_status(ws, f"the {name} lines")
        line = {k: round(aggregate(v, float(cfg.flops), dist)[0], 1) for k, v in med.items()}
        line["unit"] = "TFLOP/s"
        line["fused_is"] = "the default call: tile order TGC_PIVOT_AUTO (as tgc_ag_matmul)"
        line["fused_over_unfused"] = round(med["unfused"] / med["fused"], 4)
        line["fused_page_over_unfused"] = round(med["unfused"] / med["fused_page"], 4)
        line["fused_ready_queue_over_unfused"] = round(med["unfused"] / med["fused_ready_queue"], 4)
        line["config"] = f"{cfg.R} x ({cfg.H},{cfg.K}) shards, B ({cfg.N},{cfg.K}), cb={cfg.cb}"
        out[name] = line
        del shards, B, C, a
    return out


def bench_tgather_strided(tcfg, dev, dist, peaks, peaks_kind, pad: int = 64):
    """tgc_tgather_strided on the TGATHER workload's sizes with every source a view of
    rows padded by `pad` elements (row pitch W + pad) and the destination a view of a
    padded buffer too, graph-replayed over rotating buffer sets > 4 x L2."""
    import torch

    import tile_gather_comm_gb300 as tgc
    from tile_gather_comm_gb300.workloads import make_tg_inputs

    srcs_h = make_tg_inputs(tcfg, seed=0)
    D0, D1, D2, H, W = tcfg.shape
    per_set = tcfg.bytes_moved
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    nsets = max(2, -(-4 * l2 // per_set))
    sets = []
    for _ in range(nsets):
        srcs = []
        for s in srcs_h:
            buf = torch.empty((D0, D1, D2, H, W + pad), dtype=tcfg.dtype, device=dev)
            buf[..., :W].copy_(s.to(dev))
            srcs.append(buf[..., :W])
        dbuf = torch.empty((D0, D1, D2, tcfg.nranks * H, W + pad), dtype=tcfg.dtype, device=dev)
        sets.append((dbuf[..., :W], srcs))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for dst, srcs in sets:
            tgc.tgc_tgather_strided(dst, srcs, stream=s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for dst, srcs in sets:
                tgc.tgc_tgather_strided(dst, srcs, stream=s)
    torch.cuda.synchronize()
    reps = max(3, -(-400 // nsets))
    ms = time_device(lambda: g.replay(), reps, 3, dist, torch.cuda.current_stream()) / nsets
    gbs, _ = aggregate(ms, per_set, dist, scale=1e-9)
    per_gpu = per_set / (ms * 1e-3) * 1e-9
    out = {
        "value": round(gbs, 1), "unit": "GB/s", "us_per_launch": round(ms * 1e3, 3),
        "config": f"{tcfg.nranks} x {str(tcfg.dtype).replace('torch.', '')} {tcfg.shape} views with row pitch "
                  f"W+{pad} -> a destination view with row pitch W+{pad}",
        "bytes_per_launch": per_set, "buffer_sets": nsets, "launches_timed": reps * nsets,
        "roofline": {"bound": "hbm", "achieved": round(per_gpu, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(per_gpu / peaks["hbm_gbs"], 4),
                     "traffic": profiled_traffic(f"tgather_strided/{tcfg.name}", TGATHER_SOURCES),
                     "peak_source": f"{peaks_kind} STREAM-style copy", "kernel": "tgather_strided_rows_kernel<32>"},
    }
    del sets, g
    return out


def bench_tgather_release(tcfg, dev, dist, peaks, peaks_kind, chunk_rows: int = 128):
    """tgc_tgather_ex with per-chunk progress release (chunks of `chunk_rows` rows, the
    per-chunk counters and a gpu-scope release per chunk) on the TGATHER workload, graph-
    replayed over rotating buffer sets > 4 x L2 like the plain TGATHER line."""
    import torch

    import tile_gather_comm_gb300 as tgc
    from tile_gather_comm_gb300.workloads import make_tg_inputs

    srcs_h = make_tg_inputs(tcfg, seed=0)
    D0, D1, D2, H, W = tcfg.shape
    per_set = tcfg.bytes_moved
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    nsets = max(2, -(-4 * l2 // per_set))
    nchunks = tcfg.nranks * -(-H // chunk_rows)
    sets = []
    for _ in range(nsets):
        srcs = [x.to(dev) for x in srcs_h]
        dst = torch.empty((D0, D1, D2, tcfg.nranks * H, W), dtype=tcfg.dtype, device=dev)
        progress = torch.zeros(nchunks, dtype=torch.int32, device=dev)
        counters = torch.zeros(nchunks, dtype=torch.int32, device=dev)
        sets.append((dst, srcs, progress, counters))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    # two graphs, epochs 2 and 3, replayed in turn: every launch publishes a value its flags do
    # not hold on entry, as the call requires
    graphs = []
    with torch.cuda.stream(s):
        for dst, srcs, progress, counters in sets:
            tgc.tgc_tgather_ex(dst, srcs, progress=progress, counters=counters, chunk_rows=chunk_rows, epoch=1,
                               stream=s)
        torch.cuda.synchronize()
        for epoch in (2, 3):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for dst, srcs, progress, counters in sets:
                    tgc.tgc_tgather_ex(dst, srcs, progress=progress, counters=counters, chunk_rows=chunk_rows,
                                       epoch=epoch, stream=s)
            graphs.append(g)
    torch.cuda.synchronize()
    turn = [0]

    def replay():
        graphs[turn[0] % 2].replay()
        turn[0] += 1

    reps = max(3, -(-400 // nsets))
    ms = time_device(replay, reps, 3, dist, torch.cuda.current_stream()) / nsets
    gbs, _ = aggregate(ms, per_set, dist, scale=1e-9)
    per_gpu = per_set / (ms * 1e-3) * 1e-9
    last_epoch = 2 + (turn[0] - 1) % 2
    released = all(bool(torch.all(x[2] == last_epoch)) for x in sets)
    out = {
        "value": round(gbs, 1), "unit": "GB/s", "us_per_launch": round(ms * 1e3, 3),
        "config": f"{tcfg.nranks} x {str(tcfg.dtype).replace('torch.', '')} {tcfg.shape}, progress released per "
                  f"{chunk_rows}-row chunk ({nchunks} flags)",
        "bytes_per_launch": per_set, "buffer_sets": nsets, "launches_timed": reps * nsets,
        "all_flags_released": released,
        "roofline": {"bound": "hbm", "achieved": round(per_gpu, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(per_gpu / peaks["hbm_gbs"], 4),
                     "traffic": profiled_traffic(f"tgather_release/{tcfg.name}", TGATHER_SOURCES),
                     "peak_source": f"{peaks_kind} STREAM-style copy", "kernel": "tgather_kernel<16>"},
    }
    del sets, graphs
    return out


def bench_tgather(tcfg, dev, stream, dist, peaks, peaks_kind, args):
    """TGATHER throughput, (bytes read + bytes written) / time, over rotating buffer sets > 2 x L2,
    launched from a CUDA graph so that launch gaps do not inflate the kernel time."""
    import torch

    import tile_gather_comm_gb300 as tgc
    from tile_gather_comm_gb300.workloads import make_tg_inputs

    srcs_h = make_tg_inputs(tcfg, seed=0)
    D0, D1, D2, H, W = tcfg.shape
    per_set = tcfg.bytes_moved
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    nsets = max(2, -(-4 * l2 // per_set))
    sets = []
    for i in range(nsets):
        srcs = [s.to(dev) for s in srcs_h]
        dst = torch.empty((D0, D1, D2, tcfg.nranks * H, W), dtype=tcfg.dtype, device=dev)
        sets.append((dst, srcs))
    for dst, srcs in sets:
        tgc.tgc_tgather(dst, srcs, stream=stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(stream)
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for dst, srcs in sets:
                tgc.tgc_tgather(dst, srcs, stream=s)
    torch.cuda.synchronize()
    reps = max(3, -(-400 // nsets))
    ms_graph = time_device(lambda: g.replay(), reps, 3, dist, torch.cuda.current_stream())
    ms = ms_graph / nsets
    gbs, _ = aggregate(ms, per_set, dist, scale=1e-9)
    per_gpu = per_set / (ms * 1e-3) * 1e-9

    out = {
        "value": round(gbs, 1), "unit": "GB/s", "us_per_launch": round(ms * 1e3, 3),
        "config": f"{tcfg.nranks} x {str(tcfg.dtype).replace('torch.', '')} {tcfg.shape} -> dst DIM_3 x{tcfg.nranks}",
        "bytes_per_launch": per_set, "buffer_sets": nsets, "launches_timed": reps * nsets,
        "roofline": {"bound": "hbm", "achieved": round(per_gpu, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(per_gpu / peaks["hbm_gbs"], 4),
                     "traffic": profiled_traffic(f"tgather_flat/{tcfg.name}", TGATHER_SOURCES),
                     "peak_source": f"{peaks_kind} STREAM-style copy", "kernel": "tgather_flat_kernel<32>"},
    }
    del sets, g
    return out


def bench_tgather_context_long(dev, stream, dist, peaks, peaks_kind, args):
    """Context line: the TGATHER kernel on 8x taller sources, where the per-launch start and
    drain (about 2 us, fixed) weigh 8x less."""
    import torch

    from tile_gather_comm_gb300.workloads import TGConfig

    long_cfg = TGConfig("bw_f16_long", 8, (2, 1, 1, 8192, 1024), torch.float16, "normal")
    out = bench_tgather(long_cfg, dev, stream, dist, peaks, peaks_kind, args)
    out["note"] = ("context only: 8 x fp16 (2,1,1,8192,1024), 8x the rows of the TGATHER workload; "
                   "per-launch start and drain amortised")
    return out


def bench_e2e(cfg, shards_h, B_h, a, progress, ws, order, delay, dev, stream, dist, args):
    """The public call with host buffers, pipelined the way an application streams batches:
    every step copies its shards and B from pinned host memory (H2D stream), runs the fused
    call on them (compute stream), and copies C back to pinned host memory (D2H stream).
    Two device buffer sets let step i+1's inputs and step i-1's result move while step i
    computes; the timed region covers `steps` complete steps (first H2D to last D2H)."""
    import torch

    import tile_gather_comm_gb300 as tgc

    hs = [s.pin_memory() for s in shards_h]
    hB = B_h.pin_memory()
    hC = [torch.empty(cfg.M, cfg.N, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    sets = []
    for _ in range(2):
        sets.append(([torch.empty_like(s, device=dev) for s in hs], torch.empty_like(hB, device=dev),
                     torch.empty(cfg.M, cfg.N, dtype=torch.bfloat16, device=dev)))
    h2d = sum(s.numel() * 2 for s in hs) + hB.numel() * 2
    d2h = cfg.M * cfg.N * 2
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    epoch = [10_000_000]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for e in ev_out:
        e.record(s_out)

    def step(i):
        k = i % 2
        ds, dB, dC = sets[k]
        s_in.wait_event(ev_done[k])          # the set's previous kernel has consumed its inputs
        with torch.cuda.stream(s_in):
            for d, h in zip(ds, hs):
                d.copy_(h, non_blocking=True)
            dB.copy_(hB, non_blocking=True)
        ev_in[k].record(s_in)
        stream.wait_event(ev_in[k])
        stream.wait_event(ev_out[k])         # the set's previous result has been copied out
        epoch[0] += 1
        tgc.tgc_ag_matmul_ex(ds, dB, dC, a, cfg.cb, progress=progress, epoch=epoch[0], workspace=ws,
                             order=order, delay_ns=delay, stream=stream)
        ev_done[k].record(stream)
        s_out.wait_event(ev_done[k])
        with torch.cuda.stream(s_out):
            hC[k].copy_(dC, non_blocking=True)
        ev_out[k].record(s_out)

    steps = max(4, min(args.steps, 20))
    for i in range(2):
        step(i)
    torch.cuda.synchronize()
    dist.barrier()
    t0 = time.perf_counter()
    for i in range(steps):
        step(i)
    torch.cuda.synchronize()
    ms = (time.perf_counter() - t0) * 1e3 / steps
    check_device_status(ws, "the end-to-end region")
    dist.barrier()
    # raw pinned-copy rates on this machine, for context
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    sets[0][1].copy_(hB, non_blocking=True)
    e1.record(s_in)
    torch.cuda.synchronize()
    h2d_gbs = hB.numel() * 2 / (e0.elapsed_time(e1) * 1e-3) * 1e-9
    e0.record(s_out)
    hC[0].copy_(sets[0][2], non_blocking=True)
    e1.record(s_out)
    torch.cuda.synchronize()
    d2h_gbs = d2h / (e0.elapsed_time(e1) * 1e-3) * 1e-9
    # a step's copies alone, both directions at once (no kernel): the host link's bound on a step
    both = []
    for _ in range(3):
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        with torch.cuda.stream(s_in):
            for d, h in zip(sets[0][0], hs):
                d.copy_(h, non_blocking=True)
            sets[0][1].copy_(hB, non_blocking=True)
        with torch.cuda.stream(s_out):
            hC[1].copy_(sets[1][2], non_blocking=True)
        torch.cuda.synchronize()
        both.append(time.perf_counter() - t1)
    both_ms = statistics.median(both) * 1e3
    val, ms_max = aggregate(ms, float(cfg.flops), dist)
    return {"value": round(val, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(ms_max, 3), "steps": steps,
            "call": "tgc_ag_matmul_ex on a compute stream; pinned H2D and D2H on their own streams, "
                    "two device buffer sets (steps overlap)",
            "h2d_gbs": round(h2d_gbs, 1), "d2h_gbs": round(d2h_gbs, 1),
            "copies_only_ms": round(both_ms, 3),
            "copies_only_gbs": round((h2d + d2h) / (both_ms * 1e-3) * 1e-9, 1),
            "frac_of_copies_only": round(both_ms / ms_max, 3),
            "copies_only_note": "one step's H2D and D2H issued together with no kernel (median of 3): the "
                                "host link's bound on a step on this box, at this time"}


def cpu_baseline(cfg, shards_h, B_h, target_rows: int | None = None):
    """The oracle as it stands, on a bounded sample of output rows (all N columns, full K)."""
    import numpy as np
    import torch

    import oracle
    from tile_gather_comm_gb300.workloads import sample_rows

    oracle.build()
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    sh = [bits(s) for s in shards_h]
    Bb = bits(B_h)
    # about 10 s of host work at the large workload's size: every comm block's first and last
    # row plus seeded random rows of each block
    per_block = max(0, (2048 // max(1, cfg.nblocks)) - 2)
    rows = sample_rows(cfg, seed=0, per_block_random=per_block)
    if target_rows is not None:
        rows = rows[:target_rows]
    t0 = time.perf_counter()
    oracle.ag_matmul_rows(sh, Bb, rows)
    dt = time.perf_counter() - t0
    fl = 2.0 * len(rows) * cfg.N * cfg.K
    out = {"value": round(fl / dt * 1e-12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
           "kind": "oracle", "seconds": round(dt, 3),
           "sample": f"{len(rows)} rows of C (first and last row of each of the {cfg.nblocks} comm blocks plus "
                     f"{per_block} seeded random rows of each), all {cfg.N} columns, full K={cfg.K}; "
                     f"fp32 sequential-k dot products, OpenMP over rows",
           # the whole C at the sampled rate (labelled: not measured)
           "extrapolated_full_s": round(float(cfg.flops) / (fl / dt), 1)}
    # the same oracle on one host thread, on the first rows of that sample (a few seconds)
    threads = oracle.num_threads()
    one = rows[: max(1, min(len(rows), 16))]
    oracle.set_num_threads(1)
    try:
        t0 = time.perf_counter()
        oracle.ag_matmul_rows(sh, Bb, one)
        dt1 = time.perf_counter() - t0
    finally:
        oracle.set_num_threads(threads)
    out["single_thread"] = {"value": round(2.0 * len(one) * cfg.N * cfg.K / dt1 * 1e-12, 6), "unit": "TFLOP/s",
                            "cores": 1, "seconds": round(dt1, 3), "sample": f"the first {len(one)} rows of that sample"}
    return out


def cpu_baseline_tgather(tcfg, reps: int = 5):
    """The TGATHER oracle (element-wise byte copy) on the full workload, host cores."""
    import oracle
    from tile_gather_comm_gb300.workloads import make_tg_inputs

    oracle.build()
    srcs = [s.numpy() for s in make_tg_inputs(tcfg, seed=0)]
    oracle.tgather(srcs)
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.tgather(srcs)
    dt = (time.perf_counter() - t0) / reps
    out = {"value": round(tcfg.bytes_moved / dt * 1e-9, 2), "unit": "GB/s", "cores": oracle.num_threads(),
           "kind": "oracle", "seconds": round(dt * reps, 3),
           "sample": f"the full {tcfg.name} workload ({tcfg.bytes_moved} bytes read + written), {reps} runs"}
    threads = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        t0 = time.perf_counter()
        oracle.tgather(srcs)
        dt1 = time.perf_counter() - t0
    finally:
        oracle.set_num_threads(threads)
    out["single_thread"] = {"value": round(tcfg.bytes_moved / dt1 * 1e-9, 2), "unit": "GB/s", "cores": 1,
                            "seconds": round(dt1, 3), "sample": "one run of the same workload"}
    return out


def cpu_baseline_square():
    """The AllGather-MatMul oracle on the whole square workload (every row of C), host cores;
    on one thread, the first 16 rows of C."""
    import numpy as np
    import torch

    import oracle
    from tile_gather_comm_gb300.workloads import AG_CONFIGS, make_ag_inputs

    oracle.build()
    cfg = AG_CONFIGS["square"]
    shards_h, B_h = make_ag_inputs(cfg, seed=0)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    sh = [bits(x) for x in shards_h]
    Bb = bits(B_h)
    t0 = time.perf_counter()
    oracle.ag_matmul(sh, Bb)
    dt = time.perf_counter() - t0
    out = {"value": round(cfg.flops / dt * 1e-12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
           "kind": "oracle", "seconds": round(dt, 3),
           "sample": f"the full square workload: {cfg.R} x ({cfg.H},{cfg.K}) shards, B ({cfg.N},{cfg.K}), every "
                     f"row of C; fp32 sequential-k dot products, OpenMP over rows"}
    threads = oracle.num_threads()
    rows = list(range(16))
    oracle.set_num_threads(1)
    try:
        t0 = time.perf_counter()
        oracle.ag_matmul_rows(sh, Bb, rows)
        dt1 = time.perf_counter() - t0
    finally:
        oracle.set_num_threads(threads)
    out["single_thread"] = {"value": round(2.0 * len(rows) * cfg.N * cfg.K / dt1 * 1e-12, 6), "unit": "TFLOP/s",
                            "cores": 1, "seconds": round(dt1, 3), "sample": "the first 16 rows of C"}
    return out


# ----------------------------------------------------------------------------- reference arm (the oracle)


def run_reference(args, dist: Dist):
    import numpy as np
    import torch

    import oracle
    from tile_gather_comm_gb300.workloads import AG_CONFIGS, make_ag_inputs, sample_rows

    cfg = AG_CONFIGS[args.workload]
    oracle.build()
    threads = oracle.num_threads()
    shards_h, B_h = make_ag_inputs(cfg, seed=0)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    sh = [bits(s) for s in shards_h]
    Bb = bits(B_h)
    all_rows = sample_rows(cfg, seed=0, per_block_random=0)
    per_step = max(1, min(threads, len(all_rows)))  # one row per thread per step
    times = []
    for i in range(args.warmup + args.steps):
        rows = [all_rows[(i * per_step + j) % len(all_rows)] for j in range(per_step)]
        t0 = time.perf_counter()
        oracle.ag_matmul_rows(sh, Bb, rows)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    sec = sum(times) / len(times)
    fl = 2.0 * per_step * cfg.N * cfg.K
    val = fl / sec * 1e-12
    return {
        "metric": METRIC, "value": round(val, 6), "unit": "TFLOP/s", "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "impl": "reference",
        "config": {"workload": f"{cfg.name} (CPU oracle on a row sample)", "M": cfg.M, "N": cfg.N, "K": cfg.K,
                   "R": cfg.R, "comm_block_rows": cfg.cb},
        "cpu_baseline": {"value": round(val, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{per_step} rows of C per step (comm-block first/last rows in turn), all "
                                   f"{cfg.N} columns, full K={cfg.K}"},
        "e2e": {"value": round(val, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        # the CPU oracle runs on rank 0 alone; other ranks exit at once without work
        dist = Dist(init=False)
        if dist.rank != 0:
            return 0
        print(json.dumps(run_reference(args, dist)), flush=True)
        return 0
    dist = Dist()
    try:
        res = run_ours(args, dist)
        if dist.rank == 0:
            print(json.dumps(res), flush=True)
    finally:
        dist.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
