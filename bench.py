#!/usr/bin/env python
"""Benchmark of the training RMSNorm backward on one GB300 (per rank).

Default workload: T = 65536 tokens, H = 2048, x BF16 ~ N(0, 1) with 1 % of the
rows scaled by 30 (outlier family), dy BF16 ~ N(0, 1e-2), w FP32; one step is
one deterministic backward (main kernel + fixed-order dw reduce) through the
C ABI.  Printed as one JSON line on rank 0.

  value         achieved GB/s = algorithmic bytes of the step / its device
                time (inputs resident in HBM, L2 flushed before every step)
  e2e           the same metric through the C ABI from pinned host buffers:
                the host->device copies of the step's inputs and the
                device->host copies of dx and dw are inside the timed region
  roofline      the main kernel alone, timed with CUDA events on its stream,
                against the measured HBM copy bandwidth
  cpu_baseline  the FP64 CPU oracle on a bounded sample of the same workload

``--impl reference`` times the oracle instead (host cores, a bounded sample
per step) and prints the reference line.  ``--profile`` runs a minimal launch
sequence for ncu.  Under torchrun each rank runs an independent replica (the
path has no cross-GPU exchange on one box); value sums the ranks' bytes over
the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "bwd µs & achieved HBM GB/s (fraction of GB300 peak) per (H,T,w dtype,det mode)"
WORKLOAD = "h2048_t65536_outlier_w32"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20
ACCUM = {"plain": 0, "blocked": 1, "twosum": 2, "kahan": 3}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", choices=["det", "nondet", "fwd", "main", "all"], default=None,
                    help="run only the named loop(s) with few launches (for ncu); prints per-call times")
    ap.add_argument("--accum", choices=sorted(ACCUM), default=None,
                    help="with --profile: force the per-thread dw accumulation form")
    ap.add_argument("--graph", action="store_true",
                    help="with --profile: time CUDA-graph replays of one call (no host launch cost)")
    return ap.parse_args(argv)


# ------------------------------------------------------------------ helpers

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def workload_bytes(R: int, H: int, w_bytes: int, P: int, dh: bool = False, res: bool = False):
    """Algorithmic bytes.  Backward: x (or h_new), dy read and dx written once
    (2 bytes per element each; dh adds 2 more), rstd read (4 per row), w read,
    dw written (4 per column) and the pair's CTA partials (8 bytes per column
    per CTA) written by the main kernel and read back by the reduce.
    Forward: x read, y written, rstd written, w read; the residual route adds
    the residual read and h_new written."""
    act = (8 if dh else 6) * R * H
    rows = 4 * R
    part = 8 * P * H
    return {
        "pair": act + rows + w_bytes + 4 * H + 2 * part,
        "main": act + rows + w_bytes + part,
        "single": act + rows + w_bytes + 4 * H + part,
        "rows_only": act + rows + w_bytes + 4 * H,
        "fwd": (8 if res else 4) * R * H + rows + w_bytes,
    }


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    csrc = os.path.join(ROOT, "bwd_dw_column_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def traffic_record(kernel: str, workload: str):
    """The committed ncu record (DRAM bytes per launch, the summary file) when
    it holds for the current kernel sources; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)
    except Exception:
        return None
    ent = rec.get(f"{kernel}:{workload}")
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary when it was taken
    on the current kernel sources; else None."""
    ent = traffic_record(kernel, workload)
    return ent.get("dram_bytes_per_launch") if ent else None


class ClockSampler:
    """nvidia-smi clock / throttle samples (200 ms) while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.3)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.out.close()

    def summary(self):
        if self.proc is None:
            return None
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def make_step_fns(cake, torch, case, dev, accum=None):
    """Forward / backward callables for one workload, outputs preallocated."""
    x, dy, w, eps = case["x"], case["dy"], case["w"], case["eps"]
    res = case.get("residual")
    dh = case.get("dh")
    out = cake.cake_rmsnorm_fwd(x, w, eps, residual=res)
    y, rstd = out[0], out[1]
    hn = out[2] if res is not None else None
    h = hn if res is not None else x
    ws = cake.cake_rmsnorm_bwd_workspace(h, w.dtype, deterministic=False)
    dx = torch.empty(h.shape, dtype=torch.bfloat16, device=dev)
    dw = torch.empty(h.shape[-1], dtype=torch.float32, device=dev)

    def bwd(det):
        if accum is None:
            return lambda: cake.cake_rmsnorm_bwd(dy, h, rstd, w, dh, deterministic=det, workspace=ws, dx=dx, dw=dw)
        return lambda: cake.cake_rmsnorm_bwd_forced(dy, h, rstd, w, dh, deterministic=det, force_single=int(not det),
                                                   force_accum=accum, workspace=ws, dx=dx, dw=dw)

    def forced(form):
        return lambda: cake.cake_rmsnorm_bwd_forced(dy, h, rstd, w, dh, deterministic=form != 1, force_single=form,
                                                   force_accum=accum, workspace=ws, dx=dx, dw=dw)

    def fwd():
        return cake.cake_rmsnorm_fwd(x, w, eps, residual=res, y=y, rstd=rstd, h_new=hn)

    return {
        "fwd": fwd,
        "det": bwd(True),
        "nondet": bwd(False),
        "single_atomic": forced(1),
        "single_grid": forced(3),
        # the checkpointed step of the pages' GB300 tables: forward, forward
        # recompute, deterministic backward
        "ckpt": lambda: (fwd(), fwd(), bwd(True)()),
        "main": lambda: cake.cake_rmsnorm_bwd_main(dy, h, rstd, w, dh, workspace=ws, dx=dx, dw=dw, force_accum=accum),
        "h": h, "rstd": rstd, "ws": ws, "dx": dx, "dw": dw,
    }


def aggregate_times(times, world, device):
    """(max over ranks of the total ms, max over ranks of the mean ms): the
    job takes as long as its slowest rank."""
    import torch
    import torch.distributed as dist

    tot = torch.tensor([sum(times), statistics.mean(times)], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(tot, op=dist.ReduceOp.MAX)
    return float(tot[0]), float(tot[1])


def replica_gbs(bytes_per_step, steps, world, slowest_total_ms):
    """Whole-job GB/s of `world` replicas that each ran `steps` steps."""
    return world * steps * bytes_per_step / (slowest_total_ms * 1e-3) / 1e9


class L2Flush:
    """Leaves L2 holding none of a step's data, and no dirty lines.

    A write of a buffer larger than L2 evicts the step's inputs; a read of a
    second such buffer then evicts the written lines, so their write-back
    happens before the timed region instead of inside it (the state ncu's
    flush-and-invalidate cache control gives a kernel)."""

    def __init__(self, torch, dev, nbytes=None):
        n = nbytes or L2_FLUSH_BYTES
        self.w = torch.empty(n, dtype=torch.uint8, device=dev)
        self.r = torch.ones(n // 4, dtype=torch.float32, device=dev)
        self.out = torch.empty((), dtype=torch.float32, device=dev)
        self.torch = torch

    def __call__(self, k):
        self.w.fill_(k & 0xFF)
        self.torch.sum(self.r, dim=0, out=self.out)


def time_loop(torch, fn, steps, warmup, flush, stream):
    """Per-step device times (ms) of fn(), the L2 flushed before every step.

    The warm-up steps repeat the timed sequence (flush, then the step), so
    first-use costs of either stay out of the timed region."""
    for k in range(warmup):
        if flush is not None:
            flush(k)
        fn()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for k in range(steps):
        if flush is not None:
            flush(k)
        starts[k].record(stream)
        fn()
        ends[k].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


# ---------------------------------------------------------- our CUDA path

def describe(spec) -> str:
    kind = spec["kind"]
    wd = "w FP32" if spec["w_dtype"] is not None and str(spec["w_dtype"]).endswith("float32") else "w BF16"
    if kind == "plain":
        fam = {"gauss": "N(0,1)", "outlier": "N(0,1), 1% rows x30", "offset": "3+N(0,1)"}[spec["family"]]
        return f"x BF16 {fam}; dy BF16 N(0, std {spec['dy_std']:g}); {wd} 1+0.1N(0,1); eps 1e-6"
    if kind == "res":
        return f"x BF16 N(0,1), residual N(0, std 0.5), dy and dh BF16 N(0,1); {wd} 1+0.1N(0,1); eps 1e-6"
    view = "strided slice of [T,24,512]" if spec.get("strided") else "contiguous"
    return f"[T,{spec['heads']},256] {view}, x 3+N(0,1), dy N(0,1); shared {wd}[256]; eps 1e-6"


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    import bwd_dw_column_gb300 as cake
    import cake_inputs

    spec = cake_inputs.WORKLOADS[args.workload]
    case = cake_inputs.make(args.workload, seed=rank, device=dev)
    x, dy, w = case["x"], case["dy"], case["w"]
    dh, res = case.get("dh"), case.get("residual")
    fns = make_step_fns(cake, torch, case, dev)
    h, rstd, ws, dx, dw = fns["h"], fns["rstd"], fns["ws"], fns["dx"], fns["dw"]
    T = x.shape[0]
    nh = x.shape[1] if x.dim() == 3 else 1
    H = x.shape[-1]
    R = T * nh
    variant = cake.cake_rmsnorm_bwd_select((T, nh, H), w.dtype, deterministic=True, has_dh=dh is not None)
    nd_variant = cake.cake_rmsnorm_bwd_select((T, nh, H), w.dtype, deterministic=False, has_dh=dh is not None)
    nbytes = workload_bytes(R, H, w.numel() * w.element_size(), variant["ctas"], dh=dh is not None,
                            res=res is not None)
    flush = L2Flush(torch, dev)
    stream = torch.cuda.current_stream()
    K, Wm = args.steps, max(3, args.warmup)

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_det = time_loop(torch, fns["det"], K, Wm, flush, stream)
        t_main = time_loop(torch, fns["main"], K, Wm, flush, stream)
        t_nd = time_loop(torch, fns["nondet"], K, Wm, flush, stream)
        t_sa = time_loop(torch, fns["single_atomic"], K, Wm, flush, stream)
        t_sg = time_loop(torch, fns["single_grid"], K, Wm, flush, stream)
        t_fwd = time_loop(torch, fns["fwd"], K, Wm, flush, stream)
        t_ck = time_loop(torch, fns["ckpt"], K, Wm, flush, stream)
    torch.cuda.synchronize()
    clocks = clk.summary()

    # end to end through the C ABI from pinned host buffers: every step copies
    # the backward's inputs in and dx, dw out
    def host(t):
        if t is None:
            return None
        if not t.is_contiguous():  # a strided view travels as its whole buffer
            t = t.as_strided((t.untyped_storage().nbytes() // t.element_size(),), (1,), 0)
        return t.cpu().pin_memory()

    hx, hdy, hdh, hrstd, hw = (host(t) for t in (h, dy, dh, rstd, w))
    hdx = torch.empty(dx.shape, dtype=torch.bfloat16).pin_memory()
    hdw = torch.empty(H, dtype=torch.float32).pin_memory()
    bx = torch.empty(hx.shape, dtype=hx.dtype, device=dev)
    x2 = bx if h.is_contiguous() else bx.as_strided(h.shape, h.stride(), h.storage_offset())
    dy2, r2, w2, dx2 = (torch.empty_like(t) for t in (dy, rstd, w, dx))
    dh2 = torch.empty_like(dh) if dh is not None else None

    def e2e_step():
        bx.copy_(hx, non_blocking=True)
        dy2.copy_(hdy, non_blocking=True)
        if dh2 is not None:
            dh2.copy_(hdh, non_blocking=True)
        r2.copy_(hrstd, non_blocking=True)
        w2.copy_(hw, non_blocking=True)
        cake.cake_rmsnorm_bwd(dy2, x2, r2, w2, dh2, deterministic=True, workspace=ws, dx=dx2, dw=dw)
        hdx.copy_(dx2, non_blocking=True)
        hdw.copy_(dw, non_blocking=True)

    t_e2e = time_loop(torch, e2e_step, K, Wm, flush, stream)
    h2d = sum(t.numel() * t.element_size() for t in (hx, hdy, hdh, hrstd, hw) if t is not None)
    d2h = hdx.numel() * 2 + hdw.numel() * 4
    assert cake.cake_rmsnorm_device_status() == 0

    agg = lambda times: aggregate_times(times, world, dev)

    tot_det, mean_det = agg(t_det)
    tot_main, mean_main = agg(t_main)
    tot_nd, mean_nd = agg(t_nd)
    tot_sa, mean_sa = agg(t_sa)
    tot_sg, mean_sg = agg(t_sg)
    nd_bytes = nbytes["pair"] if nd_variant["single"] == 0 else nbytes["single"]
    tot_fwd, mean_fwd = agg(t_fwd)
    tot_ck, mean_ck = agg(t_ck)
    tot_e2e, mean_e2e = agg(t_e2e)
    gbs = lambda b, tot_ms: replica_gbs(b, K, world, tot_ms)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and spec["kind"] == "plain":
        cpu = oracle_baseline(case, T, H, budget_s=10.0)
    if world > 1:
        dist.barrier()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peak, peak_kind = measured_peak()
    achieved_main = nbytes["main"] / (mean_main * 1e-3) / 1e9
    value = gbs(nbytes["pair"], tot_det)
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": Wm,
        "ms_per_step": round(mean_det, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "impl": "ours",
        "config": {
            "workload": args.workload,
            "T": T, "heads": nh, "H": H, "w_dtype": "fp32" if w.dtype == torch.float32 else "bf16",
            "inputs": describe(spec),
            "mode": "deterministic (main + fixed-order reduce)",
            "io_dtype": "bf16 activations, fp32 rstd/dw",
            "l2": "flushed before every timed step (256 MiB write, then 256 MiB read so no dirty line is left)",
            "parallelism": f"{world} independent replicas" if world > 1 else "single GPU",
            "variant": variant,
        },
        "bwd_us": round(mean_det * 1e3, 2),
        "bytes_per_step": nbytes["pair"],
        "frac_of_peak": round(value / world / peak, 4),
        "modes": {
            "det_pair": {"us": round(mean_det * 1e3, 2), "GB/s": round(gbs(nbytes["pair"], tot_det), 1),
                         "bytes": nbytes["pair"]},
            "det_main_kernel": {"us": round(mean_main * 1e3, 2), "GB/s": round(achieved_main, 1),
                                "bytes": nbytes["main"]},
            "nondet": {"us": round(mean_nd * 1e3, 2), "GB/s": round(gbs(nd_bytes, tot_nd), 1),
                       "bytes": nd_bytes, "variant": nd_variant},
            # the single-kernel forms the non-deterministic mode may run
            # (the table picks the pair, which is faster at every measured
            # shape): FP64 L2 atomics, and the cooperative grid form
            "single_atomic": {"us": round(mean_sa * 1e3, 2), "GB/s": round(gbs(nbytes["single"], tot_sa), 1),
                              "bytes": nbytes["single"]},
            "single_grid": {"us": round(mean_sg * 1e3, 2), "GB/s": round(gbs(nbytes["pair"], tot_sg), 1),
                            "bytes": nbytes["pair"]},
            "fwd": {"us": round(mean_fwd * 1e3, 2), "GB/s": round(gbs(nbytes["fwd"], tot_fwd), 1),
                    "bytes": nbytes["fwd"]},
            "ckpt_2xfwd_bwd": {"us": round(mean_ck * 1e3, 2),
                               "GB/s": round(gbs(2 * nbytes["fwd"] + nbytes["pair"], tot_ck), 1),
                               "bytes": 2 * nbytes["fwd"] + nbytes["pair"]},
        },
        "roofline": {
            "bound": "hbm",
            "kernel": "bwd_rows_kernel (main kernel of the deterministic pair)",
            "achieved": round(achieved_main, 1),
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": round(achieved_main / peak, 4),
            "traffic": recorded_traffic("bwd_rows_kernel", args.workload),
            "traffic_summary": (traffic_record("bwd_rows_kernel", args.workload) or {}).get("summary"),
            "algorithmic_bytes": nbytes["main"],
        },
        "e2e": {
            "value": round(gbs(nbytes["pair"], tot_e2e), 1),
            "unit": "GB/s",
            "ms_per_step": round(mean_e2e, 4),
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
        },
        "gpu_launches": K * (2 + 1 + (1 if nd_variant["single"] else 2) + 1 + 1 + 1 + 4 + 2),
        "gpu_launches_detail": {"det": 2 * K, "main_only": K, "nondet": K * (1 if nd_variant["single"] else 2),
                                "single_atomic": K, "single_grid": K, "fwd": K, "ckpt_2xfwd_bwd": 4 * K,
                                "e2e": 2 * K},
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_profile(args):
    """Minimal launch sequence for profiling: inputs, one forward, then the
    chosen loop(s) of warmup + steps calls; no L2 flush, no host copies."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import bwd_dw_column_gb300 as cake
    import cake_inputs

    dev = torch.device("cuda", 0)
    case = cake_inputs.make(args.workload, seed=0, device=dev)
    fns = make_step_fns(cake, torch, case, dev, ACCUM.get(args.accum) if args.accum else None)
    names = ["fwd", "det", "nondet"] if args.profile == "all" else [args.profile]
    out = {}
    stream = torch.cuda.current_stream()
    for n in names:
        fn = fns[n]
        if args.graph:
            fn()  # first call on the device: attributes and addresses set up before capture
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                fns[n]()
            fn = graph.replay
        ts = [t * 1e3 for t in time_loop(torch, fn, args.steps, args.warmup, None, stream)]
        out[n] = {"us_median": round(statistics.median(ts), 2), "us_min": round(min(ts), 2)}
    assert cake.cake_rmsnorm_device_status() == 0
    print(json.dumps({"profile": args.workload, "accum": args.accum, "us_per_call": out}), flush=True)


# ------------------------------------------------------------ the oracle

def oracle_sample(case, H, rows):
    """Seconds the oracle's backward takes on the first `rows` rows (dx of
    those rows and dw over them), its rstd input prepared outside the timing."""
    import numpy as np
    import torch

    import oracle

    x = case["x"][:rows].cpu()
    dy = case["dy"][:rows].cpu()
    w = case["w"].cpu()
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    xv, dyv = oracle.View.contiguous(bits(x)), oracle.View.contiguous(bits(dy))
    wb = w.numpy() if w.dtype == torch.float32 else bits(w)
    _, r64, _ = oracle.fwd_rows(rows, 1, H, xv, wb, case["eps"], want_y=False, want_h=False)
    rin = r64.astype(np.float32)
    t0 = time.perf_counter()
    oracle.bwd_rows(rows, 1, H, dyv, xv, rin, wb)
    oracle.dw_cols(rows, 1, H, dyv, xv, rin)
    return time.perf_counter() - t0


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return None


def oracle_baseline(case, T, H, budget_s=10.0):
    """The oracle on a bounded sample (the leading rows) sized to ~budget_s."""
    probe = min(T, 1024)
    dt = oracle_sample(case, H, probe)
    rows = int(min(T, max(probe, probe * budget_s / max(dt, 1e-6))))
    dt = oracle_sample(case, H, rows)
    b = workload_bytes(rows, H, case["w"].numel() * case["w"].element_size(), 0)["rows_only"]
    return {
        "value": round(b / dt / 1e9, 4),
        "unit": "GB/s",
        "cores": 1,
        "kind": "oracle",
        "sample": f"FP64 C oracle backward (dx and dw) on the first {rows} of {T} rows of the workload, "
                  f"{dt:.2f} s, single thread",
        "cpu": cpu_model(),
        "host_cores": os.cpu_count(),
    }


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import cake_inputs
    import oracle
    oracle.build()
    spec = cake_inputs.WORKLOADS[args.workload]
    T, H = spec["T"], spec["H"]
    case = cake_inputs.make(args.workload, seed=0, device="cpu")
    K, Wm = args.steps, max(3, args.warmup)
    # size each step so the whole run stays within about two minutes
    probe = min(T, 512)
    dt = oracle_sample(case, H, probe)
    per_step_s = min(10.0, 120.0 / (K + Wm))
    rows = int(min(T, max(64, probe * per_step_s / max(dt, 1e-6))))
    for _ in range(Wm):
        oracle_sample(case, H, rows)
    times = [oracle_sample(case, H, rows) for _ in range(K)]
    b = workload_bytes(rows, H, case["w"].numel() * case["w"].element_size(), 0)["rows_only"]
    value = K * b / sum(times) / 1e9
    sample = f"FP64 C oracle backward (dx and dw) on the first {rows} of {T} rows per step, single thread"
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": Wm,
        "ms_per_step": round(statistics.mean(times) * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "T": T, "H": H, "rows_per_step": rows},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample,
                         "cpu": cpu_model(), "host_cores": os.cpu_count()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.profile:
        run_profile(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
