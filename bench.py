#!/usr/bin/env python
"""Benchmark of the training RMSNorm on one GB300 (per rank).

Headline workload (the largest configuration that fits one GPU): T = 131072
tokens, H = 6144, fused residual add -- x BF16 ~ N(0, 1), residual BF16 ~
N(0, std 0.5), dy (and dh, the gradient reaching h_new) BF16 ~ N(0, 1), w BF16
= 1 + 0.1 N(0, 1), eps = 1e-6.  One step is one non-deterministic backward
(what the window table runs for deterministic=False) through the C ABI.  The
same run then times every other configuration the same way and lists them
under "configs": T = 256, H = 1536; T = 65536, H = 2048 (outlier family, FP32
weight); the per-head views [32768, 24, 256] (strided) and [32768, 4, 256];
and the accuracy sweep's shapes H in {4096, 5120} x T in {4096, 44032, 65536,
131072}.  One JSON line on rank 0.

  value         achieved GB/s = algorithmic bytes of the step / its device
                time (inputs resident in HBM, L2 flushed before every step)
  e2e           the same metric through the C ABI entry point that takes host
                buffers: every step copies its inputs from page-locked host
                memory and dx and dw back, in row chunks whose copies and
                kernels overlap, all inside the timed region
  roofline      the main kernel alone, timed with CUDA events on its stream,
                against the measured HBM copy bandwidth
  cpu_baseline  the FP64 CPU oracle on a bounded sample of the same workload
  configs       per configuration: deterministic and non-deterministic
                backward, the main kernel alone (and the forward where the
                configuration asks for it), each in us, GB/s and as a fraction
                of the copy peak

``--workload NAME`` times one workload only.  ``--impl reference`` times the
oracle instead (host cores, a bounded sample per step) and prints the
reference line.  ``--profile`` runs a minimal launch sequence for ncu, and
``--record-traffic`` turns an ncu CSV of that sequence into the DRAM-traffic
record under profiles/.  Under torchrun each rank runs an independent replica
(the path has no cross-GPU exchange on one box); value sums the ranks' bytes
over the slowest rank's time.
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
HEADLINE = "h6144_t131072_res"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20
ACCUM = {"plain": 0, "blocked": 1, "twosum": 2, "kahan": 3}

# The configurations timed after the headline, with the operations each asks
# for: T = 256 H = 1536 (forward and both backward modes); T = 65536 H = 2048
# outlier family with an FP32 weight; the per-head views; the accuracy
# sweep's widths at each of its T (BF16 weight, and FP32 at T = 65536).
CONFIGS = (
    [("h1536_t256", ("fwd", "det", "nondet", "main")),
     ("h2048_t65536_outlier_w32", ("det", "nondet", "main")),
     ("heads24_t32768_strided", ("det", "nondet", "main")),
     ("heads4_t32768", ("det", "nondet", "main"))]
    + [(f"h{H}_t{T}_sweep", ("det", "nondet", "main")) for H in (4096, 5120) for T in (4096, 44032, 65536, 131072)]
    + [(f"h{H}_t65536_sweep_w32", ("det", "nondet", "main")) for H in (4096, 5120)]
)

# The pages' own GB300 latencies for exactly these shapes and weight dtypes
# (the "Speedups ... GB300 windows" commit quoted on the PR #8208 page, "GB300
# table": median CUPTI span of a CUDA-graph replay with L2 flushed) -- context
# only, measured under another protocol on another software stack.
PAGES_GB300_US = {
    "h1536_t256": {"fwd": 1.98, "det": 5.76, "nondet": 5.86},
    "h4096_t4096_sweep": {"det": 23.55, "nondet": 23.65},
    "h4096_t65536_sweep": {"det": 249.76, "nondet": 257.86},
    "h5120_t4096_sweep": {"det": 26.85, "nondet": 26.85},
    "h5120_t65536_sweep": {"det": 314.30, "nondet": 363.10},
    "h5120_t65536_sweep_w32": {"det": 313.94, "nondet": 369.71},
}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None, help="time this workload only (default: the headline + configs)")
    ap.add_argument("--no-configs", action="store_true", help="time the headline workload only")
    ap.add_argument("--tokens", type=int, default=None,
                    help="with --profile: the workload's shape at this many tokens (a smaller case for ncu)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-chunks", type=int, default=16,
                    help="row chunks of the end-to-end step (copies and kernels overlap across chunks)")
    ap.add_argument("--profile", choices=["det", "nondet", "fwd", "main", "single_atomic", "single_grid",
                                          "single_cluster", "all"], default=None,
                    help="run only the named loop(s) with few launches (for ncu); prints per-call times")
    ap.add_argument("--accum", choices=sorted(ACCUM), default=None,
                    help="with --profile: force the per-thread dw accumulation form")
    ap.add_argument("--graph", action="store_true",
                    help="with --profile: time CUDA-graph replays of one call (no host launch cost)")
    ap.add_argument("--source-hash", action="store_true", help="print the kernel sources' hash and exit")
    ap.add_argument("--record-traffic", metavar="CSV", default=None,
                    help="record the DRAM bytes per launch of --kernel in an ncu CSV (taken on the sources "
                         "whose hash --hash gives) into profiles/traffic.json for --workload")
    ap.add_argument("--kernel", default="bwd_rows_kernel")
    ap.add_argument("--hash", default=None)
    ap.add_argument("--summary", default=None, help="with --record-traffic: the profiles/ summary it backs")
    ap.add_argument("--command", default=None, help="with --record-traffic: the ncu command that made the CSV")
    ap.add_argument("--scale", type=float, default=1.0,
                    help="with --record-traffic: units of the full workload per captured unit")
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


# Host-only source: argument validation, the window table and launch dispatch.
# It decides the launch plan, which a traffic record stores and compares
# itself; every other file under csrc/ is device code or shared by it.
HOST_ONLY_SOURCES = ("cake_api.cu",)


def canonical_source(text: str) -> str:
    """C/C++/CUDA source without its comments, blank lines and the spaces
    around each line: what the compiler turns into code.  An edit to a
    comment or to indentation leaves it as it is; any other edit changes it.
    String and character literals are kept whole (a // inside one is code)."""
    out = []
    i, n = 0, len(text)
    while i < n:
        c = text[i]
        if c == "/" and i + 1 < n and text[i + 1] == "/":
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif c == "/" and i + 1 < n and text[i + 1] == "*":
            j = text.find("*/", i + 2)
            end = n if j < 0 else j + 2
            out.append("\n" * text.count("\n", i, end) or " ")
            i = end
        elif c in "\"'":
            j = i + 1
            while j < n and text[j] != c and text[j] != "\n":
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    lines = (ln.strip() for ln in "".join(out).split("\n"))
    return "\n".join(ln for ln in lines if ln)


def kernel_source_hash():
    """Hash of the kernel sources (every csrc file but the host-only ones),
    taken over their canonical form, so that comments do not count."""
    csrc = os.path.join(ROOT, "bwd_dw_column_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(csrc)):
        if f in HOST_ONLY_SOURCES:
            continue
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode() + canonical_source(fh.read()).encode())
    return h.hexdigest()[:16]


def workload_plan(workload: str):
    """The backward plan (the window table's variant) of a workload's main
    kernel, as the library picks it now; None without the library."""
    try:
        import bwd_dw_column_gb300 as cake
        import cake_inputs
        spec = cake_inputs.workload_spec(workload)
        shape = (spec["T"], spec.get("heads", 1), spec.get("H", 256))
        return cake.cake_rmsnorm_bwd_select(shape, spec["w_dtype"], deterministic=True,
                                            has_dh=spec["kind"] == "res")
    except Exception:
        return None


def traffic_json():
    return os.path.join(ROOT, "profiles", "traffic.json")


def traffic_record(kernel: str, workload: str):
    """The committed ncu record (DRAM bytes per launch, the summary file) when
    its counters were taken on the current kernel sources and with the launch
    plan the table picks now; else None."""
    try:
        with open(traffic_json()) as f:
            rec = json.load(f)
    except Exception:
        return None
    ent = rec.get(f"{kernel}:{workload}")
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    if "plan" in ent and ent["plan"] != workload_plan(workload):
        return None
    return ent


def recorded_traffic(kernel: str, workload: str):
    ent = traffic_record(kernel, workload)
    return ent.get("dram_bytes_per_launch") if ent else None


_UNITS = {"byte": 1, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9, "tbyte": 1e12,
          "nsecond": 1e-9, "usecond": 1e-6, "msecond": 1e-3, "second": 1.0,
          "ns": 1e-9, "us": 1e-6, "ms": 1e-3, "s": 1.0}


def parse_ncu_csv(path: str, kernel: str):
    """Per-launch metric values (base units) of the launches of `kernel` in an
    ncu --csv --metrics log."""
    import csv

    launches = {}
    with open(path, newline="") as f:
        lines = [ln for ln in f if ln.startswith('"')]
    for row in csv.DictReader(lines):
        name = row.get("Kernel Name", "")
        if kernel not in name:
            continue
        unit = (row.get("Metric Unit") or "").strip().lower()
        try:
            val = float(row["Metric Value"].replace(",", ""))
        except (KeyError, ValueError):
            continue
        launches.setdefault(row["ID"], {})[row["Metric Name"]] = val * _UNITS.get(unit, 1.0)
    return [launches[k] for k in sorted(launches, key=int)]


def record_traffic(args):
    """Write profiles/traffic.json's entry for (kernel, workload) from an ncu
    CSV.  The entry carries the hash of the sources the counters were taken on
    (the hash the box printed before the capture), and is refused unless that
    is the hash of the sources here: counters are never carried over to code
    they were not taken on."""
    if not args.workload:
        raise SystemExit("--record-traffic needs --workload")
    here = kernel_source_hash()
    if args.hash != here:
        raise SystemExit(f"counters taken on sources {args.hash}, but the sources here hash to {here}")
    ls = parse_ncu_csv(args.record_traffic, args.kernel)
    if not ls:
        raise SystemExit(f"no launch of {args.kernel} in {args.record_traffic}")
    per = [d["dram__bytes_read.sum"] + d["dram__bytes_write.sum"] for d in ls]
    dur = [d.get("gpu__time_duration.sum") for d in ls if d.get("gpu__time_duration.sum")]
    try:
        with open(traffic_json()) as f:
            rec = json.load(f)
    except Exception:
        rec = {}
    rec[f"{args.kernel}:{args.workload}"] = {
        "source_hash": here,
        "plan": workload_plan(args.workload),
        "dram_bytes_per_launch": int(round(statistics.mean(per) * args.scale)),
        "launches": len(per),
        "ncu_us_per_launch": round(statistics.mean(dur) * 1e6 * args.scale, 2) if dur else None,
        "scaled_from_capture": args.scale if args.scale != 1.0 else None,
        "command": args.command,
        "summary": args.summary,
    }
    with open(traffic_json(), "w") as f:
        json.dump(rec, f, indent=1, sort_keys=True)
        f.write("\n")
    print(json.dumps(rec[f"{args.kernel}:{args.workload}"]))


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


class Workload:
    """One workload's device tensors, preallocated outputs and step callables.

    Each step callable comes with the number of library kernels it launches
    and its algorithmic bytes."""

    def __init__(self, cake, torch, name, dev, seed=0, accum=None, tokens=None):
        import cake_inputs

        self.name, self.spec = name, dict(cake_inputs.workload_spec(name))
        if tokens:
            self.spec["T"] = tokens
        case = cake_inputs.make(name, seed=seed, device=dev, **({"T": tokens} if tokens else {}))
        self.case = case
        x, dy, w, eps = case["x"], case["dy"], case["w"], case["eps"]
        res, dh = case.get("residual"), case.get("dh")
        out = cake.cake_rmsnorm_fwd(x, w, eps, residual=res)
        y, rstd = out[0], out[1]
        hn = out[2] if res is not None else None
        h = hn if res is not None else x
        ws = cake.cake_rmsnorm_bwd_workspace(h, w.dtype, deterministic=False)
        dx = torch.empty(h.shape, dtype=torch.bfloat16, device=dev)
        dw = torch.empty(h.shape[-1], dtype=torch.float32, device=dev)
        self.x, self.dy, self.w, self.res, self.dh, self.h, self.rstd = x, dy, w, res, dh, h, rstd
        self.ws, self.dx, self.dw, self.y, self.hn = ws, dx, dw, y, hn
        self.T = x.shape[0]
        self.nh = x.shape[1] if x.dim() == 3 else 1
        self.H = x.shape[-1]
        self.R = self.T * self.nh
        wb = w.numel() * w.element_size()

        def variant(det, has_dh, force_single=None):
            return cake.cake_rmsnorm_bwd_select((self.T, self.nh, self.H), w.dtype, deterministic=det,
                                                has_dh=has_dh, force_single=force_single,
                                                force_accum=None if accum is None else ACCUM[accum])

        def bwd(det, ddh):
            acc = None if accum is None else ACCUM[accum]
            if acc is None:
                return lambda: cake.cake_rmsnorm_bwd(dy, h, rstd, w, ddh, deterministic=det, workspace=ws, dx=dx,
                                                     dw=dw)
            return lambda: cake.cake_rmsnorm_bwd_forced(dy, h, rstd, w, ddh, deterministic=det, force_single=0,
                                                       force_accum=acc, workspace=ws, dx=dx, dw=dw)

        def forced(form, ddh):
            return lambda: cake.cake_rmsnorm_bwd_forced(dy, h, rstd, w, ddh, deterministic=form != 1,
                                                       force_single=form, workspace=ws, dx=dx, dw=dw)

        def fwd():
            return cake.cake_rmsnorm_fwd(x, w, eps, residual=res, y=y, rstd=rstd, h_new=hn)

        self.steps = {}
        for suffix, ddh in (("", dh), ("_nodh", None)):
            if suffix and dh is None:
                continue
            vd, vn = variant(True, ddh is not None), variant(False, ddh is not None)
            nb = workload_bytes(self.R, self.H, wb, vd["ctas"], dh=ddh is not None)
            nd_pair = vn["single"] == 0
            self.steps["det" + suffix] = (bwd(True, ddh), 2, nb["pair"], vd)
            self.steps["nondet" + suffix] = (bwd(False, ddh), 2 if nd_pair else 1,
                                             nb["pair"] if nd_pair else nb["single"], vn)
            self.steps["main" + suffix] = (
                (lambda ddh=ddh: cake.cake_rmsnorm_bwd_main(dy, h, rstd, w, ddh, workspace=ws, dx=dx, dw=dw,
                                                            force_accum=None if accum is None else ACCUM[accum])),
                1, nb["main"], vd)
            if not suffix:
                va = variant(False, ddh is not None, 1)
                vg = variant(True, ddh is not None, 3)
                vc = variant(True, ddh is not None, 4)
                self.steps["single_atomic"] = (forced(1, ddh), 1, nb["single"], va)
                self.steps["single_cluster"] = (forced(4, ddh), 1, nb["rows_only"], vc)
                self.steps["single_grid"] = (forced(3, ddh), 1,
                                             workload_bytes(self.R, self.H, wb, vg["ctas"], dh=ddh is not None)["pair"],
                                             vg)
                fb = workload_bytes(self.R, self.H, wb, 0, res=res is not None)["fwd"]
                self.steps["fwd"] = (fwd, 1, fb, None)
                # the checkpointed step of the pages' GB300 tables: forward,
                # forward recompute, deterministic backward
                self.steps["ckpt_2xfwd_bwd"] = (lambda: (fwd(), fwd(), bwd(True, ddh)()), 4, 2 * fb + nb["pair"], vd)


def time_modes(torch, wl: Workload, modes, K, Wm, flush, stream, world, dev, peak):
    """Time the listed step kinds of one workload; per mode us, GB/s and the
    fraction of the copy peak (GB/s per GPU), plus the launch count."""
    out, launches = {}, 0
    for m in modes:
        fn, nl, nbytes, _ = wl.steps[m]
        times = time_loop(torch, fn, K, Wm, flush, stream)
        tot, mean = aggregate_times(times, world, dev)
        gbs = replica_gbs(nbytes, K, world, tot)
        out[m] = {"us": round(mean * 1e3, 2), "GB/s": round(gbs, 1), "frac": round(gbs / world / peak, 4),
                  "bytes": nbytes}
        launches += nl * K
    return out, launches


def short_variant(v):
    if not v:
        return None
    return {k: v[k] for k in ("single", "dw_accum", "vec_per_thread", "warps_per_row", "row_groups",
                              "rows_per_group", "stages", "ctas")}


def e2e_loop(cake, torch, wl: Workload, K, Wm, flush, stream, dev, det, chunks):
    """The backward through the public entry point that takes host buffers
    (cake_rmsnorm_bwd_host): every step copies the inputs from page-locked
    host memory to the device and dx and dw back, inside the call, in row
    chunks whose copies and kernels overlap.  A strided view travels as its
    dense rows (gathered on the host once, outside the timed region)."""
    pin = lambda t: None if t is None else t.contiguous().cpu().pin_memory()
    hx, hdy, hdh, hrstd, hw = (pin(t) for t in (wl.h, wl.dy, wl.dh, wl.rstd, wl.w))
    hdx = torch.empty(hx.shape, dtype=torch.bfloat16).pin_memory()
    hdw = torch.empty(wl.H, dtype=torch.float32).pin_memory()
    n = cake.cake_rmsnorm_bwd_host_staging_size((wl.T, wl.nh, wl.H), wl.w.dtype, has_dh=wl.dh is not None,
                                                chunks=chunks)
    staging = torch.empty(max(n, 256), dtype=torch.uint8, device=dev)

    def step():
        cake.cake_rmsnorm_bwd_host(hdy, hx, hrstd, hw, hdh, dx=hdx, dw=hdw, staging=staging, chunks=chunks,
                                   deterministic=det)

    times = time_loop(torch, step, K, Wm, flush, stream)
    h2d = sum(t.numel() * t.element_size() for t in (hx, hdy, hdh, hrstd, hw) if t is not None)
    d2h = hdx.numel() * 2 + hdw.numel() * 4
    return times, h2d, d2h


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

    head = args.workload or HEADLINE
    configs = [] if (args.no_configs or args.workload) else CONFIGS
    peak, peak_kind = measured_peak()
    flush = L2Flush(torch, dev)
    stream = torch.cuda.current_stream()
    K, Wm = args.steps, max(3, args.warmup)

    wl = Workload(cake, torch, head, dev, seed=rank)
    has_dh = wl.dh is not None
    head_modes = ["nondet", "det", "main", "fwd", "single_atomic", "single_grid", "ckpt_2xfwd_bwd"]
    if has_dh:
        head_modes += ["nondet_nodh", "det_nodh", "main_nodh"]

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    entries = []
    with ClockSampler(local) as clk:
        modes, launches = time_modes(torch, wl, head_modes, K, Wm, flush, stream, world, dev, peak)
        for name, ms in configs:
            cw = Workload(cake, torch, name, dev, seed=rank)
            cm, cl = time_modes(torch, cw, ms, K, Wm, flush, stream, world, dev, peak)
            launches += cl
            ent = {"workload": name, "T": cw.T, "heads": cw.nh, "H": cw.H,
                   "w_dtype": "fp32" if cw.w.dtype == torch.float32 else "bf16", "inputs": describe(cw.spec),
                   "modes": cm, "variant": short_variant(cw.steps["det"][3]),
                   "main_kernel_frac": cm["main"]["frac"],
                   "traffic": recorded_traffic("bwd_rows_kernel", name),
                   "traffic_summary": (traffic_record("bwd_rows_kernel", name) or {}).get("summary")}
            if cw.R >= 32768 and cw.T >= 32768:
                ent["at_least_75pct_both_modes"] = bool(cm["det"]["frac"] >= 0.75 and cm["nondet"]["frac"] >= 0.75)
            if name in PAGES_GB300_US:
                ent["pages_gb300_us"] = PAGES_GB300_US[name]
            entries.append(ent)
            del cw
            torch.cuda.empty_cache()
    torch.cuda.synchronize()
    clocks = clk.summary()

    t_e2e, h2d, d2h = e2e_loop(cake, torch, wl, K, Wm, flush, stream, dev, det=False, chunks=args.e2e_chunks)
    e2e_chunks = min(args.e2e_chunks, wl.R)
    launches += (e2e_chunks + 1) * K
    assert cake.cake_rmsnorm_device_status() == 0
    tot_e2e, mean_e2e = aggregate_times(t_e2e, world, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and wl.spec["kind"] in ("plain", "res"):
        cpu = oracle_baseline(wl.case, wl.T, wl.H, budget_s=10.0)
    if world > 1:
        dist.barrier()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    nd = modes["nondet"]
    main = modes["main"]
    nd_variant = wl.steps["nondet"][3]
    line = {
        "metric": METRIC,
        "value": nd["GB/s"],
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": Wm,
        "ms_per_step": round(nd["us"] / 1e3, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "impl": "ours",
        "config": {
            "workload": head,
            "T": wl.T, "heads": wl.nh, "H": wl.H, "w_dtype": "fp32" if wl.w.dtype == torch.float32 else "bf16",
            "inputs": describe(wl.spec),
            "mode": "non-deterministic backward (the window table's choice for deterministic=False)"
                    + (", with the gradient dh reaching h_new" if has_dh else ""),
            "io_dtype": "bf16 activations, fp32 rstd/dw",
            "l2": "flushed before every timed step (256 MiB write, then 256 MiB read so no dirty line is left)",
            "parallelism": f"{world} independent replicas" if world > 1 else "single GPU",
            "variant": short_variant(nd_variant),
        },
        "bwd_us": nd["us"],
        "bytes_per_step": nd["bytes"],
        "frac_of_peak": nd["frac"],
        "modes": modes,
        "roofline": {
            "bound": "hbm",
            "kernel": "bwd_rows_kernel (main kernel of the backward pair)",
            "achieved": round(main["GB/s"] / world, 1),
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": main["frac"],
            "traffic": recorded_traffic("bwd_rows_kernel", head),
            "traffic_summary": (traffic_record("bwd_rows_kernel", head) or {}).get("summary"),
            "algorithmic_bytes": main["bytes"],
        },
        "e2e": {
            "value": round(replica_gbs(nd["bytes"], K, world, tot_e2e), 1),
            "unit": "GB/s",
            "ms_per_step": round(mean_e2e, 4),
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "entry_point": "cake_rmsnorm_bwd_host (page-locked host buffers in and out, "
                           f"{e2e_chunks} row chunks whose copies and kernels overlap)",
        },
        "gpu_launches": launches,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "configs": entries,
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

    dev = torch.device("cuda", 0)
    wl = Workload(cake, torch, args.workload or HEADLINE, dev, accum=args.accum, tokens=args.tokens)
    names = ["fwd", "det", "nondet"] if args.profile == "all" else [args.profile]
    out = {}
    stream = torch.cuda.current_stream()
    for n in names:
        fn = wl.steps[n][0]
        if args.graph:
            fn()  # first call on the device: attributes and addresses set up before capture
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                wl.steps[n][0]()
            fn = graph.replay
        ts = [t * 1e3 for t in time_loop(torch, fn, args.steps, args.warmup, None, stream)]
        out[n] = {"us_median": round(statistics.median(ts), 2), "us_min": round(min(ts), 2)}
    assert cake.cake_rmsnorm_device_status() == 0
    print(json.dumps({"profile": wl.name, "tokens": wl.T, "accum": args.accum, "us_per_call": out,
                      "source_hash": kernel_source_hash()}), flush=True)


# ------------------------------------------------------------ the oracle

def oracle_sample(case, H, rows):
    """Seconds the oracle's backward takes on the first `rows` rows (dx of
    those rows and dw over them), its inputs (rstd; h_new on the residual
    route) prepared outside the timing."""
    import numpy as np
    import torch

    import oracle

    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    x = case["x"][:rows].cpu()
    dy = case["dy"][:rows].cpu()
    w = case["w"].cpu()
    xv, dyv = oracle.View.contiguous(bits(x)), oracle.View.contiguous(bits(dy))
    wb = w.numpy() if w.dtype == torch.float32 else bits(w)
    res = case.get("residual")
    if res is not None:
        rv = oracle.View.contiguous(bits(res[:rows].cpu()))
        _, r64, hn = oracle.fwd_rows(rows, 1, H, xv, wb, case["eps"], residual=rv, want_y=False, want_h=True)
        hv = oracle.View.contiguous(hn)
    else:
        _, r64, _ = oracle.fwd_rows(rows, 1, H, xv, wb, case["eps"], want_y=False, want_h=False)
        hv = xv
    dh = case.get("dh")
    dhv = oracle.View.contiguous(bits(dh[:rows].cpu())) if dh is not None else None
    rin = r64.astype(np.float32)
    t0 = time.perf_counter()
    oracle.bwd_rows(rows, 1, H, dyv, hv, rin, wb, dh=dhv)
    oracle.dw_cols(rows, 1, H, dyv, hv, rin)
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
    probe = min(T, 256)
    dt = oracle_sample(case, H, probe)
    rows = int(min(T, max(probe, probe * budget_s / max(dt, 1e-6))))
    dt = oracle_sample(case, H, rows)
    b = workload_bytes(rows, H, case["w"].numel() * case["w"].element_size(), 0,
                       dh=case.get("dh") is not None)["rows_only"]
    return {
        "value": round(b / dt / 1e9, 4),
        "unit": "GB/s",
        "cores": 1,
        "kind": "oracle",
        "sample": f"FP64 C oracle backward (dx and dw{', with dh' if case.get('dh') is not None else ''}) on the "
                  f"first {rows} of {T} rows of the workload, {dt:.2f} s, single thread",
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
    name = args.workload or HEADLINE
    spec = cake_inputs.workload_spec(name)
    if spec["kind"] not in ("plain", "res"):
        raise SystemExit("the reference arm times plain and residual workloads")
    T, H = spec["T"], spec["H"]
    # only the sampled leading rows are ever read: draw a prefix of the
    # workload's rows (the same generator sequence as the full workload for
    # row-wise draws)
    K, Wm = args.steps, max(3, args.warmup)
    case = cake_inputs.make(name, seed=0, device="cpu", **({"T": min(T, 4096)} if spec["kind"] == "res" else {}))
    probe = min(T, 128)
    dt = oracle_sample(case, H, probe)
    per_step_s = min(10.0, 120.0 / (K + Wm))
    rows = int(min(case["x"].shape[0], max(16, probe * per_step_s / max(dt, 1e-6))))
    for _ in range(Wm):
        oracle_sample(case, H, rows)
    times = [oracle_sample(case, H, rows) for _ in range(K)]
    b = workload_bytes(rows, H, case["w"].numel() * case["w"].element_size(), 0,
                       dh=case.get("dh") is not None)["rows_only"]
    value = K * b / sum(times) / 1e9
    sample = (f"FP64 C oracle backward (dx and dw{', with dh' if case.get('dh') is not None else ''}) on "
              f"{rows} rows of the {T}-row workload per step, single thread")
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
        "config": {"workload": name, "T": T, "H": H, "rows_per_step": rows},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample,
                         "cpu": cpu_model(), "host_cores": os.cpu_count()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.source_hash:
        print(kernel_source_hash())
    elif args.record_traffic:
        record_traffic(args)
    elif args.profile:
        run_profile(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
