#!/usr/bin/env python
"""dw accuracy sweep of the backward (run on a GPU machine; not a pytest module).

For every (H, T, input family, seed) it draws the inputs, computes rstd with
the FP64 oracle (rounded to FP32, the rstd both sides use), runs the backward
in every dw accumulation form and mode, and compares dw with the oracle's
exact-order FP64 column sums.  The score of an element is
|dw - dw64| / (1e-4 + 1e-4 |dw64|); the sweep reports the worst element over
all columns and seeds, per form.  It also scores torch's FP32 eager column
sum of dy*x*rstd -- the comparator the pages hold the kernels against.

The budget and the protocol (60 inputs of each of three families, worst
element, both weight dtypes) follow the PR #8208 page, description; dw does
not depend on the weight, so one weight dtype stands for both.

  python tests/accuracy_sweep.py [--seeds 60] [--H 4096,5120]
         [--T 4096,44032,65536,131072] [--jobs 16] [--out sweep.jsonl]
"""
from __future__ import annotations

import argparse
import json
import os
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import cake_inputs  # noqa: E402
import oracle  # noqa: E402
from tests import tolerances as tol  # noqa: E402

FORMS = [  # (name, force_single, force_accum, deterministic)
    ("pair_plain", 0, 0, True), ("pair_blocked", 0, 1, True), ("pair_kahan", 0, 3, True),
    ("pair_twosum", 0, 2, True), ("single_kahan", 1, 3, False), ("single_twosum", 1, 2, False),
    ("grid_kahan", 3, 3, True),
    ("default_det", None, None, True), ("default_nondet", None, None, False),
]


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def run_case(cake, gpu_lock, H, T, family, seed, dev):
    g = torch.Generator(device=dev)
    g.manual_seed(1000003 * seed + 7919 * T + H)
    with gpu_lock:
        x = cake_inputs.rows_input(T, H, family, g, device=dev)
        dy = cake_inputs.normal_bf16((T, H), g, device=dev)
        xh, dyh = bits(x.cpu()), bits(dy.cpu())
    xv, dyv = oracle.View.contiguous(xh), oracle.View.contiguous(dyh)
    w = np.ones(H, dtype=np.float32)  # dw does not depend on w
    _, r64, _ = oracle.fwd_rows(T, 1, H, xv, w, cake_inputs.EPS, want_y=False, want_h=False)
    rin = r64.astype(np.float32)
    results = {}
    with gpu_lock:
        r_d = torch.from_numpy(rin).to(dev)
        w_d = torch.ones(H, dtype=torch.float32, device=dev)
        ws = cake.cake_rmsnorm_bwd_workspace(x, torch.float32, deterministic=False)
        dx = torch.empty_like(x)
        for name, single, accum, det in FORMS:
            dw = torch.empty(H, dtype=torch.float32, device=dev)
            if single is None:
                cake.cake_rmsnorm_bwd(dy, x, r_d, w_d, deterministic=det, workspace=ws, dx=dx, dw=dw)
            else:
                cake.cake_rmsnorm_bwd_forced(dy, x, r_d, w_d, deterministic=det, force_single=single,
                                             force_accum=accum, workspace=ws, dx=dx, dw=dw)
            results[name] = dw
        eager = (dy.float() * x.float() * r_d[:, None]).sum(0)
        torch.cuda.synchronize()
        results = {k: v.cpu().numpy() for k, v in results.items()}
        results["torch_fp32_eager"] = eager.cpu().numpy()
        del x, dy, ws, dx
    dw64 = oracle.dw_cols(T, 1, H, dyv, xv, rin)
    return {k: float(tol.dw_budget_fraction(v, dw64).max()) for k, v in results.items()}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--seeds", type=int, default=cake_inputs.SWEEP_SEEDS)
    ap.add_argument("--H", default=",".join(map(str, cake_inputs.SWEEP_H)))
    ap.add_argument("--T", default=",".join(map(str, cake_inputs.SWEEP_T)))
    ap.add_argument("--families", default=",".join(cake_inputs.SWEEP_FAMILIES))
    ap.add_argument("--jobs", type=int, default=min(16, os.cpu_count() or 1))
    ap.add_argument("--out", default=None)
    args = ap.parse_args()

    import __graft_entry__
    __graft_entry__.build()
    import bwd_dw_column_gb300 as cake

    dev = torch.device("cuda:0")
    lock = threading.Lock()
    Hs = [int(v) for v in args.H.split(",")]
    Ts = [int(v) for v in args.T.split(",")]
    fams = args.families.split(",")
    cases = [(H, T, f, s) for H in Hs for T in Ts for f in fams for s in range(args.seeds)]
    worst = {}
    out = open(args.out, "w") if args.out else None
    t0 = time.time()
    with ThreadPoolExecutor(args.jobs) as ex:
        futs = {ex.submit(run_case, cake, lock, H, T, f, s, dev): (H, T, f, s) for H, T, f, s in cases}
        for fut in futs:
            H, T, f, s = futs[fut]
            res = fut.result()
            key = (H, T, f)
            cur = worst.setdefault(key, {})
            for k, v in res.items():
                cur[k] = max(cur.get(k, 0.0), v)
            if out:
                out.write(json.dumps({"H": H, "T": T, "family": f, "seed": s, **res}) + "\n")
    if out:
        out.close()
    assert cake.cake_rmsnorm_device_status() == 0
    names = [n for n, *_ in FORMS] + ["torch_fp32_eager"]
    print(f"# worst dw element / budget over {args.seeds} seeds; {len(cases)} cases in {time.time() - t0:.0f} s, "
          f"{args.jobs} host threads")
    print("H T family " + " ".join(names))
    for (H, T, f), cur in sorted(worst.items()):
        print(f"{H} {T} {f} " + " ".join(f"{cur[n]:.4f}" for n in names))
    summary = {n: max(c[n] for c in worst.values()) for n in names}
    print(json.dumps({"accuracy_sweep": {"seeds": args.seeds, "H": Hs, "T": Ts, "families": fams,
                                         "worst_fraction_of_budget": summary}}))


if __name__ == "__main__":
    main()
