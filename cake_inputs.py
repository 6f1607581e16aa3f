"""Seeded synthetic inputs for the training RMSNorm workloads.

This module holds no RMSNorm arithmetic: it only draws the seeded random
tensors that both the oracle checks and the CUDA path consume, so that the
two sides see the same bits.  Values are drawn in FP32 with a seeded torch
generator (on the CPU or on the device named by ``device``) and rounded to
BF16 once; FP32 weights stay FP32.

Workloads (eps = 1e-6 everywhere):

* ``plain``    -- [T, H] rows, x and dy ~ N(0, 1), w = 1 + 0.1 N(0, 1);
* ``outlier``  -- like ``plain`` but ceil(1 % of T) rows, picked by a seeded
  permutation, are scaled by 30 before rounding;
* ``offset``   -- x = 3 + N(0, 1) on every row (the mean-offset family);
* ``res``      -- adds a residual ~ N(0, 0.5) (0.5 read as the standard
  deviation, torch's ``normal(mean, std)`` convention);
* per-head     -- [T, 24, 256] strided view of a [T, 24, 512] buffer
  (strides 12288, 512, 1) and a contiguous [T, 4, 256] tensor, one shared
  w[256].

Shapes and strides follow the PR #8208 page (description: per-head views and
their strides) and the "Speedups ... GB300 windows" commit quoted there
("Key": the `res` route, `w32` FP32 weight).
"""
from __future__ import annotations

import math

import torch

EPS = 1e-6


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, gen: torch.Generator, mean: float = 0.0, std: float = 1.0,
                device="cpu", chunk_rows: int = 8192) -> torch.Tensor:
    """BF16 tensor of N(mean, std) values drawn in FP32, rounded once.

    Drawn in row chunks of the leading dimension so that no FP32 copy of a
    multi-GB tensor is ever held.
    """
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    n0 = shape[0]
    for a in range(0, n0, chunk_rows):
        b = min(n0, a + chunk_rows)
        t = torch.randn((b - a,) + tuple(shape[1:]), generator=gen, dtype=torch.float32, device=device)
        if std != 1.0:
            t.mul_(std)
        if mean != 0.0:
            t.add_(mean)
        out[a:b] = t.to(torch.bfloat16)
    return out


def weight(H: int, gen: torch.Generator, dtype: torch.dtype, device="cpu") -> torch.Tensor:
    """w = 1 + 0.1 N(0, 1), drawn in FP32, then cast to ``dtype`` (BF16 or FP32)."""
    w = 1.0 + 0.1 * torch.randn(H, generator=gen, dtype=torch.float32, device=device)
    return w.to(dtype)


def rows_input(T: int, H: int, family: str, gen: torch.Generator, device="cpu") -> torch.Tensor:
    """x [T, H] BF16 for one input family: 'gauss', 'outlier', 'offset' or
    'rowmean' (each row r drawn around its own mean m_r = 3 + N(0, 1):
    x_rj = m_r + N(0, 1), the per-row random-mean reading of the mean-offset
    family)."""
    if family == "gauss":
        return normal_bf16((T, H), gen, device=device)
    if family == "offset":
        return normal_bf16((T, H), gen, mean=3.0, device=device)
    if family == "rowmean":
        means = 3.0 + torch.randn(T, generator=gen, dtype=torch.float32, device=device)
        out = torch.empty((T, H), dtype=torch.bfloat16, device=device)
        for a in range(0, T, 8192):
            b = min(T, a + 8192)
            t = torch.randn((b - a, H), generator=gen, dtype=torch.float32, device=device)
            t.add_(means[a:b, None])
            out[a:b] = t.to(torch.bfloat16)
        return out
    if family == "outlier":
        n_out = math.ceil(0.01 * T) if T > 0 else 0
        picks = torch.randperm(T, generator=gen, device=device)[:n_out] if T > 0 else None
        out = torch.empty((T, H), dtype=torch.bfloat16, device=device)
        scale = torch.ones(T, dtype=torch.float32, device=device)
        if n_out:
            scale[picks] = 30.0
        for a in range(0, T, 8192):
            b = min(T, a + 8192)
            t = torch.randn((b - a, H), generator=gen, dtype=torch.float32, device=device)
            t.mul_(scale[a:b, None])
            out[a:b] = t.to(torch.bfloat16)
        return out
    raise ValueError(f"unknown input family {family!r}")


def plain_case(T: int, H: int, *, family: str = "gauss", w_dtype=torch.bfloat16,
               dy_std: float = 1.0, seed: int = 0, device="cpu") -> dict:
    """x, dy [T, H] BF16 and w [H] for a plain-rows workload."""
    g = _gen(seed, device)
    x = rows_input(T, H, family, g, device)
    dy = normal_bf16((T, H), g, std=dy_std, device=device)
    w = weight(H, g, w_dtype, device)
    return {"x": x, "dy": dy, "w": w, "eps": EPS}


def residual_case(T: int, H: int, *, w_dtype=torch.bfloat16, seed: int = 0, device="cpu",
                  with_dh: bool = True) -> dict:
    """x, residual, dy (and dh, the gradient reaching h_new) [T, H] BF16, w [H]."""
    g = _gen(seed, device)
    x = normal_bf16((T, H), g, device=device)
    res = normal_bf16((T, H), g, std=0.5, device=device)
    dy = normal_bf16((T, H), g, device=device)
    dh = normal_bf16((T, H), g, device=device) if with_dh else None
    w = weight(H, g, w_dtype, device)
    return {"x": x, "residual": res, "dy": dy, "dh": dh, "w": w, "eps": EPS}


def heads_case(T: int, heads: int, *, strided: bool, w_dtype=torch.float32, seed: int = 0,
               device="cpu", head_dim: int = 256) -> dict:
    """Per-head workload.

    strided=True: x is the [T, heads, 256] slice [..., :256] of a
    [T, heads, 512] buffer (strides heads*512, 512, 1); strided=False: x is a
    contiguous [T, heads, 256] tensor.  x = 3 + N(0, 1), dy ~ N(0, 1)
    contiguous [T, heads, 256], one shared w[256].
    """
    g = _gen(seed, device)
    if strided:
        buf = normal_bf16((T, heads, 2 * head_dim), g, mean=3.0, device=device)
        x = buf[:, :, :head_dim]
    else:
        buf = None
        x = normal_bf16((T, heads, head_dim), g, mean=3.0, device=device)
    dy = normal_bf16((T, heads, head_dim), g, device=device)
    w = weight(head_dim, g, w_dtype, device)
    return {"x": x, "x_buffer": buf, "dy": dy, "w": w, "eps": EPS}


# The five workloads of the benchmark and the parity tests, by name.
WORKLOADS = {
    # T=256, H=1536, plain rows, BF16 weight; fwd + both backward modes.
    "h1536_t256": dict(kind="plain", T=256, H=1536, family="gauss", w_dtype=torch.bfloat16, dy_std=1.0),
    # T=65536, H=2048, outlier family, dy ~ N(0, 1e-2), FP32 weight; both backward modes.
    "h2048_t65536_outlier_w32": dict(kind="plain", T=65536, H=2048, family="outlier",
                                     w_dtype=torch.float32, dy_std=1e-2),
    # T=131072, H=6144, fused residual add, BF16 weight; fwd + non-deterministic backward.
    "h6144_t131072_res": dict(kind="res", T=131072, H=6144, w_dtype=torch.bfloat16),
    # T=32768 per-head views, FP32 shared w[256].
    "heads24_t32768_strided": dict(kind="heads", T=32768, heads=24, strided=True, w_dtype=torch.float32),
    "heads4_t32768": dict(kind="heads", T=32768, heads=4, strided=False, w_dtype=torch.float32),
    # The accuracy sweep's widths at its T = 65536 point (x, dy ~ N(0, 1), BF16 weight), for timing.
    "h4096_t65536_sweep": dict(kind="plain", T=65536, H=4096, family="gauss", w_dtype=torch.bfloat16, dy_std=1.0),
    "h5120_t65536_sweep": dict(kind="plain", T=65536, H=5120, family="gauss", w_dtype=torch.bfloat16, dy_std=1.0),
}

# Accuracy sweep: H x T x weight dtype x input family, 60 seeds per family.
SWEEP_H = (4096, 5120)
SWEEP_T = (4096, 44032, 65536, 131072)
SWEEP_FAMILIES = ("gauss", "outlier", "offset")
SWEEP_SEEDS = 60

# The sweep's shapes as benchmark workloads (gaussian family, seed 0): a BF16
# weight at every point, and an FP32 weight at T = 65536.
for _H in SWEEP_H:
    for _T in SWEEP_T:
        WORKLOADS.setdefault(f"h{_H}_t{_T}_sweep", dict(kind="plain", T=_T, H=_H, family="gauss",
                                                         w_dtype=torch.bfloat16, dy_std=1.0))
    WORKLOADS[f"h{_H}_t65536_sweep_w32"] = dict(kind="plain", T=65536, H=_H, family="gauss",
                                                w_dtype=torch.float32, dy_std=1.0)


# Shapes the pages do not name, for profiling layouts the named workloads do
# not reach: narrow rows (per-head widths 64 and 128 as plain rows), which run
# several to a warp.
EXTRA_WORKLOADS = {
    "h64_t524288": dict(kind="plain", T=524288, H=64, family="gauss", w_dtype=torch.bfloat16, dy_std=1.0),
    "h128_t262144": dict(kind="plain", T=262144, H=128, family="gauss", w_dtype=torch.bfloat16, dy_std=1.0),
}


def workload_spec(name: str) -> dict:
    """The spec of a named workload: one of ``WORKLOADS``, else ``EXTRA_WORKLOADS``."""
    return WORKLOADS[name] if name in WORKLOADS else EXTRA_WORKLOADS[name]


def make(name: str, seed: int = 0, device="cpu", **overrides) -> dict:
    """Build one named workload (``workload_spec``), optionally with overridden sizes."""
    spec = dict(workload_spec(name))
    spec.update(overrides)
    kind = spec.pop("kind")
    if kind == "plain":
        return plain_case(spec["T"], spec["H"], family=spec["family"], w_dtype=spec["w_dtype"],
                          dy_std=spec["dy_std"], seed=seed, device=device)
    if kind == "res":
        return residual_case(spec["T"], spec["H"], w_dtype=spec["w_dtype"], seed=seed, device=device,
                             with_dh=spec.get("with_dh", True))
    if kind == "heads":
        return heads_case(spec["T"], spec["heads"], strided=spec["strided"], w_dtype=spec["w_dtype"],
                          seed=seed, device=device)
    raise ValueError(kind)
