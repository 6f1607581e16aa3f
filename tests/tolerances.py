"""Parity tolerances.

dw: per element |dw_k - dw64| <= DW_ATOL + DW_RTOL * |dw64| against the FP64
exact-order sum at the kernel's FP32 rstd (PR #8208 page, description).
y, dx: within one BF16 ulp of the FP64 value rounded to BF16; rstd: relative
error <= 1e-6 against FP64.  A dx element also passes when its error is
inside the FP32 evaluation bound of the expression rs*(g - xhat*c) near
cancellation: 4 * 2^-24 * rs * (|g| + |xhat*c|) (see ``dx_excess``).
"""
import numpy as np

DW_ATOL = 1e-4
DW_RTOL = 1e-4
RSTD_REL = 1e-6


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of BF16 values at |v| (8 significant bits; subnormal floor 2^-133)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126.0)
    return np.where(a > 0, 2.0 ** (e - 7), 2.0 ** -133)


def dw_budget_fraction(dw_k: np.ndarray, dw64: np.ndarray) -> np.ndarray:
    return np.abs(dw_k.astype(np.float64) - dw64) / (DW_ATOL + DW_RTOL * np.abs(dw64))


def _ordered(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns mapped to integers that are consecutive along the reals."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def ulp_distance(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Number of BF16 steps between two BF16 values (0: equal, 1: neighbours)."""
    return np.abs(_ordered(a_bits) - _ordered(b_bits))


U32 = 2.0 ** -24


def dx_allowance(dy: np.ndarray, h: np.ndarray, w: np.ndarray, rstd: np.ndarray) -> np.ndarray:
    """FP32 evaluation bound of dx = (dy*w)*rs - h*kk, kk = ((c'*rs)*rs)*rs,
    for every element of [R, H] rows (the kernel's order of operations).

    g = dy*w is rounded once; kk carries the sum c' = (1/H) sum g*h (at most
    64*u*sum|g*h|/H: an FMA chain per thread, a 5-level butterfly, at most 24
    warp partials), the product by 1/H and the three products by rs, about 6u
    relative in all; then h*kk and the final FMA round once more each.
    """
    rs = rstd.astype(np.float64)[:, None]
    g = dy * w[None, :]
    xh = h * rs
    H = h.shape[1]
    c = (g * xh).sum(axis=1, keepdims=True) / H
    dc = 64 * U32 * np.abs(g * xh).sum(axis=1, keepdims=True) / H
    t = g - xh * c
    return rs * (2 * U32 * (np.abs(g) + np.abs(t)) + 8 * U32 * np.abs(xh * c) + np.abs(xh) * dc)


# A dx element sits on cancellation when |dx64| is below 2^-8 of the scale
# of the terms that produce it, rs*(|g| + |xhat*c|) (+ |dh|): there one BF16
# step of dx is smaller than FP32's rounding of those terms.
CANCELLATION = 2.0 ** -8


def dx_report(dx_bits: np.ndarray, dx64: np.ndarray, dy: np.ndarray, h: np.ndarray, w: np.ndarray,
              rstd: np.ndarray, bf16_round, bf16_to_f64, dh: np.ndarray | None = None) -> dict:
    """Counts of the kernel's BF16 dx against FP64.

    n: elements compared; max_ulp: largest distance in BF16 steps from
    RNE_bf16(dx64); strict: elements more than one step away (the literal
    1-ulp bar); bounded: strict elements also farther from dx64 than one BF16
    ulp plus the FP32 evaluation bound of the expression (cancellation can
    make the exact BF16 rounding of a tiny dx unreachable from FP32
    arithmetic); off_cancellation: strict elements that are not on
    cancellation (|dx64| >= 2^-8 of the terms' scale).  The parity bar is
    bounded == 0 and off_cancellation == 0.
    """
    ref = bf16_round(dx64)
    dist = ulp_distance(dx_bits, ref)
    out = {"n": int(dist.size), "max_ulp": int(dist.max(initial=0)), "strict": 0, "bounded": 0,
           "off_cancellation": 0}
    strict = dist > 1
    if not strict.any():
        return out
    err = np.abs(bf16_to_f64(dx_bits) - dx64)
    allow = bf16_ulp(dx64) + dx_allowance(dy, h, w, rstd)
    rs = rstd.astype(np.float64)[:, None]
    g = dy * w[None, :]
    xh = h * rs
    c = (g * xh).sum(axis=1, keepdims=True) / h.shape[1]
    scale = rs * (np.abs(g) + np.abs(xh * c))
    if dh is not None:
        allow = allow + 2 * U32 * np.abs(dx64)
        scale = scale + np.abs(dh)
    bounded = strict & (err > allow)
    off = strict & (np.abs(dx64) >= CANCELLATION * scale)
    out.update(strict=int(strict.sum()), bounded=int(bounded.sum()), off_cancellation=int(off.sum()))
    return out


def dx_check(dx_bits: np.ndarray, dx64: np.ndarray, dy: np.ndarray, h: np.ndarray, w: np.ndarray,
             rstd: np.ndarray, bf16_round, bf16_to_f64, dh: np.ndarray | None = None):
    """(strict, bounded) violation counts of ``dx_report``."""
    r = dx_report(dx_bits, dx64, dy, h, w, rstd, bf16_round, bf16_to_f64, dh=dh)
    return r["strict"], r["bounded"]
