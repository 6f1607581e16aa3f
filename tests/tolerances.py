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
