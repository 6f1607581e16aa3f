"""FP64 CPU oracle of the training RMSNorm (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline and
reference arms may import this package.  The product path (the CUDA library
and its Python binding) never does, and this package imports nothing from it.

The arithmetic lives in ``cake_oracle.c`` (plain single-threaded C, FP64,
built with ``-O2 -fno-fast-math``); this module only builds it, marshals numpy
arrays into it and decodes BF16 bit patterns.  Every function cites the
passage it follows in the C source's header:

* outputs and dtypes (y BF16, rstd FP32, dx BF16, dw FP32): the "Speedups ...
  GB300 windows" commit (#8577) quoted on the PR #8208 page, intro;
* residual route returns h_new and normalises it: same commit, "Key";
* per-head views with one shared w[256]: PR #8208 page, description;
* dw is checked against FP64 computed at the kernel's FP32 rstd: PR #8208
  page, description.

Parity status: every function here is pinned by ``tests/test_oracle.py``
(finite differences, closed forms, exact sums, invariants, reductions to
special cases); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cake_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libcake_oracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_vp = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libcake_oracle.so`` (gcc, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-std=c99",
             "-fPIC", "-shared", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.cake_oracle_fwd_f64.argtypes = [_i64, _i64, _vp, _vp, ctypes.c_double, _vp, _vp, _vp]
            lib.cake_oracle_bwd_f64.argtypes = [_i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
            lib.cake_oracle_fwd_rows.argtypes = (
                [_i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _i64, _vp, ctypes.c_int,
                 ctypes.c_double, _vp, _vp, _i64, _vp, _vp, _vp, _vp])
            lib.cake_oracle_bwd_rows.argtypes = (
                [_i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _i64, _vp, _vp, ctypes.c_int,
                 _vp, _i64, _i64, _vp, _i64, _vp, _vp])
            lib.cake_oracle_dw_cols.argtypes = (
                [_i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _i64, _vp, _vp, _i64, _vp])
            lib.cake_oracle_bf16_round.argtypes = [_vp, _vp, _i64]
            for f in ("cake_oracle_fwd_f64", "cake_oracle_bwd_f64", "cake_oracle_fwd_rows",
                      "cake_oracle_bwd_rows", "cake_oracle_dw_cols"):
                getattr(lib, f).restype = ctypes.c_int
            lib.cake_oracle_bf16_round.restype = None
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (code {rc})")


# ---------------------------------------------------------------- BF16 bits

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact FP64 values of BF16 bit patterns (uint16)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_round(v: np.ndarray) -> np.ndarray:
    """Round FP64 values to BF16 (ties to even, one rounding); returns uint16 bits."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().cake_oracle_bf16_round(_ptr(v), _ptr(out), v.size)
    return out


# ------------------------------------------------------------ FP64 arrays

def fwd_f64(h: np.ndarray, w: np.ndarray, eps: float, rstd_in: np.ndarray | None = None):
    """Forward on FP64 rows h [R, H]: returns (y [R, H], rstd64 [R])."""
    h = np.ascontiguousarray(h, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    R, H = h.shape
    y = np.empty((R, H))
    r64 = np.empty(R)
    rin = None if rstd_in is None else np.ascontiguousarray(rstd_in, dtype=np.float64)
    _check(_load().cake_oracle_fwd_f64(R, H, _ptr(h), _ptr(w), float(eps), _ptr(rin), _ptr(y), _ptr(r64)), "fwd_f64")
    return y, r64


def bwd_f64(dy: np.ndarray, h: np.ndarray, rstd: np.ndarray, w: np.ndarray, dh: np.ndarray | None = None):
    """Backward on FP64 rows: returns (dx [R, H], dw [H])."""
    dy = np.ascontiguousarray(dy, dtype=np.float64)
    h = np.ascontiguousarray(h, dtype=np.float64)
    rstd = np.ascontiguousarray(rstd, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    dhc = None if dh is None else np.ascontiguousarray(dh, dtype=np.float64)
    R, H = h.shape
    dx = np.empty((R, H))
    dw = np.empty(H)
    _check(_load().cake_oracle_bwd_f64(R, H, _ptr(dy), _ptr(h), _ptr(rstd), _ptr(w), _ptr(dhc), _ptr(dx), _ptr(dw)), "bwd_f64")
    return dx, dw


# ------------------------------------------------- BF16 storage, strided views

class View:
    """A BF16 [T, nh, H] view: a flat uint16 buffer plus element strides.

    Row r is (t, k) = (r // nh, r % nh) at offset t*st + k*sh; the last
    dimension is contiguous.
    """

    def __init__(self, buf: np.ndarray, st: int, sh: int, offset: int = 0):
        assert buf.dtype == np.uint16 and buf.flags.c_contiguous
        self.buf, self.st, self.sh, self.offset = buf, int(st), int(sh), int(offset)

    @staticmethod
    def contiguous(a: np.ndarray) -> "View":
        """View of a C-contiguous uint16 array of shape [T, H] or [T, nh, H]."""
        a = np.ascontiguousarray(a, dtype=np.uint16)
        if a.ndim == 2:
            return View(a.reshape(-1), a.shape[1], a.shape[1])
        return View(a.reshape(-1), a.shape[1] * a.shape[2], a.shape[2])

    def base(self):
        return ctypes.c_void_p(self.buf.ctypes.data + 2 * self.offset)


def _rows_arg(rows):
    if rows is None:
        return None, 0
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    return rows, rows.size


def _weight(w):
    w = np.ascontiguousarray(w)
    if w.dtype == np.float32:
        return w, 1
    assert w.dtype == np.uint16, "weight is FP32 or BF16 bits (uint16)"
    return w, 0


def fwd_rows(T, nh, H, x: View, w, eps, residual: View | None = None, rstd_in=None, rows=None,
             want_y: bool = True, want_h: bool = True):
    """Forward over the listed rows (None: all).

    Returns (y FP64 [n, H], rstd64 [n], h_new BF16 bits [n, H]); y or h_new is
    None when not wanted.  y uses ``rstd_in`` (an FP32 rstd, indexed by row)
    when given, else rstd64.
    """
    rows, n = _rows_arg(rows)
    if rows is None:
        n = T * nh
    w, wf = _weight(w)
    rin = None if rstd_in is None else np.ascontiguousarray(rstd_in, dtype=np.float32)
    y = np.empty((n, H)) if want_y else None
    r64 = np.empty(n)
    hn = np.empty((n, H), dtype=np.uint16) if want_h else None
    work = np.empty(3 * H)
    res_base = residual.base() if residual is not None else None
    _check(_load().cake_oracle_fwd_rows(
        T, nh, H, x.base(), x.st, x.sh,
        res_base, residual.st if residual else 0, residual.sh if residual else 0,
        _ptr(w), wf, float(eps), _ptr(rin), _ptr(rows), n,
        _ptr(y), _ptr(r64), _ptr(hn), _ptr(work)), "fwd_rows")
    return y, r64, hn


def bwd_rows(T, nh, H, dy: View, h: View, rstd, w, dh: View | None = None, rows=None):
    """Backward dx (FP64 [n, H]) over the listed rows (None: all), at the given FP32 rstd."""
    rows, n = _rows_arg(rows)
    if rows is None:
        n = T * nh
    w, wf = _weight(w)
    rstd = np.ascontiguousarray(rstd, dtype=np.float32)
    dx = np.empty((n, H))
    work = np.empty(4 * H)
    _check(_load().cake_oracle_bwd_rows(
        T, nh, H, dy.base(), dy.st, dy.sh, h.base(), h.st, h.sh, _ptr(rstd), _ptr(w), wf,
        dh.base() if dh is not None else None, dh.st if dh else 0, dh.sh if dh else 0,
        _ptr(rows), n, _ptr(dx), _ptr(work)), "bwd_rows")
    return dx


def dw_cols(T, nh, H, dy: View, h: View, rstd, cols=None):
    """dw (FP64) for the listed columns (None: all): exact-order sum over every row."""
    cols, n = _rows_arg(cols)
    if cols is None:
        n = H
    rstd = np.ascontiguousarray(rstd, dtype=np.float32)
    dw = np.empty(n)
    _check(_load().cake_oracle_dw_cols(
        T, nh, H, dy.base(), dy.st, dy.sh, h.base(), h.st, h.sh, _ptr(rstd), _ptr(cols), n, _ptr(dw)),
        "dw_cols")
    return dw
