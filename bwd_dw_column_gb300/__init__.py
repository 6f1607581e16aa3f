"""Training RMSNorm for one NVIDIA GB300 (sm_103a): Python binding.

A thin ctypes layer over ``libcake_rmsnorm.so`` (the C ABI declared in
``include/cake_rmsnorm.h``).  It only marshals torch tensors into pointers,
strides and the current CUDA stream; every step of the forward and backward
runs in the library's kernels.  There is no CPU fallback: without the built
library, or without a CUDA device, every compute entry point raises.

Entry points (same names as the C ABI):

* ``cake_rmsnorm_fwd(x, w, eps, residual=None)`` -> ``(y, rstd)`` or
  ``(y, rstd, h_new)`` with a residual;
* ``cake_rmsnorm_bwd(dy, x, rstd, w, dh=None, deterministic=True)`` ->
  ``(dx, dw)``;
* ``cake_rmsnorm_bwd_workspace_size`` / ``cake_rmsnorm_bwd_workspace``;
* ``cake_rmsnorm_bwd_select`` (the window table's choice; host only);
* ``cake_rmsnorm_device_status``, ``cake_status_str``.

Names follow the pages' Python facade (PR #8208 page, description:
forward / backward / workspace entry points taking ``deterministic``, default
True).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "CakeError", "load_library", "cake_rmsnorm_fwd", "cake_rmsnorm_bwd", "cake_rmsnorm_bwd_forced",
    "cake_rmsnorm_bwd_main", "cake_rmsnorm_bwd_reduce", "cake_rmsnorm_bwd_noalloc",
    "cake_rmsnorm_bwd_workspace_size", "cake_rmsnorm_bwd_workspace", "cake_rmsnorm_bwd_workspace_init",
    "cake_rmsnorm_bwd_select", "cake_rmsnorm_bwd_timeout_test", "cake_rmsnorm_bwd_host",
    "cake_rmsnorm_bwd_host_staging_size",
    "cake_rmsnorm_device_status", "cake_status_str", "cake_rmsnorm_plan_occupancy", "LIB_PATH", "DW_PLAIN", "DW_BLOCKED", "DW_TWOSUM", "DW_KAHAN",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcake_rmsnorm.so")

CAKE_OK, CAKE_ERR_INVALID, CAKE_ERR_UNSUPPORTED, CAKE_ERR_WORKSPACE, CAKE_ERR_CUDA, CAKE_ERR_TIMEOUT = range(6)
CAKE_BF16, CAKE_FP32 = 0, 1
DW_PLAIN, DW_BLOCKED, DW_TWOSUM, DW_KAHAN = 0, 1, 2, 3


class CakeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {cake_status_str(status)} (status {status})")


class _Shape(ctypes.Structure):
    _fields_ = [("tokens", ctypes.c_int64), ("heads", ctypes.c_int64), ("hidden", ctypes.c_int64)]


class _Tensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("stride_token", ctypes.c_int64), ("stride_head", ctypes.c_int64)]


class _Variant(ctypes.Structure):
    _fields_ = [("single", ctypes.c_int), ("dw_accum", ctypes.c_int), ("vec_per_thread", ctypes.c_int),
                ("warps_per_row", ctypes.c_int), ("row_groups", ctypes.c_int), ("rows_per_group", ctypes.c_int),
                ("stages", ctypes.c_int),
                ("ctas", ctypes.c_int), ("rows_per_cta", ctypes.c_int64), ("smem_bytes", ctypes.c_size_t),
                ("lanes_per_row", ctypes.c_int)]


_P = ctypes.POINTER
_vp = ctypes.c_void_p
_lib = None
_lock = threading.Lock()


def load_library(path: str = LIB_PATH):
    """Load (once) and return the ctypes handle of libcake_rmsnorm.so."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        lib.cake_rmsnorm_abi_version.restype = ctypes.c_int
        lib.cake_status_str.restype = ctypes.c_char_p
        lib.cake_status_str.argtypes = [ctypes.c_int]
        lib.cake_rmsnorm_fwd.restype = ctypes.c_int
        lib.cake_rmsnorm_fwd.argtypes = [_P(_Shape), _P(_Tensor), _P(_Tensor), _vp, ctypes.c_int, ctypes.c_float,
                                         _P(_Tensor), _P(_Tensor), _vp, _vp]
        lib.cake_rmsnorm_bwd_workspace_size.restype = ctypes.c_size_t
        lib.cake_rmsnorm_bwd_workspace_size.argtypes = [_P(_Shape), ctypes.c_int, ctypes.c_int]
        lib.cake_rmsnorm_bwd_workspace_init.restype = ctypes.c_int
        lib.cake_rmsnorm_bwd_workspace_init.argtypes = [_vp, ctypes.c_size_t, _vp]
        lib.cake_rmsnorm_bwd.restype = ctypes.c_int
        lib.cake_rmsnorm_bwd.argtypes = [_P(_Shape), _P(_Tensor), _P(_Tensor), _vp, _vp, ctypes.c_int, _P(_Tensor),
                                         _P(_Tensor), _vp, _vp, ctypes.c_size_t, ctypes.c_int, _vp]
        lib.cake_rmsnorm_bwd_forced.restype = ctypes.c_int
        lib.cake_rmsnorm_bwd_forced.argtypes = [_P(_Shape), _P(_Tensor), _P(_Tensor), _vp, _vp, ctypes.c_int,
                                                _P(_Tensor), _P(_Tensor), _vp, _vp, ctypes.c_size_t, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_int, _vp]
        lib.cake_rmsnorm_bwd_main.restype = ctypes.c_int
        lib.cake_rmsnorm_bwd_main.argtypes = [_P(_Shape), _P(_Tensor), _P(_Tensor), _vp, _vp, ctypes.c_int,
                                              _P(_Tensor), _P(_Tensor), _vp, _vp, ctypes.c_size_t, ctypes.c_int, _vp]
        lib.cake_rmsnorm_bwd_reduce.restype = ctypes.c_int
        lib.cake_rmsnorm_bwd_reduce.argtypes = [_P(_Shape), ctypes.c_int, _vp, _vp, ctypes.c_size_t, _vp]
        lib.cake_rmsnorm_bwd_noalloc.restype = ctypes.c_int
        lib.cake_rmsnorm_bwd_noalloc.argtypes = [_P(_Shape), _P(_Tensor), _P(_Tensor), _vp, _vp, ctypes.c_int,
                                                 _P(_Tensor), _P(_Tensor), _vp, _vp]
        lib.cake_rmsnorm_bwd_host_staging_size.restype = ctypes.c_size_t
        lib.cake_rmsnorm_bwd_host_staging_size.argtypes = [_P(_Shape), ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.cake_rmsnorm_bwd_host.restype = ctypes.c_int
        lib.cake_rmsnorm_bwd_host.argtypes = [_P(_Shape), _vp, _vp, _vp, _vp, ctypes.c_int, _vp, _vp, _vp, _vp,
                                              ctypes.c_size_t, ctypes.c_int, ctypes.c_int, _vp]
        lib.cake_rmsnorm_bwd_timeout_test.restype = ctypes.c_int
        lib.cake_rmsnorm_bwd_timeout_test.argtypes = [_P(_Shape), _P(_Tensor), _P(_Tensor), _vp, _vp, ctypes.c_int,
                                                      _P(_Tensor), _vp, _vp, ctypes.c_size_t, ctypes.c_uint32, _vp]
        lib.cake_rmsnorm_bwd_select.restype = ctypes.c_int
        lib.cake_rmsnorm_bwd_select.argtypes = [_P(_Shape), ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int, _P(_Variant)]
        lib.cake_rmsnorm_plan_occupancy.restype = ctypes.c_int
        lib.cake_rmsnorm_plan_occupancy.argtypes = [_P(_Shape), ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                    _P(ctypes.c_int), _P(ctypes.c_int)]
        lib.cake_rmsnorm_device_status.restype = ctypes.c_int
        lib.cake_rmsnorm_device_status.argtypes = [_P(ctypes.c_int), ctypes.c_int]
        _lib = lib
        return lib


def cake_status_str(status: int) -> str:
    return load_library().cake_status_str(int(status)).decode()


def _check(status: int, what: str):
    if status != CAKE_OK:
        raise CakeError(status, what)


# ---------------------------------------------------------------- marshalling

def _rows_of(t: torch.Tensor):
    """(T, nh, H, stride_token, stride_head) of a [T, H] or [T, nh, H] view."""
    if t.dim() == 2:
        T, H = t.shape
        return T, 1, H, t.stride(0), 0
    if t.dim() == 3:
        T, nh, H = t.shape
        return T, nh, H, t.stride(0), t.stride(1)
    raise ValueError(f"expected a [T, H] or [T, nh, H] tensor, got shape {tuple(t.shape)}")


def _shape(t: torch.Tensor) -> _Shape:
    T, nh, H, _, _ = _rows_of(t)
    return _Shape(T, nh, H)


def _tensor(t: torch.Tensor | None) -> _Tensor | None:
    if t is None:
        return None
    if t.dtype != torch.bfloat16:
        raise TypeError(f"activations are BF16, got {t.dtype}")
    if t.numel() and t.stride(-1) != 1:
        raise ValueError("the hidden dimension must be contiguous")
    _, _, _, st, sh = _rows_of(t)
    return _Tensor(t.data_ptr(), st, sh)


def _same_rows(a: torch.Tensor, b: torch.Tensor, what: str):
    if a.shape != b.shape:
        raise ValueError(f"{what} has shape {tuple(b.shape)}, expected {tuple(a.shape)}")


def _w_dtype(w: torch.Tensor) -> int:
    if w.dtype == torch.bfloat16:
        return CAKE_BF16
    if w.dtype == torch.float32:
        return CAKE_FP32
    raise TypeError(f"weight is BF16 or FP32, got {w.dtype}")


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("every tensor must be on a CUDA device (no CPU path)")


# -------------------------------------------------------------------- forward

def cake_rmsnorm_fwd(x: torch.Tensor, w: torch.Tensor, eps: float = 1e-6, residual: torch.Tensor | None = None,
                     *, y: torch.Tensor | None = None, h_new: torch.Tensor | None = None,
                     rstd: torch.Tensor | None = None, stream=None):
    """Forward: returns (y, rstd), or (y, rstd, h_new) when ``residual`` is given.

    x, residual: BF16 [T, H] or [T, nh, H] views (hidden dim contiguous);
    w: [H] BF16 or FP32.  Outputs default to fresh contiguous tensors.
    """
    lib = load_library()
    _need_cuda(x, w, residual, y, h_new, rstd)
    T, nh, H, _, _ = _rows_of(x)
    if residual is not None:
        _same_rows(x, residual, "residual")
    if y is None:
        y = torch.empty(x.shape, dtype=torch.bfloat16, device=x.device)
    if rstd is None:
        rstd = torch.empty(T * nh, dtype=torch.float32, device=x.device)
    if residual is not None and h_new is None:
        h_new = torch.empty(x.shape, dtype=torch.bfloat16, device=x.device)
    _same_rows(x, y, "y")
    if rstd.dtype != torch.float32 or rstd.numel() != T * nh or not rstd.is_contiguous():
        raise ValueError("rstd must be a contiguous FP32 tensor of T*nh elements")
    w = w.contiguous()
    shape = _shape(x)
    st = lib.cake_rmsnorm_fwd(ctypes.byref(shape), ctypes.byref(_tensor(x)),
                              ctypes.byref(_tensor(residual)) if residual is not None else None,
                              ctypes.c_void_p(w.data_ptr()), _w_dtype(w), float(eps),
                              ctypes.byref(_tensor(y)),
                              ctypes.byref(_tensor(h_new)) if residual is not None else None,
                              ctypes.c_void_p(rstd.data_ptr()), _stream(stream))
    _check(st, "cake_rmsnorm_fwd")
    return (y, rstd, h_new) if residual is not None else (y, rstd)


# ------------------------------------------------------------------- backward

def cake_rmsnorm_bwd_workspace_size(x_or_shape, w_dtype=torch.bfloat16, deterministic: bool = True) -> int:
    """Workspace bytes the backward needs for this row set ([T, H] / [T, nh, H] tensor or (T, nh, H))."""
    lib = load_library()
    if isinstance(x_or_shape, torch.Tensor):
        shape = _shape(x_or_shape)
    else:
        shape = _Shape(*x_or_shape)
    wd = CAKE_FP32 if w_dtype in (torch.float32, CAKE_FP32) else CAKE_BF16
    return int(lib.cake_rmsnorm_bwd_workspace_size(ctypes.byref(shape), wd, int(bool(deterministic))))


def cake_rmsnorm_bwd_workspace(x_or_shape, w_dtype=torch.bfloat16, deterministic: bool = True,
                               device=None) -> torch.Tensor:
    """A zero-filled workspace of the right size (uint8 tensor on ``device``)."""
    n = cake_rmsnorm_bwd_workspace_size(x_or_shape, w_dtype, deterministic)
    if device is None:
        device = x_or_shape.device if isinstance(x_or_shape, torch.Tensor) else torch.device("cuda")
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device)


def _bwd(dy, x, rstd, w, dh, deterministic, workspace, dx, dw, stream, force_single, force_accum, main_only=False):
    lib = load_library()
    _need_cuda(dy, x, rstd, w, dh, workspace, dx, dw)
    _same_rows(x, dy, "dy")
    if dh is not None:
        _same_rows(x, dh, "dh")
    T, nh, H, _, _ = _rows_of(x)
    if rstd.dtype != torch.float32 or rstd.numel() != T * nh or not rstd.is_contiguous():
        raise ValueError("rstd must be a contiguous FP32 tensor of T*nh elements")
    if dx is None:
        dx = torch.empty(x.shape, dtype=torch.bfloat16, device=x.device)
    _same_rows(x, dx, "dx")
    if dw is None:
        dw = torch.empty(H, dtype=torch.float32, device=x.device)
    if dw.dtype != torch.float32 or dw.numel() != H or not dw.is_contiguous():
        raise ValueError("dw must be a contiguous FP32 tensor of H elements")
    if workspace is None:
        workspace = cake_rmsnorm_bwd_workspace(x, w.dtype, deterministic)
    w = w.contiguous()
    shape = _shape(x)
    args = [ctypes.byref(shape), ctypes.byref(_tensor(dy)), ctypes.byref(_tensor(x)),
            ctypes.c_void_p(rstd.data_ptr()), ctypes.c_void_p(w.data_ptr()), _w_dtype(w),
            ctypes.byref(_tensor(dh)) if dh is not None else None, ctypes.byref(_tensor(dx)),
            ctypes.c_void_p(dw.data_ptr()), ctypes.c_void_p(workspace.data_ptr()),
            workspace.numel() * workspace.element_size(), int(bool(deterministic))]
    if main_only:
        st = lib.cake_rmsnorm_bwd_main(*args[:-1], -1 if force_accum is None else int(force_accum), _stream(stream))
        _check(st, "cake_rmsnorm_bwd_main")
    elif force_single is None and force_accum is None:
        st = lib.cake_rmsnorm_bwd(*args, _stream(stream))
        _check(st, "cake_rmsnorm_bwd")
    else:
        st = lib.cake_rmsnorm_bwd_forced(*args, -1 if force_single is None else int(force_single),
                                         -1 if force_accum is None else int(force_accum), _stream(stream))
        _check(st, "cake_rmsnorm_bwd_forced")
    return dx, dw


def cake_rmsnorm_bwd(dy: torch.Tensor, x: torch.Tensor, rstd: torch.Tensor, w: torch.Tensor,
                     dh: torch.Tensor | None = None, deterministic: bool = True, *,
                     workspace: torch.Tensor | None = None, dx: torch.Tensor | None = None,
                     dw: torch.Tensor | None = None, stream=None):
    """Backward: returns (dx, dw).

    x is the normalised input (h_new on the residual route); dh (optional)
    is the gradient reaching h_new directly and is added into dx.  A
    workspace from ``cake_rmsnorm_bwd_workspace`` is allocated when none is
    given (pass one in to avoid the allocation on every call).
    """
    return _bwd(dy, x, rstd, w, dh, deterministic, workspace, dx, dw, stream, None, None)


def cake_rmsnorm_bwd_forced(dy, x, rstd, w, dh=None, deterministic=True, *, force_single=None,
                            force_accum=None, workspace=None, dx=None, dw=None, stream=None):
    """Backward with the variant forced (single kernel or pair; dw accumulation form)."""
    return _bwd(dy, x, rstd, w, dh, deterministic, workspace, dx, dw, stream, force_single, force_accum)


def cake_rmsnorm_bwd_main(dy, x, rstd, w, dh=None, *, workspace, dx=None, dw=None, force_accum=None, stream=None):
    """First half of the deterministic pair: dx, and the CTA dw partials into ``workspace``."""
    return _bwd(dy, x, rstd, w, dh, True, workspace, dx, dw, stream, None, force_accum, main_only=True)[0]


def cake_rmsnorm_bwd_reduce(x_or_shape, dw: torch.Tensor, workspace: torch.Tensor, has_dh: bool = False,
                            stream=None) -> torch.Tensor:
    """Second half of the deterministic pair: dw from the partials in ``workspace`` (fixed order)."""
    lib = load_library()
    shape = _shape(x_or_shape) if isinstance(x_or_shape, torch.Tensor) else _Shape(*x_or_shape)
    _need_cuda(dw, workspace)
    st = lib.cake_rmsnorm_bwd_reduce(ctypes.byref(shape), int(bool(has_dh)), ctypes.c_void_p(dw.data_ptr()),
                                     ctypes.c_void_p(workspace.data_ptr()),
                                     workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "cake_rmsnorm_bwd_reduce")
    return dw


def cake_rmsnorm_bwd_noalloc(dy: torch.Tensor, x: torch.Tensor, rstd: torch.Tensor, w: torch.Tensor,
                             dh: torch.Tensor | None = None, *, dx: torch.Tensor, dw: torch.Tensor, stream=None):
    """Non-deterministic backward whose scratch is the library's own device array.

    For callers that cannot allocate device memory for the library: no
    workspace is passed and nothing is allocated here either, so dx and dw
    must be given.  Calls share that scratch: keep them on one stream.
    """
    lib = load_library()
    _need_cuda(dy, x, rstd, w, dh, dx, dw)
    _same_rows(x, dy, "dy")
    _same_rows(x, dx, "dx")
    if dh is not None:
        _same_rows(x, dh, "dh")
    T, nh, H, _, _ = _rows_of(x)
    if rstd.dtype != torch.float32 or rstd.numel() != T * nh or not rstd.is_contiguous():
        raise ValueError("rstd must be a contiguous FP32 tensor of T*nh elements")
    if dw.dtype != torch.float32 or dw.numel() != H or not dw.is_contiguous():
        raise ValueError("dw must be a contiguous FP32 tensor of H elements")
    if not w.is_contiguous():
        raise ValueError("w must be contiguous")
    shape = _shape(x)
    st = lib.cake_rmsnorm_bwd_noalloc(ctypes.byref(shape), ctypes.byref(_tensor(dy)), ctypes.byref(_tensor(x)),
                                      ctypes.c_void_p(rstd.data_ptr()), ctypes.c_void_p(w.data_ptr()), _w_dtype(w),
                                      ctypes.byref(_tensor(dh)) if dh is not None else None,
                                      ctypes.byref(_tensor(dx)), ctypes.c_void_p(dw.data_ptr()), _stream(stream))
    _check(st, "cake_rmsnorm_bwd_noalloc")
    return dx, dw


def cake_rmsnorm_bwd_host_staging_size(x_or_shape, w_dtype=torch.bfloat16, has_dh: bool = False,
                                       chunks: int = 8) -> int:
    """Device staging bytes cake_rmsnorm_bwd_host needs for this row set."""
    lib = load_library()
    shape = _shape(x_or_shape) if isinstance(x_or_shape, torch.Tensor) else _Shape(*x_or_shape)
    wd = CAKE_FP32 if w_dtype in (torch.float32, CAKE_FP32) else CAKE_BF16
    return int(lib.cake_rmsnorm_bwd_host_staging_size(ctypes.byref(shape), wd, int(bool(has_dh)), int(chunks)))


def _host_rows(t: torch.Tensor, what: str, dtype) -> torch.Tensor:
    if t.is_cuda:
        raise ValueError(f"{what} is a host tensor here")
    if t.dtype != dtype:
        raise TypeError(f"{what} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous (dense rows)")
    return t


def cake_rmsnorm_bwd_host(dy: torch.Tensor, x: torch.Tensor, rstd: torch.Tensor, w: torch.Tensor,
                          dh: torch.Tensor | None = None, *, dx: torch.Tensor, dw: torch.Tensor,
                          staging: torch.Tensor, chunks: int = 8, deterministic: bool = True, stream=None):
    """Backward over host (CPU, preferably pinned) tensors: the chunked copies and
    kernels overlap on the device.  dx and dw are host tensors written once the
    stream reaches the end of the call; staging is a device uint8 tensor of
    cake_rmsnorm_bwd_host_staging_size bytes."""
    lib = load_library()
    for t, n in ((dy, "dy"), (x, "x"), (dh, "dh"), (dx, "dx")):
        if t is not None:
            _host_rows(t, n, torch.bfloat16)
            _same_rows(x, t, n)
    _host_rows(rstd, "rstd", torch.float32)
    _host_rows(dw, "dw", torch.float32)
    if w.is_cuda or not w.is_contiguous():
        raise ValueError("w is a contiguous host tensor here")
    _need_cuda(staging)
    T, nh, H, _, _ = _rows_of(x)
    if rstd.numel() != T * nh or dw.numel() != H:
        raise ValueError("rstd must hold T*nh and dw H elements")
    shape = _shape(x)
    st = lib.cake_rmsnorm_bwd_host(ctypes.byref(shape), ctypes.c_void_p(dy.data_ptr()), ctypes.c_void_p(x.data_ptr()),
                                   ctypes.c_void_p(rstd.data_ptr()), ctypes.c_void_p(w.data_ptr()), _w_dtype(w),
                                   ctypes.c_void_p(dh.data_ptr()) if dh is not None else None,
                                   ctypes.c_void_p(dx.data_ptr()), ctypes.c_void_p(dw.data_ptr()),
                                   ctypes.c_void_p(staging.data_ptr()), staging.numel() * staging.element_size(),
                                   int(chunks), int(bool(deterministic)), _stream(stream))
    _check(st, "cake_rmsnorm_bwd_host")
    return dx, dw


def cake_rmsnorm_bwd_timeout_test(dy: torch.Tensor, x: torch.Tensor, rstd: torch.Tensor, w: torch.Tensor, *,
                                  workspace: torch.Tensor, dx: torch.Tensor, dw: torch.Tensor,
                                  wait_limit_us: int = 2000, stream=None):
    """Run the grid form with a barrier that cannot complete, so that its bounded
    wait runs out after ``wait_limit_us`` (tests of the timeout path).  Afterwards
    the device status reads CAKE_ERR_TIMEOUT and ``workspace`` needs
    re-initialising."""
    lib = load_library()
    _need_cuda(dy, x, rstd, w, workspace, dx, dw)
    _same_rows(x, dy, "dy")
    _same_rows(x, dx, "dx")
    shape = _shape(x)
    st = lib.cake_rmsnorm_bwd_timeout_test(ctypes.byref(shape), ctypes.byref(_tensor(dy)), ctypes.byref(_tensor(x)),
                                           ctypes.c_void_p(rstd.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                           _w_dtype(w), ctypes.byref(_tensor(dx)), ctypes.c_void_p(dw.data_ptr()),
                                           ctypes.c_void_p(workspace.data_ptr()),
                                           workspace.numel() * workspace.element_size(), int(wait_limit_us),
                                           _stream(stream))
    _check(st, "cake_rmsnorm_bwd_timeout_test")


def cake_rmsnorm_bwd_workspace_init(workspace: torch.Tensor, stream=None) -> torch.Tensor:
    """Zero a workspace (an asynchronous memset on the stream)."""
    lib = load_library()
    _need_cuda(workspace)
    st = lib.cake_rmsnorm_bwd_workspace_init(ctypes.c_void_p(workspace.data_ptr()),
                                             workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "cake_rmsnorm_bwd_workspace_init")
    return workspace


def cake_rmsnorm_bwd_select(shape, w_dtype=torch.bfloat16, deterministic=True, has_dh=False,
                            force_single=None, force_accum=None) -> dict:
    """The window table's variant for (T, nh, H) -- host only, no GPU needed."""
    lib = load_library()
    v = _Variant()
    wd = CAKE_FP32 if w_dtype in (torch.float32, CAKE_FP32) else CAKE_BF16
    st = lib.cake_rmsnorm_bwd_select(ctypes.byref(_Shape(*shape)), wd, int(bool(deterministic)), int(bool(has_dh)),
                                     -1 if force_single is None else int(force_single),
                                     -1 if force_accum is None else int(force_accum), ctypes.byref(v))
    _check(st, "cake_rmsnorm_bwd_select")
    return {f: getattr(v, f) for f, _ in _Variant._fields_}


def cake_rmsnorm_plan_occupancy(shape, backward=True, has_extra=False, deterministic=True, force_accum=None):
    """(planned, resident) CTAs per SM for the kernel a call would launch (needs the GPU)."""
    lib = load_library()
    a, b = ctypes.c_int(0), ctypes.c_int(0)
    st = lib.cake_rmsnorm_plan_occupancy(ctypes.byref(_Shape(*shape)), int(bool(backward)), int(bool(has_extra)),
                                         int(bool(deterministic)), -1 if force_accum is None else int(force_accum),
                                         ctypes.byref(a), ctypes.byref(b))
    _check(st, "cake_rmsnorm_plan_occupancy")
    return a.value, b.value


def cake_rmsnorm_device_status(clear: bool = True) -> int:
    """The kernels' device status word (0, or 5 after a bounded wait ran out).  Synchronises."""
    lib = load_library()
    code = ctypes.c_int(0)
    _check(lib.cake_rmsnorm_device_status(ctypes.byref(code), int(bool(clear))), "cake_rmsnorm_device_status")
    return code.value


# the training facade (autograd function and the pages' Python names)
from .train import (CakeRMSNormFunction, cake_rmsnorm, cake_rmsnorm_train_backward,  # noqa: E402
                    cake_rmsnorm_train_backward_workspace, cake_rmsnorm_train_backward_workspace_bytes,
                    cake_rmsnorm_train_forward)

__all__ += ["CakeRMSNormFunction", "cake_rmsnorm", "cake_rmsnorm_train_forward", "cake_rmsnorm_train_backward",
            "cake_rmsnorm_train_backward_workspace_bytes", "cake_rmsnorm_train_backward_workspace"]
