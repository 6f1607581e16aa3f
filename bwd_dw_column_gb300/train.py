"""Training facade: the RMSNorm as a torch autograd function.

The PR #8208 page ("feat(cake_rmsnorm): opt-in non-deterministic weight
gradient for the autograd RMSNorm", description) lists the package's Python
names: ``cake_rmsnorm``, ``cake_rmsnorm_train_forward``,
``cake_rmsnorm_train_backward``, ``cake_rmsnorm_train_backward_workspace_bytes``,
``cake_rmsnorm_train_backward_workspace`` and ``CakeRMSNormFunction``, each
taking ``deterministic`` (default True).  They are defined here over the C ABI
entry points of this package; every step runs in the library's kernels, and
CPU tensors are rejected (there is no CPU path).

Autograd contract:

* plain route: ``y = cake_rmsnorm(x, w, eps)``; backward gives dx (BF16, x's
  shape) and dw;
* residual route: ``y, h_new = cake_rmsnorm(x, w, eps, residual=res)`` with
  h_new = BF16(x + res) normalised; the gradient reaching h_new directly
  (dh_new) is folded into the one dx the backward computes, which is the
  gradient of both x and res;
* dw is computed in FP32 by the kernels; for a BF16 weight autograd receives
  it rounded to BF16 (the parameter's dtype), for an FP32 weight unchanged.

Only x/h_new, rstd and w are saved for the backward.  The forward is bitwise
reproducible, so a checkpointed step (forward, forward recompute, backward:
the "2xfwd+bwd" operation of the pages' GB300 tables) gives the same
gradients as the plain step.

Workspace: a backward without a caller-owned workspace takes one from a
per-(device, stream) cache that grows to the largest size asked for, so a
training step allocates and zero-fills it once, not on every backward.  The
forms that need it zero leave it zero after every call, and calls on one
stream are ordered, so reusing it is safe.
"""
from __future__ import annotations

import threading

import torch

from . import (cake_rmsnorm_bwd, cake_rmsnorm_bwd_workspace, cake_rmsnorm_bwd_workspace_size,
               cake_rmsnorm_fwd)

_ws_lock = threading.Lock()
_ws_cache: dict = {}


def _cached_workspace(x: torch.Tensor, w_dtype, deterministic: bool) -> torch.Tensor:
    """The (device, current stream) workspace, grown to fit this call."""
    need = max(cake_rmsnorm_bwd_workspace_size(x, w_dtype, deterministic), 256)
    key = (x.device.index, torch.cuda.current_stream(x.device).cuda_stream)
    with _ws_lock:
        ws = _ws_cache.get(key)
        if ws is None or ws.numel() < need:
            ws = torch.zeros(need, dtype=torch.uint8, device=x.device)
            _ws_cache[key] = ws
        return ws

__all__ = [
    "CakeRMSNormFunction", "cake_rmsnorm", "cake_rmsnorm_train_forward", "cake_rmsnorm_train_backward",
    "cake_rmsnorm_train_backward_workspace_bytes", "cake_rmsnorm_train_backward_workspace",
]


def cake_rmsnorm_train_forward(x: torch.Tensor, w: torch.Tensor, eps: float = 1e-6,
                               residual: torch.Tensor | None = None, deterministic: bool = True, **kw):
    """Forward: (y, rstd) or (y, rstd, h_new).  The forward is the same
    program in both modes; ``deterministic`` is accepted for a uniform
    signature."""
    del deterministic
    return cake_rmsnorm_fwd(x, w, eps, residual=residual, **kw)


def cake_rmsnorm_train_backward(dy: torch.Tensor, x: torch.Tensor, rstd: torch.Tensor, w: torch.Tensor,
                                dh: torch.Tensor | None = None, deterministic: bool = True, **kw):
    """Backward: (dx, dw FP32).  x is h_new on the residual route."""
    return cake_rmsnorm_bwd(dy, x, rstd, w, dh, deterministic, **kw)


def cake_rmsnorm_train_backward_workspace_bytes(x_or_shape, w_dtype=torch.bfloat16, deterministic: bool = True) -> int:
    """Workspace bytes the backward needs for this row set."""
    return cake_rmsnorm_bwd_workspace_size(x_or_shape, w_dtype, deterministic)


def cake_rmsnorm_train_backward_workspace(x_or_shape, w_dtype=torch.bfloat16, deterministic: bool = True,
                                          device=None) -> torch.Tensor:
    """A zero-filled workspace for the backward."""
    return cake_rmsnorm_bwd_workspace(x_or_shape, w_dtype, deterministic, device)


class CakeRMSNormFunction(torch.autograd.Function):
    """y = RMSNorm(x [+ residual]) * w with the library's forward and backward.

    ``apply(x, w, eps, residual, deterministic, workspace)``: residual and
    workspace may be None.  A caller-owned workspace (from
    ``cake_rmsnorm_train_backward_workspace``, sized for x, w's dtype and the
    mode) replaces the per-(device, stream) cached one; calls sharing one
    workspace must be stream-ordered.
    """

    @staticmethod
    def forward(ctx, x, w, eps=1e-6, residual=None, deterministic=True, workspace=None):
        if residual is None:
            y, rstd = cake_rmsnorm_fwd(x, w, eps)
            h = x
        else:
            y, rstd, h = cake_rmsnorm_fwd(x, w, eps, residual=residual)
        ctx.save_for_backward(h, rstd, w)
        ctx.has_res = residual is not None
        ctx.deterministic = bool(deterministic)
        ctx.workspace = workspace
        return (y, h) if ctx.has_res else y

    @staticmethod
    def backward(ctx, dy, dh=None):
        h, rstd, w = ctx.saved_tensors
        if dy is None:
            dy = torch.zeros(h.shape, dtype=torch.bfloat16, device=h.device)
        dy = dy.to(torch.bfloat16).contiguous()
        if dh is not None:
            dh = dh.to(torch.bfloat16).contiguous()
        ws = ctx.workspace if ctx.workspace is not None else _cached_workspace(h, w.dtype, ctx.deterministic)
        dx, dw = cake_rmsnorm_bwd(dy, h, rstd, w, dh if ctx.has_res else None, ctx.deterministic, workspace=ws)
        gw = dw if w.dtype == torch.float32 else dw.to(w.dtype)
        return dx, gw, None, (dx if ctx.has_res else None), None, None


def cake_rmsnorm(x: torch.Tensor, w: torch.Tensor, eps: float = 1e-6, residual: torch.Tensor | None = None,
                 deterministic: bool = True, workspace: torch.Tensor | None = None):
    """Differentiable RMSNorm: y, or (y, h_new) with a residual."""
    return CakeRMSNormFunction.apply(x, w, eps, residual, deterministic, workspace)
