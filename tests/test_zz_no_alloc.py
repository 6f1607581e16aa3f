"""The backward entry point that needs no caller scratch.

Callers that cannot allocate device memory for the library (inside a
framework that owns every allocation, or on a path that must not call
cudaMalloc mid-step) use cake_rmsnorm_bwd_noalloc, whose scratch is a device
array owned by the library.  These checks call it through the C ABI twice in
a row and compare it with the workspace-taking entry point running the same
kernel (cake_rmsnorm_bwd_forced, non-deterministic, the single kernel):
dx within one BF16 step (it is in fact the same bits) and dw within the
per-element budget the parity tests use.  The file is named to run last, and
it passes on its own in a fresh process as well as after the other tests.
"""
import numpy as np
import pytest
import torch

import cake_inputs
from tests import tolerances as tol

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(scope="module")
def cake():
    import __graft_entry__
    __graft_entry__.build()
    import bwd_dw_column_gb300 as cake
    return cake


def _bits(t):
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _case(kind):
    if kind == "plain":
        return cake_inputs.plain_case(700, 2048, family="outlier", w_dtype=torch.float32, dy_std=1e-2, seed=21,
                                      device=DEV)
    if kind == "bf16w":
        return cake_inputs.plain_case(301, 1536, w_dtype=torch.bfloat16, seed=22, device=DEV)
    return cake_inputs.heads_case(40, 24, strided=True, w_dtype=torch.float32, seed=23, device=DEV)


@pytest.mark.parametrize("kind", ["plain", "bf16w", "heads"])
def test_noalloc_matches_workspace_entry_point(cake, kind):
    c = _case(kind)
    x, dy, w = c["x"], c["dy"], c["w"]
    H = x.shape[-1]
    _, rstd = cake.cake_rmsnorm_fwd(x, w, c["eps"])
    ref_dx, ref_dw = cake.cake_rmsnorm_bwd_forced(dy, x, rstd, w, deterministic=False, force_single=1)
    torch.cuda.synchronize()
    dx = torch.empty(x.shape, dtype=torch.bfloat16, device=DEV)
    dw = torch.empty(H, dtype=torch.float32, device=DEV)
    for _ in range(2):  # two calls in a row share the built-in scratch
        dx.fill_(0)
        dw.fill_(float("nan"))
        cake.cake_rmsnorm_bwd_noalloc(dy, x, rstd, w, dx=dx, dw=dw)
        torch.cuda.synchronize()
        assert tol.ulp_distance(_bits(dx), _bits(ref_dx)).max() <= 1
        a, b = dw.cpu().numpy().astype(np.float64), ref_dw.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(a))
        assert tol.dw_budget_fraction(a, b).max() <= 1.0
    assert cake.cake_rmsnorm_device_status() == 0


def test_noalloc_rejects_too_many_columns(cake):
    lib = cake.load_library()
    from bwd_dw_column_gb300 import _Shape
    big = _Shape(4, 1, 8200)
    st = lib.cake_rmsnorm_bwd_noalloc(big, None, None, None, None, 0, None, None, None, None)
    assert st == cake.CAKE_ERR_WORKSPACE
