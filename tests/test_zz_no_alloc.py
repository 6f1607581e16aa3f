"""The backward entry point that needs no caller scratch.

Some callers cannot give the library device memory: code inside a framework
that owns every allocation, or a step that must not call cudaMalloc (it can
synchronise the device) part-way through.  They call
cake_rmsnorm_bwd_noalloc, whose scratch (the single kernel's arrival counter
and FP64 column accumulators) is a device array the library owns.

These checks call it through the C ABI twice in a row on the same inputs and
hold both results to the FP64 oracle with the bars of the parity tests: dx
within one BF16 step of RNE_bf16(dx64) (FP32-evaluation allowance near
cancellation, strict count reported) and dw within 1e-4 + 1e-4 |dw64| per
element.  dx must also be the same bits as the workspace-taking entry point
gives, as in every other variant.  The cases cover plain rows with an FP32
and a BF16 weight, a strided per-head view, H = 8192 (the array then holds
one copy of the accumulators instead of eight) and the residual route with a
gradient into h_new.

The file is named to be collected last, and it passes on its own in a fresh
process as well as after the other tests.
"""
import numpy as np
import pytest
import torch

import cake_inputs
import oracle
from tests import tolerances as tol
from tests.test_parity import DEV, bits, oracle_bwd_inputs, rows_f64, to_dev, view_of, w64, wbits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cake():
    import __graft_entry__
    __graft_entry__.build()
    import bwd_dw_column_gb300 as cake
    return cake


def _case(kind):
    if kind == "plain_w32":
        return cake_inputs.plain_case(700, 2048, family="outlier", w_dtype=torch.float32, dy_std=1e-2, seed=21)
    if kind == "plain_bf16w":
        return cake_inputs.plain_case(301, 1536, w_dtype=torch.bfloat16, seed=22)
    if kind == "heads":
        return cake_inputs.heads_case(40, 24, strided=True, w_dtype=torch.float32, seed=23)
    if kind == "h8192":
        return cake_inputs.plain_case(33, 8192, w_dtype=torch.float32, seed=24)
    return cake_inputs.residual_case(77, 6144, seed=25)


@pytest.mark.parametrize("kind", ["plain_w32", "plain_bf16w", "heads", "h8192", "residual_dh"])
def test_noalloc_against_the_oracle(cake, kind):
    c = _case(kind)
    x, dy, w, res = c["x"], c["dy"], c["w"], c.get("residual")
    dh = c.get("dh")
    T = x.shape[0]
    nh = x.shape[1] if x.dim() == 3 else 1
    H = x.shape[-1]
    # both sides take the oracle's rstd (and h_new on the residual route)
    rin, hn = oracle_bwd_inputs(x, w, c["eps"], res)
    h = torch.from_numpy(hn.view(np.int16)).view(torch.bfloat16).reshape(x.shape) if res is not None else x
    hv, dyv = view_of(h), view_of(dy)
    dhv = view_of(dh) if dh is not None else None
    dx64 = oracle.bwd_rows(T, nh, H, dyv, hv, rin, wbits(w), dh=dhv)
    dw64 = oracle.dw_cols(T, nh, H, dyv, hv, rin)
    dyf, hf = rows_f64(dy), rows_f64(h)
    dhf = rows_f64(dh) if dh is not None else None

    h_d, dy_d, w_d, dh_d = to_dev(h), to_dev(dy), w.to(DEV), to_dev(dh)
    r_d = torch.from_numpy(rin).to(DEV)
    ref_dx, _ = cake.cake_rmsnorm_bwd(dy_d, h_d, r_d, w_d, dh_d, deterministic=False)
    torch.cuda.synchronize()
    ref_bits = bits(ref_dx).reshape(-1, H)

    dx = torch.empty(h.shape, dtype=torch.bfloat16, device=DEV)
    dw = torch.empty(H, dtype=torch.float32, device=DEV)
    for call in range(2):  # two calls in a row share the built-in scratch
        dx.fill_(0)
        dw.fill_(float("nan"))
        cake.cake_rmsnorm_bwd_noalloc(dy_d, h_d, r_d, w_d, dh_d, dx=dx, dw=dw)
        torch.cuda.synchronize()
        dxb = bits(dx).reshape(-1, H)
        strict, bounded = tol.dx_check(dxb, dx64, dyf, hf, w64(w), rin, oracle.bf16_round,
                                       oracle.bf16_bits_to_f64, dh=dhf)
        assert bounded == 0, f"call {call}: dx {strict} strict / {bounded} bounded violations"
        np.testing.assert_array_equal(dxb, ref_bits)
        dwk = dw.cpu().numpy()
        assert np.all(np.isfinite(dwk))
        frac = float(tol.dw_budget_fraction(dwk, dw64).max())
        assert frac <= 1.0, f"call {call}: dw worst {frac:.4f} of budget"
    assert cake.cake_rmsnorm_device_status() == 0


def test_noalloc_rejects_too_many_columns(cake):
    lib = cake.load_library()
    from bwd_dw_column_gb300 import _Shape
    big = _Shape(4, 1, 8200)
    st = lib.cake_rmsnorm_bwd_noalloc(big, None, None, None, None, 0, None, None, None, None)
    assert st == cake.CAKE_ERR_WORKSPACE
