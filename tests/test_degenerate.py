"""Degenerate inputs through the CUDA path, against the oracle: all-zero rows
(rstd from eps alone), constant rows, rows far below and far above unit
scale, zero upstream gradients, and the cancellation case w = 1, dy = x*rstd
(dx ~ 0).  Same bars as the parity tests."""
import numpy as np
import pytest
import torch

import cake_inputs
from tests.test_parity import DEV, bits, cake, check_bwd, check_fwd  # noqa: F401  (cake: the fixture)

pytestmark = pytest.mark.gpu

VARIANTS = [(0, 0), (0, 1), (1, 1), (3, 3)]


def _mixed_rows(T, H, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((T, H), generator=g)
    x[0:50] = 0.0                 # mean square 0: rstd = 1/sqrt(eps)
    x[50:100] = 0.75              # constant rows (exact in BF16)
    x[100:150] *= 1e-30           # squares underflow FP32: eps decides rstd
    x[150:200] *= 1e6             # rstd near 1e-6 (rstd^3 stays a normal FP32 number)
    return x.to(torch.bfloat16), g


def test_degenerate_rows(cake):
    T, H = 300, 2048
    x, g = _mixed_rows(T, H, 3)
    dy = torch.randn((T, H), generator=g).to(torch.bfloat16)
    dy[200:250] = 0.0             # zero upstream gradient: dx = 0 on those rows
    w = (1.0 + 0.1 * torch.randn(H, generator=g)).to(torch.float32)
    eps = cake_inputs.EPS
    check_fwd(cake, x, w, eps)
    check_bwd(cake, x, dy, w, eps, variants=VARIANTS)


def test_zero_gradient_gives_zero_dx_and_dw(cake):
    c = cake_inputs.plain_case(129, 1536, seed=4)
    dy = torch.zeros_like(c["dy"])
    x, w = c["x"].to(DEV), c["w"].to(DEV)
    _, rstd = cake.cake_rmsnorm_fwd(x, w, c["eps"])
    for det in (True, False):
        dx, dw = cake.cake_rmsnorm_bwd(dy.to(DEV), x, rstd, w, deterministic=det)
        torch.cuda.synchronize()
        assert np.all((bits(dx) & 0x7fff) == 0)  # +0 or -0 only
        assert not dw.abs().max().item()


def test_residual_zero_dy_passes_dh_through(cake):
    c = cake_inputs.residual_case(77, 6144, seed=9)
    dy = torch.zeros_like(c["dy"])
    check_bwd(cake, c["x"], dy, c["w"], c["eps"], residual=c["residual"], dh=c["dh"], variants=[(0, 1), (1, 1)])
    _, rstd, h_new = cake.cake_rmsnorm_fwd(c["x"].to(DEV), c["w"].to(DEV), c["eps"], residual=c["residual"].to(DEV))
    dx, dw = cake.cake_rmsnorm_bwd(dy.to(DEV), h_new, rstd, c["w"].to(DEV), c["dh"].to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(dx.cpu(), c["dh"])  # dx = bf16(0 + dh) = dh
    assert not dw.abs().max().item()


def test_unit_weight_normalised_gradient(cake):
    # w = 1 and dy = x*rstd: the row's gradient is parallel to x, so dx
    # cancels to ~0 (the case the dx bar's FP32-evaluation allowance is for)
    T, H = 64, 1024
    g = torch.Generator().manual_seed(6)
    x = torch.randn((T, H), generator=g).to(torch.bfloat16)
    xf = x.double()
    rs = 1.0 / torch.sqrt((xf * xf).mean(dim=1, keepdim=True) + cake_inputs.EPS)
    dy = (xf * rs).to(torch.bfloat16)
    w = torch.ones(H, dtype=torch.float32)
    check_bwd(cake, x, dy, w, cake_inputs.EPS, variants=[(0, 0), (1, 1)])
