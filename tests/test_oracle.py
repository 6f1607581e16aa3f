"""Pins for the FP64 oracle: each check ties it to something other than itself.

* finite differences of the FP64 forward (dx, dw, the residual gradient);
* torch autograd on an FP64 restatement of the forward;
* closed forms: H = 1, a constant row, a hand-worked two-element row;
* invariants: sum_j h_j dx_j = 0 at eps = 0, scale invariance at eps = 0;
* dw as an exact-order FP64 sum: bitwise equal to a Python-float loop in
  ascending row order, within the recursive-summation bound of math.fsum, and
  exactly equal to a Fraction sum on an exactly summable input;
* strided per-head views against gathered contiguous copies;
* BF16 rounding against torch's FP32 -> BF16 cast, plus ties, overflow and
  the double-rounding trap that an FP64 -> FP32 -> BF16 path would fall into.

Any plausible slip in the oracle (a dropped 1/H, a wrong sign, w indexed by
row, rstd applied twice or not at all, eps outside the root, a stride mix-up,
y ignoring the kernel's rstd) breaks at least one of these.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle


def _rng(seed=0):
    return np.random.default_rng(seed)


def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# ----------------------------------------------------------- finite differences

def _loss(h, w, dy, eps, dh=None):
    y, _ = oracle.fwd_f64(h, w, eps)
    val = math.fsum((y * dy).ravel())
    if dh is not None:
        val += math.fsum((h * dh).ravel())
    return val


@pytest.mark.parametrize("R,H,eps", [(3, 5, 1e-6), (2, 16, 0.25), (4, 1, 0.5), (1, 7, 0.0)])
@pytest.mark.parametrize("with_dh", [False, True])
def test_finite_differences(R, H, eps, with_dh):
    rng = _rng(R * 100 + H)
    h = rng.normal(size=(R, H))
    w = 1.0 + 0.3 * rng.normal(size=H)
    dy = rng.normal(size=(R, H))
    dh = rng.normal(size=(R, H)) if with_dh else None
    _, r64 = oracle.fwd_f64(h, w, eps)
    dx, dw = oracle.bwd_f64(dy, h, r64, w, dh)
    step = 1e-5
    fd_dx = np.empty_like(h)
    for idx in np.ndindex(h.shape):
        hp, hm = h.copy(), h.copy()
        hp[idx] += step
        hm[idx] -= step
        fd_dx[idx] = (_loss(hp, w, dy, eps, dh) - _loss(hm, w, dy, eps, dh)) / (2 * step)
    fd_dw = np.empty_like(w)
    for j in range(H):
        wp, wm = w.copy(), w.copy()
        wp[j] += step
        wm[j] -= step
        fd_dw[j] = (_loss(h, wp, dy, eps, dh) - _loss(h, wm, dy, eps, dh)) / (2 * step)
    scale = 1.0 + np.abs(fd_dx).max()
    assert np.abs(dx - fd_dx).max() <= 1e-7 * scale
    assert np.abs(dw - fd_dw).max() <= 1e-7 * (1.0 + np.abs(fd_dw).max())


def test_torch_autograd_fp64():
    rng = _rng(7)
    R, H, eps = 6, 24, 1e-3
    h = rng.normal(size=(R, H))
    w = 1.0 + 0.1 * rng.normal(size=H)
    dy = rng.normal(size=(R, H))
    th = torch.tensor(h, requires_grad=True)
    tw = torch.tensor(w, requires_grad=True)
    y = th * torch.rsqrt((th * th).mean(dim=1, keepdim=True) + eps) * tw
    (y * torch.tensor(dy)).sum().backward()
    yo, r64 = oracle.fwd_f64(h, w, eps)
    dx, dw = oracle.bwd_f64(dy, h, r64, w)
    np.testing.assert_allclose(yo, y.detach().numpy(), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dx, th.grad.numpy(), rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(dw, tw.grad.numpy(), rtol=1e-11, atol=1e-13)


# ----------------------------------------------------------------- closed forms

def test_h1_closed_form():
    x = np.array([[0.5], [-2.0], [3.0]])
    w = np.array([1.5])
    dy = np.array([[1.0], [0.25], [-3.0]])
    for eps in (0.0, 0.1):
        y, r64 = oracle.fwd_f64(x, w, eps)
        np.testing.assert_allclose(r64, 1.0 / np.sqrt(x[:, 0] ** 2 + eps), rtol=1e-15)
        np.testing.assert_allclose(y[:, 0], w[0] * x[:, 0] / np.sqrt(x[:, 0] ** 2 + eps), rtol=1e-15)
        dx, dw = oracle.bwd_f64(dy, x, r64, w)
        # d/dx [w x (x^2+eps)^(-1/2)] = w eps (x^2+eps)^(-3/2)
        np.testing.assert_allclose(dx[:, 0], dy[:, 0] * w[0] * eps / (x[:, 0] ** 2 + eps) ** 1.5,
                                   rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(dw[0], np.sum(dy[:, 0] * x[:, 0] / np.sqrt(x[:, 0] ** 2 + eps)), rtol=1e-15)


def test_constant_row():
    H, c, eps = 12, -1.75, 0.0625
    w = np.linspace(0.5, 2.0, H)
    y, r64 = oracle.fwd_f64(np.full((1, H), c), w, eps)
    rs = 1.0 / math.sqrt(c * c + eps)
    assert r64[0] == pytest.approx(rs, rel=1e-15)
    np.testing.assert_allclose(y[0], c * rs * w, rtol=1e-15)


def test_hand_worked_two_elements():
    # h = [3, 4], w = [1, 2], dy = [1, 1], eps = 0:
    # ms = 25/2, r = rstd = 1/sqrt(12.5), r^2 = 2/25.
    # g = [1, 2], xhat = [3r, 4r], c = (3r + 8r)/2 = 11r/2,
    # dx = r (g - xhat c) = r [1 - 33/50, 2 - 44/50] ... with r^2 = 2/25:
    #    1 - 3r*11r/2 = 1 - 33/25 = -8/25,  2 - 4r*11r/2 = 2 - 44/25 = 6/25
    # dw = dy * xhat = [3r, 4r];  y = h r w = [3r, 8r].
    r = 1.0 / math.sqrt(12.5)
    h = np.array([[3.0, 4.0]])
    w = np.array([1.0, 2.0])
    y, r64 = oracle.fwd_f64(h, w, 0.0)
    assert r64[0] == pytest.approx(r, rel=1e-15)
    np.testing.assert_allclose(y[0], [3 * r, 8 * r], rtol=1e-15)
    dx, dw = oracle.bwd_f64(np.ones((1, 2)), h, r64, w)
    np.testing.assert_allclose(dx[0], [r * -8 / 25, r * 6 / 25], rtol=1e-13)
    np.testing.assert_allclose(dw, [3 * r, 4 * r], rtol=1e-15)


def test_zero_gradient():
    rng = _rng(3)
    h = rng.normal(size=(4, 9))
    w = rng.normal(size=9)
    _, r64 = oracle.fwd_f64(h, w, 1e-6)
    dx, dw = oracle.bwd_f64(np.zeros_like(h), h, r64, w)
    assert not dx.any() and not dw.any()


def test_unit_weight_normalised_dy_gives_zero_dx():
    # with w = 1, eps = 0 and dy = xhat, the gradient is along the row itself,
    # which the normalisation removes: dx = 0.
    rng = _rng(4)
    h = rng.normal(size=(3, 10))
    w = np.ones(10)
    _, r64 = oracle.fwd_f64(h, w, 0.0)
    dx, _ = oracle.bwd_f64(h * r64[:, None], h, r64, w)
    assert np.abs(dx).max() < 1e-14


# ------------------------------------------------------------------- invariants

def test_orthogonality_at_eps0():
    rng = _rng(5)
    R, H = 8, 33
    h = rng.normal(size=(R, H)) * rng.uniform(0.1, 10, size=(R, 1))
    w = 1.0 + 0.2 * rng.normal(size=H)
    dy = rng.normal(size=(R, H))
    _, r64 = oracle.fwd_f64(h, w, 0.0)
    dx, _ = oracle.bwd_f64(dy, h, r64, w)
    dots = (h * dx).sum(axis=1)
    scale = (np.abs(h * dy * w).sum(axis=1)) * r64
    assert np.all(np.abs(dots) <= 1e-13 * scale)


def test_scale_invariance_at_eps0():
    rng = _rng(6)
    h = rng.normal(size=(5, 16))
    w = 1.0 + 0.1 * rng.normal(size=16)
    dy = rng.normal(size=(5, 16))
    alpha = 7.25
    y1, r1 = oracle.fwd_f64(h, w, 0.0)
    y2, r2 = oracle.fwd_f64(alpha * h, w, 0.0)
    np.testing.assert_allclose(y2, y1, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(r2 * alpha, r1, rtol=1e-15)
    dx1, dw1 = oracle.bwd_f64(dy, h, r1, w)
    dx2, dw2 = oracle.bwd_f64(dy, alpha * h, r2, w)
    np.testing.assert_allclose(dx2 * alpha, dx1, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dw2, dw1, rtol=1e-14)


# ------------------------------------------------------------- dw column sums

def _bf16_rows(rng, shape, scale=1.0):
    return _bf16_bits(torch.tensor(rng.normal(size=shape) * scale, dtype=torch.float32).to(torch.bfloat16))


def test_dw_is_exact_order_fp64_sum():
    rng = _rng(8)
    T, H = 3000, 8
    dy = _bf16_rows(rng, (T, H))
    x = _bf16_rows(rng, (T, H), 3.0)
    rstd = rng.uniform(0.2, 2.0, size=T).astype(np.float32)
    dw = oracle.dw_cols(T, 1, H, oracle.View.contiguous(dy), oracle.View.contiguous(x), rstd)
    dyd, xd, rd = oracle.bf16_bits_to_f64(dy), oracle.bf16_bits_to_f64(x), rstd.astype(np.float64)
    for j in range(H):
        terms = [float(dyd[r, j]) * float(xd[r, j]) * float(rd[r]) for r in range(T)]
        # each term is exact in FP64: 8 x 8 significant bits times a 24-bit rstd.
        for r in range(0, T, 97):
            assert Fraction(terms[r]) == Fraction(float(dyd[r, j])) * Fraction(float(xd[r, j])) * Fraction(float(rd[r]))
        s = 0.0
        for t in terms:  # ascending rows, one IEEE-754 double rounding per add
            s += t
        assert dw[j] == s
        exact = math.fsum(terms)
        bound = (T - 1) * 2.0 ** -53 * math.fsum(abs(t) for t in terms)
        assert abs(dw[j] - exact) <= bound


def test_dw_exact_on_exactly_summable_input():
    rng = _rng(9)
    T, H = 500, 4
    dyv = rng.integers(-8, 9, size=(T, H)).astype(np.float32)
    xv = rng.integers(-8, 9, size=(T, H)).astype(np.float32)
    dy = _bf16_bits(torch.tensor(dyv).to(torch.bfloat16))
    x = _bf16_bits(torch.tensor(xv).to(torch.bfloat16))
    rstd = np.full(T, 0.5, dtype=np.float32)
    dw = oracle.dw_cols(T, 1, H, oracle.View.contiguous(dy), oracle.View.contiguous(x), rstd)
    for j in range(H):
        exact = sum((Fraction(int(a)) * Fraction(int(b)) * Fraction(1, 2) for a, b in zip(dyv[:, j], xv[:, j])),
                    Fraction(0))
        assert Fraction(dw[j]) == exact


def test_dw_uses_given_rstd():
    rng = _rng(10)
    T, H = 64, 16
    dy, x = _bf16_rows(rng, (T, H)), _bf16_rows(rng, (T, H))
    rstd = rng.uniform(0.5, 1.5, size=T).astype(np.float32)
    a = oracle.dw_cols(T, 1, H, oracle.View.contiguous(dy), oracle.View.contiguous(x), rstd)
    b = oracle.dw_cols(T, 1, H, oracle.View.contiguous(dy), oracle.View.contiguous(x), 2 * rstd)
    np.testing.assert_array_equal(b, 2 * a)


# ------------------------------------------------- BF16 storage entry points

def test_bf16_entry_points_match_fp64_rows():
    rng = _rng(11)
    T, H = 7, 40
    x = _bf16_rows(rng, (T, H), 2.0)
    dy = _bf16_rows(rng, (T, H))
    w = _bf16_bits(torch.tensor(1 + 0.1 * rng.normal(size=H), dtype=torch.float32).to(torch.bfloat16))
    xv, dyv, wv = oracle.View.contiguous(x), oracle.View.contiguous(dy), w
    y, r64, hn = oracle.fwd_rows(T, 1, H, xv, wv, 1e-6)
    np.testing.assert_array_equal(hn, x)
    yf, rf = oracle.fwd_f64(oracle.bf16_bits_to_f64(x), oracle.bf16_bits_to_f64(w), 1e-6)
    np.testing.assert_array_equal(y, yf)
    np.testing.assert_array_equal(r64, rf)
    rk = r64.astype(np.float32)
    dx = oracle.bwd_rows(T, 1, H, dyv, xv, rk, wv)
    dxf, dwf = oracle.bwd_f64(oracle.bf16_bits_to_f64(dy), oracle.bf16_bits_to_f64(x), rk.astype(np.float64),
                              oracle.bf16_bits_to_f64(w))
    np.testing.assert_array_equal(dx, dxf)
    np.testing.assert_array_equal(oracle.dw_cols(T, 1, H, dyv, xv, rk), dwf)


def test_y_uses_kernel_rstd():
    rng = _rng(12)
    T, H = 4, 16
    x = _bf16_rows(rng, (T, H))
    w = (1 + 0.1 * rng.normal(size=H)).astype(np.float32)
    xv = oracle.View.contiguous(x)
    _, r64, _ = oracle.fwd_rows(T, 1, H, xv, w, 1e-6)
    rk = (r64 * 1.5).astype(np.float32)
    y, _, _ = oracle.fwd_rows(T, 1, H, xv, w, 1e-6, rstd_in=rk)
    expect = oracle.bf16_bits_to_f64(x) * rk.astype(np.float64)[:, None] * w.astype(np.float64)[None, :]
    np.testing.assert_allclose(y, expect, rtol=1e-15)


def test_row_and_column_subsets():
    rng = _rng(13)
    T, H = 9, 24
    x, dy = _bf16_rows(rng, (T, H)), _bf16_rows(rng, (T, H))
    w = (1 + 0.1 * rng.normal(size=H)).astype(np.float32)
    xv, dyv = oracle.View.contiguous(x), oracle.View.contiguous(dy)
    y, r64, hn = oracle.fwd_rows(T, 1, H, xv, w, 1e-6)
    rows = [8, 0, 5]
    ys, rs, hs = oracle.fwd_rows(T, 1, H, xv, w, 1e-6, rows=rows)
    np.testing.assert_array_equal(ys, y[rows])
    np.testing.assert_array_equal(rs, r64[rows])
    rk = r64.astype(np.float32)
    dx = oracle.bwd_rows(T, 1, H, dyv, xv, rk, w)
    np.testing.assert_array_equal(oracle.bwd_rows(T, 1, H, dyv, xv, rk, w, rows=rows), dx[rows])
    dw = oracle.dw_cols(T, 1, H, dyv, xv, rk)
    cols = [23, 1, 7]
    np.testing.assert_array_equal(oracle.dw_cols(T, 1, H, dyv, xv, rk, cols=cols), dw[cols])


def test_per_head_strided_equals_gathered():
    rng = _rng(14)
    T, nh, D = 5, 3, 16
    buf = _bf16_rows(rng, (T, nh, 2 * D), 2.0)  # [T, nh, 2D] buffer; the view is [..., :D]
    dy = _bf16_rows(rng, (T, nh, D))
    w = (1 + 0.1 * rng.normal(size=D)).astype(np.float32)
    strided = oracle.View(buf.reshape(-1), nh * 2 * D, 2 * D)
    gathered = np.ascontiguousarray(buf[:, :, :D]).reshape(T * nh, D)
    gv = oracle.View.contiguous(gathered)
    dyv = oracle.View.contiguous(dy)
    dyg = oracle.View.contiguous(dy.reshape(T * nh, D))
    y1, r1, h1 = oracle.fwd_rows(T, nh, D, strided, w, 1e-6)
    y2, r2, h2 = oracle.fwd_rows(T * nh, 1, D, gv, w, 1e-6)
    np.testing.assert_array_equal(y1, y2)
    np.testing.assert_array_equal(r1, r2)
    np.testing.assert_array_equal(h1, h2)
    rk = r1.astype(np.float32)
    np.testing.assert_array_equal(oracle.bwd_rows(T, nh, D, dyv, strided, rk, w),
                                  oracle.bwd_rows(T * nh, 1, D, dyg, gv, rk, w))
    np.testing.assert_array_equal(oracle.dw_cols(T, nh, D, dyv, strided, rk),
                                  oracle.dw_cols(T * nh, 1, D, dyg, gv, rk))


# --------------------------------------------------------------- residual route

def test_residual_sum_matches_torch_and_zero_residual_is_plain():
    rng = _rng(15)
    T, H = 6, 32
    xt = torch.tensor(rng.normal(size=(T, H)) * 4, dtype=torch.float32).to(torch.bfloat16)
    rt = torch.tensor(rng.normal(size=(T, H)) * 0.5, dtype=torch.float32).to(torch.bfloat16)
    x, res = _bf16_bits(xt), _bf16_bits(rt)
    w = (1 + 0.1 * rng.normal(size=H)).astype(np.float32)
    xv, rv = oracle.View.contiguous(x), oracle.View.contiguous(res)
    y, r64, hn = oracle.fwd_rows(T, 1, H, xv, w, 1e-6, residual=rv)
    # torch adds two BF16 tensors in FP32 and rounds once; with 8-bit
    # significands that equals the correctly rounded sum.
    np.testing.assert_array_equal(hn, _bf16_bits(xt + rt))
    y2, r2, _ = oracle.fwd_rows(T, 1, H, oracle.View.contiguous(hn), w, 1e-6)
    np.testing.assert_array_equal(y, y2)
    np.testing.assert_array_equal(r64, r2)
    zero = oracle.View.contiguous(np.zeros((T, H), dtype=np.uint16))
    y3, r3, h3 = oracle.fwd_rows(T, 1, H, xv, w, 1e-6, residual=zero)
    np.testing.assert_array_equal(h3, x)
    y4, r4, _ = oracle.fwd_rows(T, 1, H, xv, w, 1e-6)
    np.testing.assert_array_equal(y3, y4)


def test_residual_gradient_adds_dh():
    rng = _rng(16)
    T, H = 5, 16
    h, dy, dh = _bf16_rows(rng, (T, H)), _bf16_rows(rng, (T, H)), _bf16_rows(rng, (T, H))
    w = (1 + 0.1 * rng.normal(size=H)).astype(np.float32)
    rk = rng.uniform(0.5, 1.5, size=T).astype(np.float32)
    hv, dyv, dhv = oracle.View.contiguous(h), oracle.View.contiguous(dy), oracle.View.contiguous(dh)
    a = oracle.bwd_rows(T, 1, H, dyv, hv, rk, w)
    b = oracle.bwd_rows(T, 1, H, dyv, hv, rk, w, dh=dhv)
    np.testing.assert_allclose(b - a, oracle.bf16_bits_to_f64(dh), rtol=0, atol=1e-15 * (1 + np.abs(a).max()))


# ------------------------------------------------------------------ BF16 rounding

def test_bf16_round_matches_torch_cast():
    rng = _rng(17)
    vals = np.concatenate([
        rng.normal(size=20000).astype(np.float32),
        (rng.normal(size=2000) * 1e-39).astype(np.float32),   # FP32 subnormals
        (rng.normal(size=2000) * 1e37).astype(np.float32),
        np.array([0.0, -0.0, 3.3895314e38, 3.3961776e38, -3.4e38, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8],
                 dtype=np.float32),
    ])
    ours = oracle.bf16_round(vals.astype(np.float64))
    theirs = _bf16_bits(torch.tensor(vals).to(torch.bfloat16))
    np.testing.assert_array_equal(ours, theirs)


def test_bf16_round_ties_and_double_rounding():
    one = 0x3F80
    # ties go to even: 1 + 2^-8 -> 1;  1 + 3*2^-8 -> 1 + 2^-6
    assert oracle.bf16_round(np.array([1 + 2 ** -8]))[0] == one
    assert oracle.bf16_round(np.array([1 + 3 * 2 ** -8]))[0] == one + 2
    # just above a tie by less than half an FP32 ulp: one correct rounding
    # goes up, whereas rounding to FP32 first would land on the tie and go down.
    assert oracle.bf16_round(np.array([1 + 2 ** -8 + 2 ** -40]))[0] == one + 1
    assert oracle.bf16_round(np.array([-(1 + 2 ** -8 + 2 ** -40)]))[0] == 0x8000 | (one + 1)
    # overflow past the largest finite BF16 plus half an ulp -> inf
    assert oracle.bf16_round(np.array([2.0 ** 128]))[0] == 0x7F80
    assert oracle.bf16_round(np.array([-1e300]))[0] == 0xFF80

