"""The training facade (autograd function and the pages' Python names).

GPU tests hold one autograd run per route to the FP64 oracle -- plain rows
with an FP32 and a BF16 weight, the residual route with a gradient into h_new
(x.grad and residual.grad are both the one dx), and a strided per-head view --
with the parity bars: dx within one BF16 step of RNE_bf16(dx64), an FP32
w.grad within the dw budget, a BF16 w.grad within the dw budget plus the
half BF16 step of its own rounding.  The oracle takes its own rstd rounded to FP32, as in the
parity tests.  Further GPU tests check that autograd gives exactly the bits
of the C ABI entry points, in both modes; that a checkpointed step (forward,
forward recompute, backward) gives the same gradient bits as the plain step;
and that the cached workspace is reused, not reallocated.  The CPU tests
check the names and that CPU tensors are rejected (there is no CPU path).
"""
import numpy as np
import pytest
import torch
import torch.utils.checkpoint as ckpt

import cake_inputs
import oracle
from tests import tolerances as tol

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None

NAMES = ["CakeRMSNormFunction", "cake_rmsnorm", "cake_rmsnorm_train_forward", "cake_rmsnorm_train_backward",
         "cake_rmsnorm_train_backward_workspace_bytes", "cake_rmsnorm_train_backward_workspace"]


@pytest.fixture(scope="module")
def cake():
    import __graft_entry__
    __graft_entry__.build()
    import bwd_dw_column_gb300 as cake
    yield cake


def test_facade_names(cake):
    for n in NAMES:
        assert n in cake.__all__ and callable(getattr(cake, n))


def test_facade_rejects_cpu_tensors(cake):
    c = cake_inputs.plain_case(4, 64, seed=1)
    x = c["x"].clone().requires_grad_()
    with pytest.raises(ValueError):
        cake.cake_rmsnorm(x, c["w"])
    with pytest.raises(ValueError):
        cake.cake_rmsnorm_train_backward(c["dy"], c["x"], torch.ones(4), c["w"])


def _leaf(t):
    return t.to(DEV).detach().requires_grad_()


def _leaf_view(t):
    """A leaf that is a strided view (keeps the [T, nh, H] strides of t)."""
    flat = t.as_strided((t.untyped_storage().nbytes() // t.element_size(),), (1,), 0).to(DEV)
    base = flat.detach().requires_grad_()
    return base, base.as_strided(t.shape, t.stride(), t.storage_offset())


@pytest.mark.gpu
@pytest.mark.parametrize("T,H,w_dtype", [(300, 2048, torch.float32), (77, 1536, torch.bfloat16), (5, 6144, torch.float32)])
@pytest.mark.parametrize("det", [True, False])
def test_autograd_plain_matches_entry_points(cake, T, H, w_dtype, det):
    c = cake_inputs.plain_case(T, H, w_dtype=w_dtype, seed=T + H)
    x, w, dy = _leaf(c["x"]), _leaf(c["w"]), c["dy"].to(DEV)
    y = cake.cake_rmsnorm(x, w, c["eps"], deterministic=det)
    y.backward(dy)
    y2, rstd = cake.cake_rmsnorm_train_forward(x.detach(), w.detach(), c["eps"])
    dx, dw = cake.cake_rmsnorm_train_backward(dy, x.detach(), rstd, w.detach(), deterministic=det)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
    assert torch.equal(x.grad, dx)
    assert w.grad.dtype == w_dtype
    assert torch.equal(w.grad, dw if w_dtype == torch.float32 else dw.to(w_dtype))


@pytest.mark.gpu
@pytest.mark.parametrize("with_dh", [True, False])
def test_autograd_residual_matches_entry_points(cake, with_dh):
    c = cake_inputs.residual_case(129, 6144, seed=7)
    x, res, w = _leaf(c["x"]), _leaf(c["residual"]), _leaf(c["w"])
    dy, dh = c["dy"].to(DEV), c["dh"].to(DEV)
    y, h_new = cake.cake_rmsnorm(x, w, c["eps"], residual=res)
    if with_dh:
        torch.autograd.backward([y, h_new], [dy, dh])
    else:
        y.backward(dy)
    y2, rstd, hn2 = cake.cake_rmsnorm_train_forward(x.detach(), w.detach(), c["eps"], residual=res.detach())
    dx, dw = cake.cake_rmsnorm_train_backward(dy, hn2, rstd, w.detach(), dh if with_dh else None)
    torch.cuda.synchronize()
    assert torch.equal(y, y2) and torch.equal(h_new, hn2)
    assert torch.equal(x.grad, dx) and torch.equal(res.grad, dx)
    assert torch.equal(w.grad, dw.to(w.dtype))


@pytest.mark.gpu
def test_autograd_per_head_view(cake):
    c = cake_inputs.heads_case(64, 24, strided=True, seed=5)
    base, x = _leaf_view(c["x"])
    w, dy = _leaf(c["w"]), c["dy"].to(DEV)
    assert x.stride() == c["x"].stride()
    y = cake.cake_rmsnorm(x, w, c["eps"])
    y.backward(dy)
    xd = x.detach()
    _, rstd = cake.cake_rmsnorm_train_forward(xd, w.detach(), c["eps"])
    dx, dw = cake.cake_rmsnorm_train_backward(dy, xd, rstd, w.detach())
    torch.cuda.synchronize()
    # the gradient lands in the strided rows of the base buffer; the gaps stay zero
    g = base.grad.as_strided(x.shape, x.stride(), x.storage_offset())
    assert torch.equal(g, dx)
    gaps = base.grad.clone()
    gaps.as_strided(x.shape, x.stride(), x.storage_offset()).zero_()
    assert not gaps.any()
    assert torch.equal(w.grad, dw)


@pytest.mark.gpu
@pytest.mark.parametrize("det", [True, False])
def test_checkpointed_step_is_bitwise(cake, det):
    """forward, forward recompute, backward: the same gradient bits as forward + backward."""
    c = cake_inputs.residual_case(256, 2048, w_dtype=torch.float32, seed=11)
    calls = {"n": 0}

    def block(x, res, w):
        calls["n"] += 1
        y, h_new = cake.cake_rmsnorm(x, w, c["eps"], residual=res, deterministic=det)
        return (y.float() * 0.5).to(torch.bfloat16), h_new

    def run(checkpointed):
        x, res, w = _leaf(c["x"]), _leaf(c["residual"]), _leaf(c["w"])
        if checkpointed:
            out, h_new = ckpt.checkpoint(block, x, res, w, use_reentrant=False)
        else:
            out, h_new = block(x, res, w)
        torch.autograd.backward([out, h_new], [c["dy"].to(DEV), c["dh"].to(DEV)])
        torch.cuda.synchronize()
        return out.detach(), x.grad, res.grad, w.grad

    plain = run(False)
    n_plain = calls["n"]
    again = run(True)
    assert calls["n"] - n_plain == 2  # the checkpointed step ran the forward twice
    for a, b in zip(plain, again):
        assert torch.equal(a, b)


@pytest.mark.gpu
def test_caller_workspace(cake):
    c = cake_inputs.plain_case(1000, 4096, w_dtype=torch.float32, seed=2)
    ws = cake.cake_rmsnorm_train_backward_workspace(c["x"].to(DEV), torch.float32, deterministic=True)
    assert ws.numel() >= cake.cake_rmsnorm_train_backward_workspace_bytes(c["x"].to(DEV), torch.float32, True)
    grads = []
    for workspace in (ws, None):
        x, w = _leaf(c["x"]), _leaf(c["w"])
        cake.cake_rmsnorm(x, w, c["eps"], workspace=workspace).backward(c["dy"].to(DEV))
        grads.append((x.grad, w.grad))
    torch.cuda.synchronize()
    assert torch.equal(grads[0][0], grads[1][0]) and torch.equal(grads[0][1], grads[1][1])


def _host_bits(t):
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _oracle_grads(x, w, dy, eps, residual=None, dh=None):
    """(dx64, dw64, rin, h rows, dy rows, dh rows) from the FP64 oracle for a
    CPU case; rin is the oracle's rstd rounded to FP32."""
    from tests.test_parity import oracle_bwd_inputs, rows_f64, view_of, wbits
    T = x.shape[0]
    nh = x.shape[1] if x.dim() == 3 else 1
    H = x.shape[-1]
    rin, hn = oracle_bwd_inputs(x, w, eps, residual)
    h = torch.from_numpy(hn.view(np.int16)).view(torch.bfloat16).reshape(x.shape) if residual is not None else x
    hv, dyv = view_of(h), view_of(dy)
    dhv = view_of(dh) if dh is not None else None
    dx64 = oracle.bwd_rows(T, nh, H, dyv, hv, rin, wbits(w), dh=dhv)
    dw64 = oracle.dw_cols(T, nh, H, dyv, hv, rin)
    return dx64, dw64, rin, rows_f64(h), rows_f64(dy), (rows_f64(dh) if dh is not None else None)


def _check_grads(xgrad, wgrad, w, dx64, dw64, rin, hf, dyf, dhf):
    H = w.numel()
    rep = tol.dx_report(_host_bits(xgrad).reshape(-1, H), dx64, dyf, hf, w.double().numpy(), rin,
                        oracle.bf16_round, oracle.bf16_bits_to_f64, dh=dhf)
    assert rep["bounded"] == 0 and rep["off_cancellation"] == 0, rep
    assert wgrad.dtype == w.dtype
    if w.dtype == torch.float32:
        assert float(tol.dw_budget_fraction(wgrad.cpu().numpy(), dw64).max()) <= 1.0
    else:
        # the FP32 dw within its budget, then rounded once to BF16
        g = oracle.bf16_bits_to_f64(_host_bits(wgrad))
        allow = tol.DW_ATOL + tol.DW_RTOL * np.abs(dw64) + tol.bf16_ulp(dw64) / 2
        assert np.all(np.abs(g - dw64) <= allow)


@pytest.mark.gpu
@pytest.mark.parametrize("w_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("det", [True, False])
def test_autograd_plain_against_oracle(cake, w_dtype, det):
    c = cake_inputs.plain_case(257, 2048, w_dtype=w_dtype, seed=41)
    dx64, dw64, rin, hf, dyf, _ = _oracle_grads(c["x"], c["w"], c["dy"], c["eps"])
    x, w = _leaf(c["x"]), _leaf(c["w"])
    cake.cake_rmsnorm(x, w, c["eps"], deterministic=det).backward(c["dy"].to(DEV))
    torch.cuda.synchronize()
    _check_grads(x.grad, w.grad, c["w"], dx64, dw64, rin, hf, dyf, None)


@pytest.mark.gpu
def test_autograd_residual_against_oracle(cake):
    c = cake_inputs.residual_case(129, 6144, seed=42)
    dx64, dw64, rin, hf, dyf, dhf = _oracle_grads(c["x"], c["w"], c["dy"], c["eps"], c["residual"], c["dh"])
    x, res, w = _leaf(c["x"]), _leaf(c["residual"]), _leaf(c["w"])
    y, h_new = cake.cake_rmsnorm(x, w, c["eps"], residual=res)
    torch.autograd.backward([y, h_new], [c["dy"].to(DEV), c["dh"].to(DEV)])
    torch.cuda.synchronize()
    _check_grads(x.grad, w.grad, c["w"], dx64, dw64, rin, hf, dyf, dhf)
    assert torch.equal(res.grad, x.grad)  # one dx is the gradient of both


@pytest.mark.gpu
def test_autograd_per_head_against_oracle(cake):
    c = cake_inputs.heads_case(48, 24, strided=True, seed=43)
    dx64, dw64, rin, hf, dyf, _ = _oracle_grads(c["x"], c["w"], c["dy"], c["eps"])
    base, x = _leaf_view(c["x"])
    w = _leaf(c["w"])
    cake.cake_rmsnorm(x, w, c["eps"]).backward(c["dy"].to(DEV))
    torch.cuda.synchronize()
    g = base.grad.as_strided(x.shape, x.stride(), x.storage_offset())
    _check_grads(g, w.grad, c["w"], dx64, dw64, rin, hf, dyf, None)


@pytest.mark.gpu
def test_backward_reuses_the_cached_workspace(cake):
    from bwd_dw_column_gb300 import train
    c = cake_inputs.plain_case(300, 1536, seed=44)
    stream_key = (0, torch.cuda.current_stream().cuda_stream)
    seen = []
    for _ in range(3):
        x, w = _leaf(c["x"]), _leaf(c["w"])
        cake.cake_rmsnorm(x, w, c["eps"]).backward(c["dy"].to(DEV))
        seen.append(train._ws_cache[stream_key].data_ptr())
    torch.cuda.synchronize()
    assert len(set(seen)) == 1
