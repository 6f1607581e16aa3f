"""The training facade (autograd function and the pages' Python names).

GPU tests check that autograd reaches exactly the results of the C ABI entry
points, which the parity tests pin to the oracle: dx and dw bitwise, on the
plain, residual and per-head routes, in both modes; and that a checkpointed
step (forward, forward recompute, backward) gives the same gradient bits as
the plain step.  The CPU tests check the names and that CPU tensors are
rejected (there is no CPU path).
"""
import pytest
import torch
import torch.utils.checkpoint as ckpt

import cake_inputs

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
