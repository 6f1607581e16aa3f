"""The kernels' timeout path, made to run out from the host.

Every wait in the kernels is bounded: a wait that runs out records
CAKE_ERR_TIMEOUT in the device status word, and the kernel returns instead of
hanging.  cake_rmsnorm_bwd_timeout_test launches the cooperative grid form
with its grid barrier expecting one arrival more than there are CTAs (an
arrival that never comes) and a short wait limit.  The checks: the call ends
by itself within a second, the device status reads CAKE_ERR_TIMEOUT (and is
cleared by reading it), the barrier counter holds every CTA's arrival and its
generation did not move, dx is still correct, and after the workspace is
re-initialised the same form and the default backward pass parity against
the oracle again.  Nothing here faults or hangs the GPU: the wait gives up by
its own limit.
"""
import time

import numpy as np
import pytest
import torch

import cake_inputs
import oracle
from tests import tolerances as tol
from tests.test_parity import DEV, bits, oracle_bwd_inputs, rows_f64, view_of, w64, wbits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cake():
    import __graft_entry__
    __graft_entry__.build()
    import bwd_dw_column_gb300 as cake
    yield cake
    assert cake.cake_rmsnorm_device_status() == 0


def test_grid_barrier_wait_runs_out_and_recovers(cake):
    T, H = 900, 1536
    c = cake_inputs.plain_case(T, H, w_dtype=torch.float32, seed=31)
    x, dy, w = c["x"], c["dy"], c["w"]
    rin, _ = oracle_bwd_inputs(x, w, c["eps"])
    xv, dyv = view_of(x), view_of(dy)
    dx64 = oracle.bwd_rows(T, 1, H, dyv, xv, rin, wbits(w))
    dw64 = oracle.dw_cols(T, 1, H, dyv, xv, rin)
    x_d, dy_d, w_d, r_d = x.to(DEV), dy.to(DEV), w.to(DEV), torch.from_numpy(rin).to(DEV)
    ws = cake.cake_rmsnorm_bwd_workspace(x_d, w.dtype, deterministic=True)
    ctas = cake.cake_rmsnorm_bwd_select((T, 1, H), w.dtype, deterministic=True, force_single=3)["ctas"]
    dx = torch.empty_like(x_d)
    dw = torch.full((H,), 7.0, device=DEV)

    assert cake.cake_rmsnorm_device_status(clear=True) == 0
    t0 = time.perf_counter()
    try:
        cake.cake_rmsnorm_bwd_timeout_test(dy_d, x_d, r_d, w_d, workspace=ws, dx=dx, dw=dw, wait_limit_us=2000)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
        status = cake.cake_rmsnorm_device_status(clear=True)
    finally:
        cake.cake_rmsnorm_device_status(clear=True)
    assert status == cake.CAKE_ERR_TIMEOUT
    assert elapsed < 1.0, f"the timed-out launch took {elapsed:.3f} s"
    words = ws[:512].cpu().view(torch.int32)
    assert int(words[64]) == ctas and int(words[65]) == 0  # every CTA arrived; the generation never moved
    assert torch.all(dw == 7.0)  # the reduce after the barrier never ran
    # dx is computed before the barrier: it is complete and correct
    rep = tol.dx_report(bits(dx), dx64, rows_f64(dy), rows_f64(x), w64(w), rin, oracle.bf16_round,
                        oracle.bf16_bits_to_f64)
    assert rep["bounded"] == 0 and rep["off_cancellation"] == 0, rep

    # recovery: re-initialise the workspace, then the grid form and the default backward pass parity
    cake.cake_rmsnorm_bwd_workspace_init(ws)
    for force in (3, None):
        if force is None:
            dx2, dw2 = cake.cake_rmsnorm_bwd(dy_d, x_d, r_d, w_d, deterministic=True, workspace=ws)
        else:
            dx2, dw2 = cake.cake_rmsnorm_bwd_forced(dy_d, x_d, r_d, w_d, deterministic=True, force_single=force,
                                                    workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(dx2, dx)
        assert float(tol.dw_budget_fraction(dw2.cpu().numpy(), dw64).max()) <= 1.0
    words = ws[:512].cpu().view(torch.int32)
    assert int(words[64]) == 0 and int(words[65]) == 1
    assert cake.cake_rmsnorm_device_status() == 0


def test_timeout_test_rejects_a_bad_limit(cake):
    x = torch.zeros((4, 256), dtype=torch.bfloat16, device=DEV)
    w = torch.ones(256, device=DEV)
    ws = cake.cake_rmsnorm_bwd_workspace(x, w.dtype, deterministic=True)
    for limit in (0, 2_000_000):
        with pytest.raises(cake.CakeError) as e:
            cake.cake_rmsnorm_bwd_timeout_test(x, x, torch.ones(4, device=DEV), w, workspace=ws,
                                              dx=torch.empty_like(x), dw=torch.empty(256, device=DEV),
                                              wait_limit_us=limit)
        assert e.value.status == cake.CAKE_ERR_INVALID
