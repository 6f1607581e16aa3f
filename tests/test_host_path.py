"""The backward from and to host memory (cake_rmsnorm_bwd_host).

The rows live in host memory and go to the device in chunks whose copies in,
main kernels and copies out overlap; one fixed-order reduce over every
chunk's partials gives dw.  These checks hold it to the FP64 oracle with the
parity bars (dx within one BF16 step of RNE_bf16(dx64) with the FP32
allowance near cancellation; dw within 1e-4 + 1e-4 |dw64|), and check that
its dx is the same bits as the device entry point's, that dw is bitwise
reproducible for a given chunk count, that pageable host memory gives the
same results as page-locked memory, and the edge cases: one chunk, more
chunks than rows, the residual route with dh, a per-head view passed as its
rows, and T = 0.
"""
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


def _run_host(cake, dy, h, rin, w, dh, chunks, pinned=True):
    T = h.shape[0]
    nh = h.shape[1] if h.dim() == 3 else 1
    H = h.shape[-1]
    pin = (lambda t: t.contiguous().pin_memory()) if pinned else (lambda t: t.contiguous().clone())
    hx, hdy, hr, hw = pin(h), pin(dy), pin(torch.from_numpy(rin)), pin(w)
    hdh = pin(dh) if dh is not None else None
    dx = torch.empty(h.shape, dtype=torch.bfloat16)
    dw = torch.empty(H, dtype=torch.float32)
    if pinned:
        dx, dw = dx.pin_memory(), dw.pin_memory()
    n = cake.cake_rmsnorm_bwd_host_staging_size((T, nh, H), w.dtype, has_dh=dh is not None, chunks=chunks)
    staging = torch.empty(max(n, 256), dtype=torch.uint8, device=DEV)
    dx.fill_(7.0)
    dw.fill_(float("nan"))
    cake.cake_rmsnorm_bwd_host(hdy, hx, hr, hw, hdh, dx=dx, dw=dw, staging=staging, chunks=chunks)
    torch.cuda.current_stream().synchronize()
    return dx, dw


CASES = [
    ("plain_w32", lambda: cake_inputs.plain_case(1000, 2048, family="outlier", w_dtype=torch.float32, seed=51), (1, 3, 8)),
    ("bf16w_odd", lambda: cake_inputs.plain_case(777, 1536, w_dtype=torch.bfloat16, seed=52), (5, 64)),
    ("few_rows", lambda: cake_inputs.plain_case(5, 4096, w_dtype=torch.bfloat16, seed=53), (8,)),
    ("residual_dh", lambda: cake_inputs.residual_case(300, 6144, seed=54), (4,)),
    ("heads_rows", lambda: cake_inputs.heads_case(40, 24, strided=False, w_dtype=torch.float32, seed=55), (6,)),
]


@pytest.mark.parametrize("name,make,chunk_list", CASES, ids=[c[0] for c in CASES])
def test_host_path_against_the_oracle(cake, name, make, chunk_list):
    c = make()
    x, dy, w, res, dh = c["x"], c["dy"], c["w"], c.get("residual"), c.get("dh")
    T = x.shape[0]
    nh = x.shape[1] if x.dim() == 3 else 1
    H = x.shape[-1]
    rin, hn = oracle_bwd_inputs(x, w, c["eps"], res)
    h = torch.from_numpy(hn.view(np.int16)).view(torch.bfloat16).reshape(x.shape) if res is not None else x
    hv, dyv = view_of(h), view_of(dy)
    dhv = view_of(dh) if dh is not None else None
    dx64 = oracle.bwd_rows(T, nh, H, dyv, hv, rin, wbits(w), dh=dhv)
    dw64 = oracle.dw_cols(T, nh, H, dyv, hv, rin)
    ref_dx, _ = cake.cake_rmsnorm_bwd(dy.to(DEV), h.to(DEV), torch.from_numpy(rin).to(DEV), w.to(DEV),
                                      dh.to(DEV) if dh is not None else None)
    torch.cuda.synchronize()
    ref_bits = bits(ref_dx).reshape(-1, H)
    for chunks in chunk_list:
        runs = [_run_host(cake, dy, h, rin, w, dh, chunks) for _ in range(2)]
        runs.append(_run_host(cake, dy, h, rin, w, dh, chunks, pinned=False))
        dxb = bits(runs[0][0]).reshape(-1, H)
        rep = tol.dx_report(dxb, dx64, rows_f64(dy), rows_f64(h), w64(w), rin, oracle.bf16_round,
                            oracle.bf16_bits_to_f64, dh=rows_f64(dh) if dh is not None else None)
        assert rep["bounded"] == 0 and rep["off_cancellation"] == 0, (chunks, rep)
        np.testing.assert_array_equal(dxb, ref_bits)  # dx: the device entry point's bits
        frac = float(tol.dw_budget_fraction(runs[0][1].numpy(), dw64).max())
        assert frac <= 1.0, (chunks, frac)
        for dxr, dwr in runs[1:]:  # reproducible, pinned or pageable
            assert torch.equal(dxr, runs[0][0]) and torch.equal(dwr, runs[0][1])


def test_host_path_empty(cake):
    x = torch.empty((0, 512), dtype=torch.bfloat16)
    dw = torch.full((512,), 3.0)
    staging = torch.empty(256, dtype=torch.uint8, device=DEV)
    cake.cake_rmsnorm_bwd_host(x, x, torch.empty(0), torch.ones(512), dx=torch.empty_like(x), dw=dw,
                               staging=staging)
    assert not dw.any()
