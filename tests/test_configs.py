"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times (the default window table, both backward modes).

* T=256, H=1536 plain, BF16 weight: every output against the oracle.
* T=65536, H=2048, outlier family, dy ~ N(0, 1e-2), FP32 weight: rstd, dx and
  dw of every row and column; y of sampled rows.
* T=131072, H=6144 with the fused residual: rstd and h_new of every row
  (h_new bitwise), dw of every column, y and dx of sampled rows (the oracle
  computes them one row at a time).
* Per-head views at T=32768 ([T,24,256] strided slice of [T,24,512], and
  contiguous [T,4,256]): every row and column.
* The accuracy sweep's widths H=4096 and H=5120 at T=65536: rstd of every
  row, dw of every column, y and dx of sampled rows.

Inputs are drawn on the device from seeded generators and copied to the host
for the oracle.  The backward's rstd (and on the residual route its h_new)
are the oracle's, so no oracle input comes from the CUDA path.
"""
import numpy as np
import pytest
import torch

import cake_inputs
import oracle
from tests import report
from tests import tolerances as tol

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(scope="module")
def cake():
    import __graft_entry__
    __graft_entry__.build()
    import bwd_dw_column_gb300 as cake
    yield cake
    assert cake.cake_rmsnorm_device_status() == 0


def bits(t):
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def host_view(t):
    """Oracle view of a device BF16 tensor (strided views keep their strides)."""
    if t.dim() == 3 and not t.is_contiguous():
        flat = t.as_strided((t.untyped_storage().nbytes() // 2,), (1,), 0)
        return oracle.View(bits(flat), t.stride(0), t.stride(1), t.storage_offset())
    return oracle.View.contiguous(bits(t))


def wbits(w):
    w = w.cpu()
    return w.numpy() if w.dtype == torch.float32 else bits(w)


def sample_rows(R, n=48, seed=0):
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, 1, R - 2, R - 1], rng.integers(0, R, size=n)]))
    return rows[(rows >= 0) & (rows < R)]


def check_dx(dx_bits_rows, dx64, dyv_rows, hv_rows, w64, rin_rows, dh_rows=None):
    rep = tol.dx_report(dx_bits_rows, dx64, dyv_rows, hv_rows, w64, rin_rows, oracle.bf16_round,
                        oracle.bf16_bits_to_f64, dh=dh_rows)
    assert rep["bounded"] == 0 and rep["off_cancellation"] == 0, f"dx: {rep}"
    return rep


def rows_of(view: oracle.View, rows, nh, H):
    """FP64 values of the listed rows of a view (host side, vectorised)."""
    T = (len(view.buf) - view.offset - H) // view.st + 1 if view.st else 1
    base = view.buf[view.offset:]
    a = np.lib.stride_tricks.as_strided(base, shape=(T, nh, H), strides=(2 * view.st, 2 * view.sh, 2),
                                        writeable=False)
    rows = np.asarray(rows)
    return oracle.bf16_bits_to_f64(a[rows // nh, rows % nh])


def run_workload(cake, x, dy, w, eps, residual=None, dh=None, full_dx=True, sampled=None, name=None):
    T = x.shape[0]
    nh = x.shape[1] if x.dim() == 3 else 1
    H = x.shape[-1]
    R = T * nh
    xv = host_view(x)
    rv = host_view(residual) if residual is not None else None
    wb = wbits(w)
    # forward: the kernel against the oracle
    out = cake.cake_rmsnorm_fwd(x, w, eps, residual=residual)
    torch.cuda.synchronize()
    _, r64, hn = oracle.fwd_rows(T, nh, H, xv, wb, eps, residual=rv, want_y=False, want_h=residual is not None)
    rk = out[1].cpu().numpy().astype(np.float64)
    assert np.all(np.abs(rk / r64 - 1) <= tol.RSTD_REL)
    rows = sample_rows(R) if sampled is None else sampled
    y64, _, _ = oracle.fwd_rows(T, nh, H, xv, wb, eps, residual=rv, rows=rows, want_h=False)
    yk = bits(out[0]).reshape(R, H)[rows]
    assert tol.ulp_distance(yk, oracle.bf16_round(y64)).max() <= 1
    if residual is not None:
        np.testing.assert_array_equal(bits(out[2]).reshape(R, H), hn.reshape(R, H))
    del out
    # backward at the oracle's rstd (and h_new)
    rin = r64.astype(np.float32)
    if residual is not None:
        h_d = torch.from_numpy(hn.view(np.int16)).view(torch.bfloat16).reshape(x.shape).to(DEV)
        hv = oracle.View.contiguous(hn.reshape(R, H))
    else:
        h_d, hv = x, xv
    dyv = host_view(dy)
    dhv = host_view(dh) if dh is not None else None
    r_d = torch.from_numpy(rin).to(DEV)
    dw64 = oracle.dw_cols(T, nh, H, dyv, hv, rin)
    dx_rows = np.arange(R) if full_dx else rows
    dx64 = oracle.bwd_rows(T, nh, H, dyv, hv, rin, wb, dh=dhv, rows=None if full_dx else dx_rows)
    dyf, hf = rows_of(dyv, dx_rows, nh, H), rows_of(hv, dx_rows, nh, H)
    dhf = rows_of(dhv, dx_rows, nh, H) if dh is not None else None
    w64 = w.double().cpu().numpy()
    dx_bits = None
    dx_rep = None
    worst = {}
    for det in (True, False):
        dws = []
        for _ in range(2):
            dx, dw = cake.cake_rmsnorm_bwd(dy, h_d, r_d, w, dh, deterministic=det)
            torch.cuda.synchronize()
            dws.append(dw.cpu().numpy())
            b = bits(dx).reshape(R, H)
            if dx_bits is None:
                dx_bits = b
                dx_rep = check_dx(b[dx_rows], dx64, dyf, hf, w64, rin[dx_rows], dhf)
            else:
                assert np.array_equal(b, dx_bits)  # dx: same bits in both modes and calls
            del dx
        if det:
            np.testing.assert_array_equal(dws[0], dws[1])
        frac = max(float(tol.dw_budget_fraction(d, dw64).max()) for d in dws)
        assert frac <= 1.0, frac
        worst["det" if det else "nondet"] = frac
    what = name or f"T={T} nh={nh} H={H}"
    rows_note = "every row" if full_dx else f"{len(dx_rows)} sampled rows"
    report.record(f"full size {what}: dx of {rows_note}, dw of every column", dx=dx_rep,
                  dw_worst=max(worst.values()), dw_det=worst["det"], dw_nondet=worst["nondet"])
    return worst


def test_h1536_t256(cake):
    c = cake_inputs.make("h1536_t256", seed=0, device=DEV)
    run_workload(cake, c["x"], c["dy"], c["w"], c["eps"], name="h1536_t256")


def test_h2048_t65536_outlier_w32(cake):
    c = cake_inputs.make("h2048_t65536_outlier_w32", seed=0, device=DEV)
    run_workload(cake, c["x"], c["dy"], c["w"], c["eps"], name="h2048_t65536_outlier_w32")


def test_h6144_t131072_residual(cake):
    c = cake_inputs.make("h6144_t131072_res", seed=0, device=DEV)
    run_workload(cake, c["x"], c["dy"], c["w"], c["eps"], residual=c["residual"], dh=c["dh"], full_dx=False,
                 name="h6144_t131072_res")


@pytest.mark.parametrize("name", ["heads24_t32768_strided", "heads4_t32768"])
def test_per_head(cake, name):
    c = cake_inputs.make(name, seed=0, device=DEV)
    run_workload(cake, c["x"], c["dy"], c["w"], c["eps"], name=name)


@pytest.mark.parametrize("name", ["h4096_t65536_sweep", "h5120_t65536_sweep", "h4096_t44032_sweep",
                                  "h5120_t131072_sweep", "h4096_t131072_sweep"])
def test_sweep_widths(cake, name):
    # the accuracy sweep's widths at its large T: 32 columns per thread (H =
    # 4096) and 24 (H = 5120); dx of sampled rows, dw of every column
    c = cake_inputs.make(name, seed=0, device=DEV)
    run_workload(cake, c["x"], c["dy"], c["w"], c["eps"], full_dx=False, name=name)


@pytest.mark.parametrize("T,H", [(131072, 64), (65536, 128), (65536, 200), (65536, 384), (32768, 640), (32768, 832)])
def test_narrow_row_layouts_at_size(cake, T, H):
    # rows of a quarter of a warp (H = 64), of half a warp (H = 128 at 8
    # columns per thread; H = 200 at 16, part of each thread's second vector
    # idle) and of one warp at 16, 24 and 32 columns per thread, at tens of
    # thousands of rows: dx of every row, dw of every column, both modes
    c = cake_inputs.plain_case(T, H, family="outlier", w_dtype=torch.float32, seed=T + H, device=DEV)
    run_workload(cake, c["x"], c["dy"], c["w"], c["eps"], name=f"T={T} H={H} outlier, w FP32")


@pytest.mark.parametrize("T,H", [(65536, 2048), (32768, 4096), (20000, 512)])
def test_single_kernel_forms_at_size(cake, T, H):
    """Every one-kernel form -- FP64 atomics, the tree, the cooperative grid
    and the cluster form -- at tens of thousands of rows, with the table's
    accumulation: dw of every column against the oracle, dx the same bits as
    the pair's (forms the layout does not offer are skipped)."""
    c = cake_inputs.plain_case(T, H, family="outlier", w_dtype=torch.float32, seed=T + H, device=DEV)
    x, dy, w = c["x"], c["dy"], c["w"]
    xv, dyv = host_view(x), host_view(dy)
    _, r64, _ = oracle.fwd_rows(T, 1, H, xv, wbits(w), c["eps"], want_y=False, want_h=False)
    rin = r64.astype(np.float32)
    dw64 = oracle.dw_cols(T, 1, H, dyv, xv, rin)
    r_d = torch.from_numpy(rin).to(DEV)
    ws = cake.cake_rmsnorm_bwd_workspace(x, w.dtype, deterministic=False)
    ref_dx, _ = cake.cake_rmsnorm_bwd(dy, x, r_d, w, deterministic=True, workspace=ws)
    torch.cuda.synchronize()
    ref_bits = bits(ref_dx)
    worst = {}
    for form in (1, 2, 3, 4):
        try:
            dx, dw = cake.cake_rmsnorm_bwd_forced(dy, x, r_d, w, deterministic=form != 1, force_single=form,
                                                  workspace=ws)
        except cake.CakeError as e:
            assert form == 2 and e.status == 2  # the tree form needs 8 columns per thread
            continue
        torch.cuda.synchronize()
        assert np.array_equal(bits(dx), ref_bits)
        worst[form] = float(tol.dw_budget_fraction(dw.cpu().numpy(), dw64).max())
        assert worst[form] <= 1.0, worst
        del dx, dw
    report.record(f"one-kernel forms T={T} H={H}", dw_worst=max(worst.values()),
                  **{f"form{k}": round(v, 4) for k, v in worst.items()})
