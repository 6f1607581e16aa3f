"""GPU parity: the CUDA path (through the C ABI) against the FP64 oracle,
element by element, on seeded synthetic inputs.

Bars (restated in tests/tolerances.py):
  y     within one BF16 step of RNE_bf16(y64);
  rstd  relative error <= 1e-6 against rstd64;
  h_new bitwise equal to the oracle's RNE_bf16(x + residual);
  dx    within one BF16 step of RNE_bf16(dx64) at the rstd the backward was
        given (with the documented FP32-evaluation allowance near
        cancellation; strict counts are reported as well);
  dw    per element |dw - dw64| <= 1e-4 + 1e-4 |dw64| (worst element
        reported as a fraction of that budget);
  determinism: dx bitwise identical across calls, modes and variants; dw
        bitwise identical across calls in deterministic mode.

The backward's rstd input is the oracle's rstd64 rounded to FP32 and, on the
residual route, its x input is the oracle's h_new: no oracle input ever comes
from the CUDA path.
"""
import math

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


def to_dev(t: torch.Tensor | None) -> torch.Tensor | None:
    """Copy to the GPU keeping a strided view strided (copy its whole storage)."""
    if t is None:
        return None
    if t.is_contiguous():
        return t.to(DEV)
    flat = t.as_strided((t.untyped_storage().nbytes() // t.element_size(),), (1,), 0)
    return flat.to(DEV).as_strided(t.shape, t.stride(), t.storage_offset())


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def view_of(t: torch.Tensor) -> oracle.View:
    """Oracle view of a (possibly strided) CPU BF16 tensor [T, H] or [T, nh, H]."""
    base = t
    if t.dim() == 3 and not t.is_contiguous():
        base = t.as_strided((t.untyped_storage().nbytes() // 2,), (1,), 0)
        flat = base.contiguous().view(torch.int16).numpy().view(np.uint16)
        return oracle.View(flat, t.stride(0), t.stride(1), t.storage_offset())
    b = bits(t)
    return oracle.View.contiguous(b)


class Guarded:
    """An output tensor inside a larger device buffer whose margins (256 bytes
    on each side, which keeps 16- and 256-byte alignment) hold a known byte
    pattern: a kernel that writes outside its output changes them."""

    PATTERN = 0xA5

    def __init__(self, shape, dtype, zero: bool = False, pad_bytes: int = 256):
        self.el = torch.empty((), dtype=dtype).element_size()
        self.n = math.prod(shape)
        self.pad = pad_bytes // self.el
        self.buf = torch.empty(self.n + 2 * self.pad, dtype=dtype, device=DEV)
        self.buf.view(torch.uint8).fill_(self.PATTERN)
        self.t = self.buf[self.pad:self.pad + self.n].view(shape)
        if zero:
            self.t.zero_()

    def intact(self) -> bool:
        b = self.buf.view(torch.uint8)
        lo, hi = self.pad * self.el, (self.pad + self.n) * self.el
        return bool((b[:lo] == self.PATTERN).all()) and bool((b[hi:] == self.PATTERN).all())


def wbits(w: torch.Tensor):
    return w.numpy() if w.dtype == torch.float32 else bits(w)


def w64(w: torch.Tensor):
    return w.double().numpy()


def rows_f64(t: torch.Tensor) -> np.ndarray:
    T = t.shape[0]
    H = t.shape[-1]
    return t.reshape(-1, H).double().numpy() if t.is_contiguous() else t.contiguous().reshape(-1, H).double().numpy()


# --------------------------------------------------------------------- fwd

def check_fwd(cake, x, w, eps, residual=None):
    T = x.shape[0]
    nh = x.shape[1] if x.dim() == 3 else 1
    H = x.shape[-1]
    y64, r64, hn = oracle.fwd_rows(T, nh, H, view_of(x), wbits(w), eps,
                                   residual=view_of(residual) if residual is not None else None)
    x_d = to_dev(x)
    assert x_d.stride() == x.stride()
    gy, gr = Guarded(x.shape, torch.bfloat16), Guarded((T * nh,), torch.float32)
    gh = Guarded(x.shape, torch.bfloat16) if residual is not None else None
    out = cake.cake_rmsnorm_fwd(x_d, w.to(DEV), eps, residual=to_dev(residual), y=gy.t, rstd=gr.t,
                                h_new=gh.t if gh is not None else None)
    torch.cuda.synchronize()
    assert gy.intact() and gr.intact() and (gh is None or gh.intact()), "forward wrote outside its outputs"
    y, rstd = out[0], out[1]
    yb = bits(y).reshape(-1, H)
    assert tol.ulp_distance(yb, oracle.bf16_round(y64)).max(initial=0) <= 1
    rk = rstd.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(rk / r64 - 1) <= tol.RSTD_REL)
    if residual is not None:
        np.testing.assert_array_equal(bits(out[2]).reshape(-1, H), hn)
    # a recomputed forward is the same bits (checkpointed recompute)
    out2 = cake.cake_rmsnorm_fwd(x_d, w.to(DEV), eps, residual=to_dev(residual))
    torch.cuda.synchronize()
    assert torch.equal(out2[0], y) and torch.equal(out2[1], rstd)
    return r64, hn


# rows of at most 256 columns run on part of a warp (1003 x 64: eight rows
# per warp, the last warp partly empty; 517 x 128: four; 333 x 200: two);
# rows of 264 to 1024 on one warp at 16 to 32 columns per thread (5 x 520,
# 1001 x 640, 77 x 1024)
FWD_SHAPES = [(1, 8), (3, 24), (1003, 64), (517, 128), (333, 200), (37, 256), (5, 520), (1001, 640), (77, 1024),
              (300, 1536), (129, 2048), (33, 4096), (17, 5120), (40, 6144), (9, 8192)]


@pytest.mark.parametrize("T,H", FWD_SHAPES)
@pytest.mark.parametrize("w_dtype", [torch.bfloat16, torch.float32])
def test_fwd_plain(cake, T, H, w_dtype):
    c = cake_inputs.plain_case(T, H, w_dtype=w_dtype, seed=T + H)
    check_fwd(cake, c["x"], c["w"], c["eps"])


@pytest.mark.parametrize("T,H", [(1, 8), (37, 256), (300, 1536), (65, 6144)])
def test_fwd_residual(cake, T, H):
    c = cake_inputs.residual_case(T, H, seed=H)
    check_fwd(cake, c["x"], c["w"], c["eps"], residual=c["residual"])


def test_fwd_outlier_and_offset_families(cake):
    for fam in ("outlier", "offset", "rowmean"):
        c = cake_inputs.plain_case(500, 2048, family=fam, w_dtype=torch.float32, seed=3)
        check_fwd(cake, c["x"], c["w"], c["eps"])


@pytest.mark.parametrize("T,heads,strided", [(1, 24, True), (7, 24, True), (300, 24, True), (5, 4, False),
                                             (300, 4, False)])
def test_fwd_per_head(cake, T, heads, strided):
    c = cake_inputs.heads_case(T, heads, strided=strided, seed=T)
    check_fwd(cake, c["x"], c["w"], c["eps"])


def test_fwd_empty(cake):
    x = torch.empty((0, 256), dtype=torch.bfloat16, device=DEV)
    w = torch.ones(256, dtype=torch.bfloat16, device=DEV)
    y, rstd = cake.cake_rmsnorm_fwd(x, w)
    assert y.shape == (0, 256) and rstd.numel() == 0


# --------------------------------------------------------------------- bwd

VARIANTS = [(f, acc) for f in (0, 1, 2, 3, 4) for acc in (0, 1, 2, 3)]


def oracle_bwd_inputs(x, w, eps, residual=None):
    """rstd (FP32 of the oracle's rstd64) and the normalised input h (bits)."""
    T = x.shape[0]
    nh = x.shape[1] if x.dim() == 3 else 1
    H = x.shape[-1]
    _, r64, hn = oracle.fwd_rows(T, nh, H, view_of(x), wbits(w), eps,
                                 residual=view_of(residual) if residual is not None else None, want_y=False,
                                 want_h=residual is not None)
    return r64.astype(np.float32), hn


def check_bwd(cake, x, dy, w, eps, residual=None, dh=None, variants=VARIANTS, dw_gate=1.0):
    """Run every listed (single, accum) variant; return the worst dw fraction."""
    T = x.shape[0]
    nh = x.shape[1] if x.dim() == 3 else 1
    H = x.shape[-1]
    rin, hn = oracle_bwd_inputs(x, w, eps, residual)
    if residual is not None:
        h_cpu = torch.from_numpy(hn.view(np.int16)).view(torch.bfloat16).reshape(x.shape)
    else:
        h_cpu = x
    hv, dyv = view_of(h_cpu), view_of(dy)
    dhv = view_of(dh) if dh is not None else None
    dx64 = oracle.bwd_rows(T, nh, H, dyv, hv, rin, wbits(w), dh=dhv)
    dw64 = oracle.dw_cols(T, nh, H, dyv, hv, rin)
    dyf, hf = rows_f64(dy), rows_f64(h_cpu)
    dhf = rows_f64(dh) if dh is not None else None
    h_d, dy_d, w_d = to_dev(h_cpu), to_dev(dy), w.to(DEV)
    assert h_d.stride() == h_cpu.stride()
    r_d = torch.from_numpy(rin).to(DEV)
    dh_d = to_dev(dh)
    gws = Guarded((cake.cake_rmsnorm_bwd_workspace_size(h_d, w.dtype, deterministic=False),), torch.uint8,
                  zero=True)
    ws = gws.t
    gdx, gdw = Guarded(h_cpu.shape, torch.bfloat16), Guarded((H,), torch.float32)
    dx_ref_bits = None
    dx_rep = None
    worst = 0.0
    for single, acc in variants:
        det = single != 1  # the pair, the tree and the grid form are deterministic
        outs = []
        for rep in range(2):
            try:
                dx, dw = cake.cake_rmsnorm_bwd_forced(dy_d, h_d, r_d, w_d, dh_d, deterministic=det,
                                                      force_single=single, force_accum=acc, workspace=ws,
                                                      dx=gdx.t, dw=gdw.t)
            except cake.CakeError as e:
                # the tree form exists for the 8-columns-per-thread layout only
                assert single == 2 and e.status == 2
                break
            torch.cuda.synchronize()
            assert gdx.intact() and gdw.intact() and gws.intact(), \
                f"backward wrote outside dx, dw or the workspace (single={single}, accum={acc})"
            outs.append((bits(dx).reshape(-1, H), dw.cpu().numpy()))
        if not outs:
            continue
        (dxb, dwk), (dxb2, dwk2) = outs
        np.testing.assert_array_equal(dxb, dxb2)
        if det:
            np.testing.assert_array_equal(dwk, dwk2)
        if dx_ref_bits is None:
            dx_rep = tol.dx_report(dxb, dx64, dyf, hf, w64(w), rin, oracle.bf16_round, oracle.bf16_bits_to_f64,
                                   dh=dhf)
            assert dx_rep["bounded"] == 0 and dx_rep["off_cancellation"] == 0, f"dx: {dx_rep}"
            dx_ref_bits = dxb
        else:
            np.testing.assert_array_equal(dxb, dx_ref_bits)  # dx: same bits in every variant
        for dwv in (dwk, dwk2):
            frac = tol.dw_budget_fraction(dwv, dw64).max(initial=0.0)
            worst = max(worst, float(frac))
            assert frac <= dw_gate, f"dw worst {frac:.4f} of budget (single={single}, accum={acc})"
    # the default entry point in both modes gives the same dx bits
    for det in (True, False):
        dx, dw = cake.cake_rmsnorm_bwd(dy_d, h_d, r_d, w_d, dh_d, deterministic=det, workspace=ws, dx=gdx.t,
                                       dw=gdw.t)
        torch.cuda.synchronize()
        assert gdx.intact() and gdw.intact() and gws.intact(), "backward wrote outside dx, dw or the workspace"
        np.testing.assert_array_equal(bits(dx).reshape(-1, H), dx_ref_bits)
        frac = float(tol.dw_budget_fraction(dw.cpu().numpy(), dw64).max(initial=0.0))
        worst = max(worst, frac)
        assert frac <= dw_gate
    report.record(f"bwd T={T} nh={nh} H={H} w={'fp32' if w.dtype == torch.float32 else 'bf16'}"
                  f"{' dh' if dh is not None else ''}{' res' if residual is not None else ''} variants={len(variants)}",
                  dx=dx_rep, dw_worst=worst)
    return worst


# rows of 136 to 256 run at half a warp per row, two rows per warp: 2 x 136
# and 333 x 200 leave part of each thread's second vector idle, 1001 x 256
# spans several CTAs and ends on a tile whose second half-warp has no row;
# rows of 384 to 1024 run on one warp at 16 to 32 columns per thread (61 x
# 384 as one CTA, 700 x 512, 1003 x 640, 257 x 832 over several); rows of at
# most 64 columns on a quarter of a warp and of 72 to 128 on half a warp at 8
# columns per thread (1003 x 64 and 517 x 128 end on a partly empty warp)
BWD_SHAPES = [(1, 8), (2, 16), (3, 24), (1003, 64), (33, 72), (517, 128), (2, 136), (37, 256), (333, 200),
              (1001, 256), (61, 384), (700, 512), (1003, 640), (257, 832), (5, 520), (300, 1536), (129, 2048),
              (33, 4096), (17, 5120), (40, 6144), (9, 8192), (1000, 2048),
              # one CTA with fewer rows than row groups: the combine reads only the live groups
              (1, 1536), (2, 2048), (2, 4096), (1, 6144), (5, 1536)]


@pytest.mark.parametrize("T,H", BWD_SHAPES)
@pytest.mark.parametrize("w_dtype", [torch.bfloat16, torch.float32])
def test_bwd_plain(cake, T, H, w_dtype):
    c = cake_inputs.plain_case(T, H, w_dtype=w_dtype, seed=7 * T + H)
    check_bwd(cake, c["x"], c["dy"], c["w"], c["eps"])


@pytest.mark.parametrize("family", ["outlier", "offset", "rowmean"])
@pytest.mark.parametrize("T,H", [(700, 2048), (2500, 1536), (2501, 256)])
def test_bwd_families(cake, family, T, H):
    # the input families of the accuracy sweep, through every form; 2500 rows
    # take the blocked dw sums
    c = cake_inputs.plain_case(T, H, family=family, w_dtype=torch.float32, seed=T + len(family))
    check_bwd(cake, c["x"], c["dy"], c["w"], c["eps"], variants=[(0, 0), (0, 1), (1, 1), (3, 3)])


@pytest.mark.parametrize("H", [8, 64, 256, 520, 1536, 2048, 4096, 6144, 8192])
def test_one_row_dw_is_one_rounding(cake, H):
    """One row: dw_j = dy_j * x_j * rstd with a single rounding to FP32.  The
    BF16 product is exact in FP32, the multiply-add by rstd rounds once, and
    every accumulation form and every form of the column reduction leaves that
    value as it is.  FP64 holds the exact product (16 + 24 significant bits),
    so the equality is bit for bit.  The CTA's other row groups own no row:
    any bit of theirs in the group combine, or a slot read from the wrong
    place, breaks it."""
    c = cake_inputs.plain_case(1, H, seed=H + 5)
    x, dy, w = c["x"], c["dy"], c["w"]
    rin, _ = oracle_bwd_inputs(x, w, c["eps"])
    want = (rows_f64(dy)[0] * rows_f64(x)[0] * np.float64(rin[0])).astype(np.float32)
    x_d, dy_d, w_d = x.to(DEV), dy.to(DEV), w.to(DEV)
    r_d = torch.from_numpy(rin).to(DEV)
    runs = [("table det", lambda: cake.cake_rmsnorm_bwd(dy_d, x_d, r_d, w_d, None, deterministic=True)),
            ("table nondet", lambda: cake.cake_rmsnorm_bwd(dy_d, x_d, r_d, w_d, None, deterministic=False))]
    for single, acc in VARIANTS:
        runs.append((f"form {single} accum {acc}",
                     lambda single=single, acc=acc: cake.cake_rmsnorm_bwd_forced(
                         dy_d, x_d, r_d, w_d, None, deterministic=single != 1, force_single=single, force_accum=acc)))
    checked = 0
    for name, fn in runs:
        try:
            _, dw = fn()
        except cake.CakeError as e:
            assert e.status == 2, name  # the tree form exists for some layouts only
            continue
        torch.cuda.synchronize()
        got = dw.cpu().numpy()
        bad = np.flatnonzero(got.view(np.uint32) != want.view(np.uint32))
        assert bad.size == 0, f"{name}: {bad.size} columns differ, first {bad[0]}: {got[bad[0]]!r} != {want[bad[0]]!r}"
        checked += 1
    assert checked >= 18


@pytest.mark.parametrize("T,H", [(3, 256), (300, 1536), (77, 6144)])
def test_bwd_residual(cake, T, H):
    c = cake_inputs.residual_case(T, H, seed=H + 1)
    check_bwd(cake, c["x"], c["dy"], c["w"], c["eps"], residual=c["residual"], dh=c["dh"])
    check_bwd(cake, c["x"], c["dy"], c["w"], c["eps"], residual=c["residual"], dh=None,
              variants=[(0, 2), (1, 2)])


@pytest.mark.parametrize("T,heads,strided", [(1, 24, True), (7, 24, True), (300, 24, True), (5, 4, False),
                                             (300, 4, False)])
def test_bwd_per_head(cake, T, heads, strided):
    c = cake_inputs.heads_case(T, heads, strided=strided, seed=T + heads)
    check_bwd(cake, c["x"], c["dy"], c["w"], c["eps"])


def test_per_head_equals_gathered_rows(cake):
    # the strided [T, 24, 256] view gives the same dx bits and (deterministic)
    # the same dw bits as its gathered contiguous copy ... when the partition
    # is the same, i.e. the same row count: compare [T, 24, 256] with
    # [T*24, 1, 256] (both 24*T rows of 256).
    c = cake_inputs.heads_case(64, 24, strided=True, seed=5)
    x, dy, w = c["x"], c["dy"], c["w"]
    rin, _ = oracle_bwd_inputs(x, w, c["eps"])
    r_d = torch.from_numpy(rin).to(DEV)
    dx1, dw1 = cake.cake_rmsnorm_bwd(dy.to(DEV), to_dev(x), r_d, w.to(DEV), deterministic=True)
    xg = x.contiguous().reshape(64 * 24, 256)
    dx2, dw2 = cake.cake_rmsnorm_bwd(dy.reshape(64 * 24, 256).to(DEV), xg.to(DEV), r_d, w.to(DEV), deterministic=True)
    torch.cuda.synchronize()
    assert torch.equal(dx1.reshape(-1, 256), dx2)
    assert torch.equal(dw1, dw2)


def test_bwd_empty(cake):
    x = torch.empty((0, 2048), dtype=torch.bfloat16, device=DEV)
    w = torch.ones(2048, dtype=torch.float32, device=DEV)
    dw = torch.full((2048,), 7.0, device=DEV)
    cake.cake_rmsnorm_bwd(x, x, torch.empty(0, device=DEV), w, dw=dw, workspace=torch.zeros(256, dtype=torch.uint8,
                                                                                               device=DEV))
    torch.cuda.synchronize()
    assert not dw.any()


def test_single_kernel_leaves_workspace_clean(cake):
    c = cake_inputs.plain_case(700, 2048, seed=11)
    rin, _ = oracle_bwd_inputs(c["x"], c["w"], c["eps"])
    x, dy, w, r = c["x"].to(DEV), c["dy"].to(DEV), c["w"].to(DEV), torch.from_numpy(rin).to(DEV)
    ws = cake.cake_rmsnorm_bwd_workspace(x, w.dtype, deterministic=False)
    first = None
    for _ in range(5):
        _, dw = cake.cake_rmsnorm_bwd_forced(dy, x, r, w, deterministic=False, force_single=1, workspace=ws)
        torch.cuda.synchronize()
        if first is None:
            first = dw.clone()
        # FP64 accumulation: repeated calls agree to FP32 rounding of the same sum
        assert torch.allclose(dw, first, rtol=1e-6, atol=1e-6)
    head = ws[: 512 + 8 * 2048 * 8].cpu()  # the counters and the 8 accumulator banks
    assert not head.any()


def test_grid_form_barrier_words(cake):
    # the cooperative form's barrier leaves its counter at zero and advances
    # its generation once per call; dw is the same bits every call
    c = cake_inputs.plain_case(900, 1536, seed=12)
    rin, _ = oracle_bwd_inputs(c["x"], c["w"], c["eps"])
    x, dy, w, r = c["x"].to(DEV), c["dy"].to(DEV), c["w"].to(DEV), torch.from_numpy(rin).to(DEV)
    ws = cake.cake_rmsnorm_bwd_workspace(x, w.dtype, deterministic=True)
    first = None
    for call in range(3):
        _, dw = cake.cake_rmsnorm_bwd_forced(dy, x, r, w, deterministic=True, force_single=3, workspace=ws)
        torch.cuda.synchronize()
        words = ws[:512].cpu().view(torch.int32)
        assert int(words[64]) == 0 and int(words[65]) == call + 1
        if first is None:
            first = dw.clone()
        assert torch.equal(dw, first)
    assert cake.cake_rmsnorm_device_status() == 0


@pytest.mark.parametrize("H", [8, 256, 512, 1536, 2048, 4096, 5120, 6144, 8192])
def test_table_plans_only_resident_ctas(cake, H):
    # every CTA of a plan's grid is resident at once: the table never asks for
    # more CTAs per SM than the register file and shared memory hold
    for backward in (False, True):
        for extra in (False, True):
            for det in (True, False):
                for accum in (None, 0, 1, 2, 3):
                    if not backward and (accum is not None or not det):
                        continue
                    planned, resident = cake.cake_rmsnorm_plan_occupancy((65536, 1, H), backward, extra, det, accum)
                    assert 1 <= planned <= resident, (H, backward, extra, det, accum, planned, resident)


def test_cluster_form_needs_no_workspace(cake):
    # the cluster form keeps its partials in the cluster's shared memory: it
    # runs through the C ABI with no workspace at all, deterministic, and
    # within the budget
    from bwd_dw_column_gb300 import _Shape, _Tensor
    import ctypes
    T, H = 200, 2048
    c = cake_inputs.plain_case(T, H, w_dtype=torch.float32, seed=13)
    rin, _ = oracle_bwd_inputs(c["x"], c["w"], c["eps"])
    xv, dyv = view_of(c["x"]), view_of(c["dy"])
    dw64 = oracle.dw_cols(T, 1, H, dyv, xv, rin)
    x, dy, w, r = c["x"].to(DEV), c["dy"].to(DEV), c["w"].to(DEV), torch.from_numpy(rin).to(DEV)
    lib = cake.load_library()
    outs = []
    for _ in range(2):
        dx = torch.empty_like(x)
        dw = torch.empty(H, device=DEV)
        st = lib.cake_rmsnorm_bwd_forced(ctypes.byref(_Shape(T, 1, H)), ctypes.byref(_Tensor(dy.data_ptr(), H, 0)),
                                         ctypes.byref(_Tensor(x.data_ptr(), H, 0)), r.data_ptr(), w.data_ptr(), 1,
                                         None, ctypes.byref(_Tensor(dx.data_ptr(), H, 0)), dw.data_ptr(), None, 0,
                                         1, 4, -1, torch.cuda.current_stream().cuda_stream)
        assert st == 0
        torch.cuda.synchronize()
        outs.append((dx, dw))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    assert float(tol.dw_budget_fraction(outs[0][1].cpu().numpy(), dw64).max()) <= 1.0
    ref_dx, _ = cake.cake_rmsnorm_bwd(dy, x, r, w, deterministic=True)
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], ref_dx)
    assert cake.cake_rmsnorm_device_status() == 0
