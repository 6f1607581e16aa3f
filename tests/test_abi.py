"""The C ABI without a GPU: the library builds and loads, exports every
function the header declares, and its host-side logic (argument validation,
the window table, workspace sizing) behaves as documented.  No call here
launches a kernel."""
import ctypes
import json
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cake_rmsnorm.h")


@pytest.fixture(scope="module")
def cake():
    from bwd_dw_column_gb300 import _build
    _build.build()
    import bwd_dw_column_gb300 as cake
    cake.load_library()
    return cake


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cake_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("cake_rmsnorm_fwd", "cake_rmsnorm_bwd", "cake_rmsnorm_bwd_workspace_size"):
        assert required in names


def test_library_exports_every_declared_symbol(cake):
    lib = cake.load_library()
    for name in _declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", cake.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (cake_[a-z0-9_]+)\b", out))
    assert set(_declared_functions()) <= exported


def test_abi_version_and_status_strings(cake):
    lib = cake.load_library()
    assert lib.cake_rmsnorm_abi_version() == 1
    for code in range(6):
        assert cake.cake_status_str(code)
    assert cake.cake_status_str(99) == "unknown status"


def test_library_is_sm103a_only(cake):
    out = subprocess.run(["cuobjdump", "--list-elf", cake.LIB_PATH], capture_output=True, text=True).stdout
    archs = set(re.findall(r"sm_(\d+a?)", out))
    assert archs == {"103a"}, archs


# ------------------------------------------------------------ window table

@pytest.mark.parametrize("H", [8, 16, 256, 512, 1536, 2048, 4096, 5120, 6144, 8192])
@pytest.mark.parametrize("T", [1, 37, 256, 65536, 131072])
def test_select_is_a_valid_launch(cake, H, T):
    for det in (True, False):
        v = cake.cake_rmsnorm_bwd_select((T, 1, H), deterministic=det)
        threads = 32 * (v["row_groups"] * v["warps_per_row"] + 1)
        assert threads <= (832 if v["vec_per_thread"] == 1 else 416)
        assert v["smem_bytes"] <= 227 * 1024
        assert 2 <= v["stages"] <= 16
        assert v["vec_per_thread"] * 32 * v["warps_per_row"] * 8 >= H
        assert v["ctas"] * v["rows_per_cta"] >= T and (v["ctas"] - 1) * v["rows_per_cta"] < T
        assert v["ctas"] <= 152 * 4
        # both modes run the pair (no single-kernel form beats it on GB300)
        assert v["single"] == 0
    # the non-deterministic mode still offers every single-kernel form
    for form in (1, 3):
        assert cake.cake_rmsnorm_bwd_select((T, 1, H), deterministic=False, force_single=form)["single"] == form


def test_every_width_plans_a_valid_launch(cake):
    # every supported H (multiples of 8 up to 8192), with and without dh and
    # for every dw accumulation form: the plan fits the kernel it launches
    for H in range(8, 8193, 8):
        for T, dh, acc in ((65536, False, None), (7, True, None), (3000, False, 2), (3000, True, 3)):
            v = cake.cake_rmsnorm_bwd_select((T, 1, H), deterministic=True, has_dh=dh, force_accum=acc)
            warps = v["row_groups"] * v["warps_per_row"] + 1
            bound = 544 if v["rows_per_group"] == 2 else (832 if v["vec_per_thread"] == 1 else 416)
            assert 32 * warps <= bound, (H, T, v)
            assert v["smem_bytes"] <= 227 * 1024, (H, T, v)
            assert 2 <= v["stages"] <= 16, (H, T, v)
            assert v["vec_per_thread"] * 32 * v["warps_per_row"] * 8 >= H, (H, v)
            assert v["ctas"] * v["rows_per_cta"] >= T > (v["ctas"] - 1) * v["rows_per_cta"], (H, T, v)
            if v["warps_per_row"] > 1:
                assert v["row_groups"] <= 14, (H, v)


def test_row_layout_depends_on_h_alone(cake):
    for H in (200, 256, 1536, 2048, 6144):
        layouts = set()
        for T in (1, 5, 300, 70000):
            for det in (True, False):
                for dh in (False, True):
                    v = cake.cake_rmsnorm_bwd_select((T, 1, H), deterministic=det, has_dh=dh)
                    layouts.add((v["vec_per_thread"], v["warps_per_row"], v["lanes_per_row"]))
        assert len(layouts) == 1, (H, layouts)


@pytest.mark.parametrize("H,layout", [(8, (4, 2, 8)), (64, (4, 2, 8)), (72, (8, 2, 4)), (128, (8, 2, 4)),
                                      (136, (16, 2, 2)), (200, (16, 2, 2)), (256, (16, 2, 2)), (264, (32, 2, 1)),
                                      (512, (32, 2, 1))])
def test_part_warp_rows(cake, H, layout):
    # rows of at most 256 columns take part of a warp at 16 columns per
    # thread: an eighth up to 64 columns, a quarter to 128, a half to 256;
    # wider rows keep whole warps.  layout = (lanes per row, vectors per
    # thread, rows per group)
    v = cake.cake_rmsnorm_bwd_select((4096, 1, H), deterministic=True)
    assert (v["lanes_per_row"], v["vec_per_thread"], v["rows_per_group"]) == layout, v
    assert v["warps_per_row"] == 1


@pytest.mark.parametrize("shape,one", [((1, 1, 1536), True), ((16, 1, 1536), True), ((17, 1, 1536), False),
                                       ((96, 1, 256), True), ((97, 1, 256), False), ((4, 24, 256), True),
                                       ((4, 1, 6144), True), ((5, 1, 6144), False)])
def test_small_row_sets_run_as_one_cta(cake, shape, one):
    # up to 24576 elements the pair is one CTA whose main kernel writes dw
    # (one launch); beyond, several CTAs and the fixed-order reduce
    for det in (True, False):
        v = cake.cake_rmsnorm_bwd_select(shape, deterministic=det)
        assert (v["ctas"] == 1) == one, (shape, v)


@pytest.mark.parametrize("shape,groups", [((64, 1, 1536), 2), ((304, 1, 1536), 2), ((305, 1, 1536), 6),
                                          ((16, 1, 1536), 6), ((256, 1, 4096), 2), ((1024, 1, 4096), 3),
                                          ((256, 1, 256), 4), ((256, 1, 6144), 2)])
def test_few_rows_of_several_warps_take_two_groups(cake, shape, groups):
    # up to two rows per SM, rows of several warps run as CTAs of two row
    # groups (more CTAs share the rows); one-CTA row sets and rows of one warp
    # keep their groups
    v = cake.cake_rmsnorm_bwd_select(shape, deterministic=True)
    assert v["row_groups"] == groups, (shape, v)


def test_partition_depends_on_shape_alone(cake):
    a = cake.cake_rmsnorm_bwd_select((65536, 1, 2048), deterministic=True)
    b = cake.cake_rmsnorm_bwd_select((65536, 1, 2048), deterministic=True)
    assert a == b
    heads = cake.cake_rmsnorm_bwd_select((32768, 24, 256), deterministic=True)
    assert heads["ctas"] * heads["rows_per_cta"] >= 32768 * 24


def test_forced_variants(cake):
    for accum in (cake.DW_PLAIN, cake.DW_BLOCKED, cake.DW_TWOSUM, cake.DW_KAHAN):
        v = cake.cake_rmsnorm_bwd_select((1000, 1, 2048), deterministic=False, force_single=1, force_accum=accum)
        assert v["single"] == 1 and v["dw_accum"] == accum
        v = cake.cake_rmsnorm_bwd_select((1000, 1, 2048), deterministic=True, force_single=0, force_accum=accum)
        assert v["single"] == 0 and v["dw_accum"] == accum
    with pytest.raises(cake.CakeError) as e:
        cake.cake_rmsnorm_bwd_select((1000, 1, 2048), deterministic=True, force_single=1)
    assert e.value.status == 1


@pytest.mark.parametrize("shape,accum", [
    ((1, 1, 1536), 0), ((2048, 1, 2048), 0),                 # plain FP32 sums
    ((2049, 1, 2048), 1), ((131072, 1, 6144), 1),            # blocked
    ((32768, 4, 256), 1),                                    # 131072 rows of the per-head view
    ((131073, 1, 4096), 3), ((32768, 24, 256), 3),           # Kahan past the blocked window
    ((1 << 20, 1, 256), 3), (((1 << 20) + 1, 1, 256), 2),    # TwoSum beyond
])
def test_accuracy_windows(cake, shape, accum):
    # the per-thread dw sums the table takes by the rows each column sums
    for det in (True, False):
        assert cake.cake_rmsnorm_bwd_select(shape, deterministic=det)["dw_accum"] == accum


@pytest.mark.parametrize("shape,status", [
    ((10, 1, 12), 2),          # H not a multiple of 8
    ((10, 1, 8200), 2),        # H above the maximum
    ((-1, 1, 256), 1),         # negative T
    ((10, 0, 256), 1),         # no heads
    ((1 << 30, 4, 256), 2),    # 2^32 rows
])
def test_select_rejects_bad_shapes(cake, shape, status):
    with pytest.raises(cake.CakeError) as e:
        cake.cake_rmsnorm_bwd_select(shape)
    assert e.value.status == status


def test_workspace_size(cake):
    assert cake.cake_rmsnorm_bwd_workspace_size((0, 1, 2048)) == 0
    n = cake.cake_rmsnorm_bwd_workspace_size((65536, 1, 2048))
    v = cake.cake_rmsnorm_bwd_select((65536, 1, 2048))
    assert n >= v["ctas"] * 2048 * 8 + 2048 * 8
    assert n < 64 << 20
    big = cake.cake_rmsnorm_bwd_workspace_size((131072, 1, 6144), deterministic=False)
    assert big >= 6144 * 8


# ------------------------------------------------------ argument validation
# Fake, never-dereferenced device addresses: validation rejects the call
# before any CUDA runtime call is made.  A call that passes validation would
# launch a kernel on those addresses, so such calls are made only where no
# GPU is present (the launch then fails with CAKE_ERR_CUDA, 4).


def _no_gpu() -> bool:
    import torch
    return not torch.cuda.is_available()


def _past_validation(call) -> None:
    """Check that a call with fake addresses passes validation -- only where
    there is no GPU to launch on."""
    if _no_gpu():
        assert call() == 4

def _T(addr, st, sh=0):
    from bwd_dw_column_gb300 import _Tensor
    return _Tensor(addr, st, sh)


def _S(T, nh, H):
    from bwd_dw_column_gb300 import _Shape
    return _Shape(T, nh, H)


def _fwd(cake, shape, x, res, w, y, hn, rstd, eps=1e-6, wd=0):
    lib = cake.load_library()
    r = lambda t: ctypes.byref(t) if t is not None else None
    return lib.cake_rmsnorm_fwd(r(shape), r(x), r(res), w, wd, eps, r(y), r(hn), rstd, None)


def test_fwd_validation(cake):
    A = 0x100000
    ok_shape = _S(4, 1, 64)
    good = lambda: _T(A, 64)
    _past_validation(lambda: _fwd(cake, ok_shape, good(), None, A, good(), None, A + 4096))
    assert _fwd(cake, None, good(), None, A, good(), None, A) == 1
    assert _fwd(cake, ok_shape, None, None, A, good(), None, A) == 1
    assert _fwd(cake, ok_shape, _T(A + 2, 64), None, A, good(), None, A) == 2      # misaligned x
    assert _fwd(cake, ok_shape, _T(A, 60), None, A, good(), None, A) == 2          # stride not 16 B
    assert _fwd(cake, ok_shape, good(), None, A + 8, good(), None, A) == 2         # misaligned w
    assert _fwd(cake, ok_shape, good(), None, A, good(), None, A + 2) == 2         # misaligned rstd
    assert _fwd(cake, ok_shape, good(), good(), A, good(), None, A) == 1           # residual without h_new
    assert _fwd(cake, ok_shape, good(), None, A, good(), good(), A) == 1           # h_new without residual
    assert _fwd(cake, ok_shape, good(), None, A, good(), None, A, eps=float("nan")) == 1
    assert _fwd(cake, ok_shape, good(), None, A, good(), None, A, wd=7) == 1
    assert _fwd(cake, _S(0, 1, 64), None, None, None, None, None, None) == 0      # T = 0: no-op


def _bwd(cake, shape, dy, x, rstd, w, dh, dx, dw, ws, nbytes, det=1, wd=0):
    lib = cake.load_library()
    r = lambda t: ctypes.byref(t) if t is not None else None
    return lib.cake_rmsnorm_bwd(r(shape), r(dy), r(x), rstd, w, wd, r(dh), r(dx), dw, ws, nbytes, det, None)


def test_bwd_validation(cake):
    A, B = 0x100000, 0x10000000  # inputs at A, dx at B (1.2 MB of rows apart)
    shape = _S(300, 1, 2048)
    need = cake.cake_rmsnorm_bwd_workspace_size((300, 1, 2048))
    t = lambda: _T(A, 2048)
    o = lambda: _T(B, 2048)
    assert _bwd(cake, shape, t(), t(), A, A, None, o(), A, A, 4096) == 3          # workspace too small
    assert _bwd(cake, shape, t(), t(), A, A, None, o(), A, None, need) == 3       # no workspace
    assert _bwd(cake, shape, t(), t(), A, A, None, o(), A, A + 16, need) == 2     # workspace not 256-B aligned
    assert _bwd(cake, shape, t(), t(), None, A, None, o(), A, A, need) == 1       # no rstd
    assert _bwd(cake, shape, t(), t(), A, A, None, o(), None, A, need) == 1       # no dw
    assert _bwd(cake, shape, _T(A, 2040), t(), A, A, None, o(), A, A, need) == 2  # rows overlap
    assert _bwd(cake, _S(300, 1, 2044), t(), t(), A, A, None, o(), A, A, need) == 2
    assert _bwd(cake, shape, t(), t(), A, A, None, o(), A, A, need, wd=3) == 1
    heads = _S(16, 24, 256)
    assert _bwd(cake, heads, _T(A, 24 * 256, 256), _T(A, 24 * 512, 100), A, A, None,
                _T(B, 24 * 256, 256), A, A, 1 << 24) == 2                           # head stride not 16 B


def test_bwd_rejects_dx_sharing_memory(cake):
    A, B, D = 0x100000, 0x10000000, 0x20000000
    shape = _S(300, 1, 2048)
    rows = 300 * 2048 * 2
    t = lambda a: _T(a, 2048)
    # dx is dy, or x, or dh, or straddles the end of x: rejected before the workspace check
    assert _bwd(cake, shape, t(A), t(B), A, A, None, t(A), A, A, 0) == 1
    assert _bwd(cake, shape, t(A), t(B), A, A, None, t(B), A, A, 0) == 1
    assert _bwd(cake, shape, t(A), t(B), A, A, t(D), t(D), A, A, 0) == 1
    assert _bwd(cake, shape, t(A), t(B), A, A, None, t(B + rows - 4096), A, A, 0) == 1
    # disjoint dx gets as far as the workspace check
    assert _bwd(cake, shape, t(A), t(B), A, A, t(D), t(B + rows), A, A, 0) == 3


def test_bwd_rejects_output_rows_that_overlap(cake):
    A, B = 0x100000, 0x10000000
    heads = _S(16, 24, 256)
    x = _T(A, 24 * 256, 256)
    assert _bwd(cake, heads, x, x, A, A, None, _T(B, 24 * 256, 256), A, A, 0) == 3   # contiguous [T, 24, 256]
    assert _bwd(cake, heads, x, x, A, A, None, _T(B, 256, 256), A, A, 0) == 1        # token rows repeat heads
    assert _bwd(cake, heads, x, x, A, A, None, _T(B, 0, 256), A, A, 0) == 1          # every token on one row set
    assert _bwd(cake, heads, x, x, A, A, None, _T(B, 24 * 512, 512), A, A, 0) == 3   # strided, disjoint
    # head-major [nh, T, 256] storage: heads step past all tokens
    assert _bwd(cake, heads, x, x, A, A, None, _T(B, 256, 16 * 256), A, A, 0) == 3
    assert _bwd(cake, heads, x, x, A, A, None, _T(B, 256, 8 * 256), A, A, 0) == 1


def test_fwd_rejects_outputs_sharing_memory(cake):
    A, B, C = 0x100000, 0x10000000, 0x20000000
    s = _S(4, 1, 64)
    t = lambda a: _T(a, 64)
    # y over x exactly (in place) is allowed: it gets past validation
    _past_validation(lambda: _fwd(cake, s, t(A), None, A, t(A), None, C))
    assert _fwd(cake, s, t(A), None, A, t(A + 128), None, C) == 1        # y straddles rows of x
    assert _fwd(cake, s, t(A), t(B), A, t(C), t(C), C) == 1              # y and h_new share memory
    assert _fwd(cake, s, t(A), t(B), A, t(C), t(B + 128), C) == 1        # h_new straddles the residual
    _past_validation(lambda: _fwd(cake, s, t(A), t(B), A, t(C), t(A), C))  # h_new over x in place
    assert _fwd(cake, _S(4, 2, 64), _T(A, 128, 64), None, A, _T(C, 64, 64), None, C) == 1  # y rows overlap


def test_timeout_test_entry_validates_its_limit(cake):
    lib = cake.load_library()
    A = 0x100000
    for limit in (0, 1000001):
        st = lib.cake_rmsnorm_bwd_timeout_test(ctypes.byref(_S(4, 1, 256)), ctypes.byref(_T(A, 256)),
                                               ctypes.byref(_T(A, 256)), A, A, 0, ctypes.byref(_T(A, 256)), A, A,
                                               1 << 20, limit, None)
        assert st == 1


def test_row_groups_fit_named_barriers(cake):
    # A row that spans several warps syncs on named barrier 1 + g (row group
    # g); the consumer-wide barrier is id 15.  No plan may give a group an id
    # of 15 or more, nor more warps than a CTA of the row kernels holds.
    for H in range(8, 8193, 8):
        for det in (True, False):
            v = cake.cake_rmsnorm_bwd_select((4096, 1, H), deterministic=det)
            if v["warps_per_row"] > 1:
                assert v["row_groups"] <= 14
            # consumer warps + the producer within the kernel's largest CTA
            # (832 threads; 544 for two rows per group)
            assert v["row_groups"] * v["warps_per_row"] + 1 <= (26 if v["rows_per_group"] == 1 else 17)


@pytest.mark.parametrize("tune", ["groups=12", "groups=24", "groups=12,cps=1"])
def test_row_group_override_is_capped(cake, tune):
    # the tuning override cannot push a multi-warp row past the barrier ids
    code = ("import bwd_dw_column_gb300 as c, json; "
            "print(json.dumps([c.cake_rmsnorm_bwd_select((65536, 1, H)) for H in (1152, 1536, 2048, 1040)]))")
    env = dict(os.environ, CAKE_TUNE=tune)
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, cwd=ROOT, check=True)
    for v in json.loads(out.stdout.strip().splitlines()[-1]):
        assert v["warps_per_row"] > 1
        assert v["row_groups"] <= 14
        assert v["row_groups"] * v["warps_per_row"] + 1 <= (26 if v["vec_per_thread"] == 1 else 13)


@pytest.mark.parametrize("T,H", [(1, 1536), (16, 1536), (256, 1536), (256, 4096), (1000, 6144), (4096, 256),
                                 (70000, 2048)])
def test_cluster_form_selection(cake, T, H):
    # one cluster of at most 8 CTAs (the portable cluster size) covering every
    # row, with room for its partial in shared memory; no workspace needed
    v = cake.cake_rmsnorm_bwd_select((T, 1, H), deterministic=True, force_single=4)
    assert v["single"] == 4 and 1 <= v["ctas"] <= 8
    assert v["ctas"] * v["rows_per_cta"] >= T > (v["ctas"] - 1) * v["rows_per_cta"]
    assert v["smem_bytes"] <= 227 * 1024 and v["smem_bytes"] >= 1024 + 4 * H + 8 * H
    A, B = 0x100000, 0x40000000
    # past validation with no workspace
    _past_validation(lambda: _bwd_forced(cake, _S(T, 1, H), _T(A, H), _T(A, H), A, A, None, _T(B, H), A, None, 0, 1, 4))


def _bwd_forced(cake, shape, dy, x, rstd, w, dh, dx, dw, ws, nbytes, det, single, accum=-1):
    lib = cake.load_library()
    r = lambda t: ctypes.byref(t) if t is not None else None
    return lib.cake_rmsnorm_bwd_forced(r(shape), r(dy), r(x), rstd, w, 0, r(dh), r(dx), dw, ws, nbytes, det, single,
                                       accum, None)


def test_tree_form_selection(cake):
    # rows of 256 run at half a warp per row in every form, the tree included,
    # so that dx has the same bits whichever form is picked
    v = cake.cake_rmsnorm_bwd_select((32768, 4, 256), deterministic=True, force_single=2)
    assert v["single"] == 2 and v["vec_per_thread"] == 2 and v["lanes_per_row"] == 16
    v = cake.cake_rmsnorm_bwd_select((32768, 4, 128), deterministic=True, force_single=2)
    assert v["single"] == 2 and v["vec_per_thread"] == 2 and v["lanes_per_row"] == 8
    v = cake.cake_rmsnorm_bwd_select((32768, 4, 64), deterministic=True, force_single=2)
    assert v["single"] == 2 and v["vec_per_thread"] == 2 and v["lanes_per_row"] == 4
    v = cake.cake_rmsnorm_bwd_select((1000, 1, 512), deterministic=False, force_single=2)
    assert v["single"] == 2
    for H in (2048, 8192):  # 32 and 24 columns per thread: no tree form
        with pytest.raises(cake.CakeError) as e:
            cake.cake_rmsnorm_bwd_select((1000, 1, H), deterministic=True, force_single=2)
        assert e.value.status == 2
    # the workspace the size query reports holds every form, the tree included
    n = cake.cake_rmsnorm_bwd_workspace_size((32768, 4, 256))
    v = cake.cake_rmsnorm_bwd_select((32768, 4, 256), force_single=2)
    groups = (v["ctas"] + 15) // 16
    assert n >= 256 + 8 * 8 * 256 + v["ctas"] * 256 * 8 + groups * 256 * 8


C_CLIENT = r"""
#include "cake_rmsnorm.h"
#include <stdio.h>
int main(void) {
    cake_shape s = {65536, 1, 2048};
    cake_variant v;
    cake_status st = cake_rmsnorm_bwd_select(&s, CAKE_FP32, 1, 0, -1, -1, &v);
    size_t ws = cake_rmsnorm_bwd_workspace_size(&s, CAKE_FP32, 1);
    cake_shape bad = {4, 1, 12};  /* H not a multiple of 8 */
    cake_status st_bad = cake_rmsnorm_bwd_select(&bad, CAKE_FP32, 1, 0, -1, -1, &v);
    printf("%d %zu %d %d %s\n", (int)st, ws, (int)st_bad, cake_rmsnorm_abi_version(), cake_status_str(st_bad));
    return 0;
}
"""


def test_header_is_plain_c_and_the_library_links_from_c(cake, tmp_path):
    # the boundary needs no C++ and no torch: a C99 client compiles against
    # the header, links the library and calls its host-only entry points
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only",
                           "-x", "c", HEADER])
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(cake.LIB_PATH)
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), str(src),
                           "-L", libdir, "-lcake_rmsnorm", "-Wl,-rpath," + libdir, "-o", str(exe)])
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    assert out[0] == "0" and int(out[1]) > 0 and out[2] == "2" and out[3] == "1"


def test_host_path_validation(cake):
    # the backward from host memory: argument errors come back before any
    # CUDA call; T = 0 zero-fills dw on the host at once
    import numpy as np
    lib = cake.load_library()
    S = _S(100, 1, 2048)
    A = 0x100000
    need = cake.cake_rmsnorm_bwd_host_staging_size((100, 1, 2048), has_dh=False, chunks=4)
    assert need > 0
    assert cake.cake_rmsnorm_bwd_host_staging_size((100, 1, 2048), chunks=0) == 0
    assert cake.cake_rmsnorm_bwd_host_staging_size((100, 1, 2048), chunks=65) == 0
    call = lambda shape, chunks, staging, nbytes, dw=A: lib.cake_rmsnorm_bwd_host(
        ctypes.byref(shape), A, A, A, A, 0, None, A, dw, staging, nbytes, chunks, 1, None)
    assert call(S, 0, A, need) == 1            # chunks out of range
    assert call(S, 65, A, need) == 1
    assert call(S, 4, None, need) == 3         # no staging
    assert call(S, 4, A, need - 1) == 3        # staging too small
    assert call(S, 4, A + 16, need) == 2       # staging not 256-byte aligned
    assert call(_S(100, 1, 12), 4, A, need) == 2  # H not a multiple of 8
    dw = np.full(2048, 5.0, dtype=np.float32)
    assert call(_S(0, 1, 2048), 4, None, 0, dw=dw.ctypes.data) == 0
    assert not dw.any()
