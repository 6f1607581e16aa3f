"""Row layouts the window table does not pick, held to the oracle.

The developer override CAKE_TUNE reaches kernel builds that no table plan
uses today -- 8 columns per thread on 16 warps with two rows per group,
16 columns per thread, 32 columns on two CTAs per SM, narrow rows on whole
warps instead of part of one, or on part of one at 8 columns per thread.  The override is read
once per process, so each layout runs in a child process that applies the
parity checks of tests/test_parity.py (dx against the oracle and the same
bits across forms, calls and modes; dw within the budget) to a few shapes.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
sys.path.insert(0, {root!r})
import torch
import cake_inputs
import __graft_entry__
__graft_entry__.build()
import bwd_dw_column_gb300 as cake
from tests.test_parity import check_bwd, check_fwd
for T, H in {shapes!r}:
    v = cake.cake_rmsnorm_bwd_select((T, 1, H))
    assert (v["vec_per_thread"], v["rows_per_group"]) == {want!r}, v
    c = cake_inputs.plain_case(T, H, w_dtype=torch.float32, seed=T + H)
    check_bwd(cake, c["x"], c["dy"], c["w"], c["eps"], variants=[(0, 0), (0, 1), (0, 3), (1, 1), (3, 1), (4, 1)])
    check_fwd(cake, c["x"], c["w"], c["eps"])
assert cake.cake_rmsnorm_device_status() == 0
print("ok")
"""

LAYOUTS = [
    ("vpt=1", [(300, 4096), (37, 3584)], (1, 2)),        # 16 warps per row, two rows per group
    ("vpt=2,fvpt=3", [(300, 2048), (45, 1024)], (2, 1)),  # 16 columns per thread
    ("vpt=4,groups=1,cps=2", [(300, 4096)], (4, 1)),     # 32 columns, two CTAs per SM
    ("half=0", [(300, 256), (77, 64)], (1, 1)),           # rows of <= 256 columns on whole warps
    ("narrow=0", [(1003, 64), (77, 8)], (1, 4)),         # quarter-warp rows at 8 columns per thread
]


@pytest.mark.parametrize("tune,shapes,want", LAYOUTS, ids=[l[0] for l in LAYOUTS])
def test_tuned_layout_parity(tune, shapes, want):
    env = dict(os.environ, CAKE_TUNE=tune)
    code = CHILD.format(root=ROOT, shapes=shapes, want=want)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, cwd=ROOT,
                       timeout=900)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-4000:]
