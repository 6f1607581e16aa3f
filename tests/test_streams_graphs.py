"""Stream and graph use of the entry points, as a training framework makes it.

* A forward and a deterministic backward captured together in a CUDA graph
  and replayed give the same bits as the eager calls (after one eager call on
  the device, which sets the kernels' attributes and looks up the status
  word before capture).
* Two backwards on two streams with their own workspaces, running
  concurrently, give each stream the bits it gives alone.
"""
import pytest
import torch

import cake_inputs

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(scope="module")
def cake():
    import __graft_entry__
    __graft_entry__.build()
    import bwd_dw_column_gb300 as cake
    yield cake
    assert cake.cake_rmsnorm_device_status() == 0


@pytest.mark.parametrize("T,H,res", [(4096, 2048, False), (513, 6144, True), (16, 1536, False)])
def test_graph_replay_matches_eager(cake, T, H, res):
    c = (cake_inputs.residual_case(T, H, seed=61, device=DEV) if res
         else cake_inputs.plain_case(T, H, w_dtype=torch.float32, seed=61, device=DEV))
    x, dy, w, r, dh = c["x"], c["dy"], c["w"], c.get("residual"), c.get("dh")
    ws = cake.cake_rmsnorm_bwd_workspace(x, w.dtype, deterministic=True)
    y = torch.empty_like(x)
    rstd = torch.empty(T, dtype=torch.float32, device=DEV)
    hn = torch.empty_like(x) if res else None
    dx = torch.empty_like(x)
    dw = torch.empty(H, dtype=torch.float32, device=DEV)

    def step():
        cake.cake_rmsnorm_fwd(x, w, c["eps"], residual=r, y=y, rstd=rstd, h_new=hn)
        cake.cake_rmsnorm_bwd(dy, hn if res else x, rstd, w, dh, deterministic=True, workspace=ws, dx=dx, dw=dw)

    step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (y, rstd, dx, dw)]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(2):
        for t in (y, rstd, dx, dw):
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for a, b in zip((y, rstd, dx, dw), eager):
            assert torch.equal(a, b)


def test_concurrent_streams(cake):
    cases = [cake_inputs.plain_case(20000, 2048, w_dtype=torch.float32, seed=62, device=DEV),
             cake_inputs.plain_case(30000, 4096, w_dtype=torch.bfloat16, seed=63, device=DEV)]
    outs_alone, outs_together, bufs = [], [], []
    for c in cases:
        _, rstd = cake.cake_rmsnorm_fwd(c["x"], c["w"], c["eps"])
        ws = cake.cake_rmsnorm_bwd_workspace(c["x"], c["w"].dtype, deterministic=True)
        bufs.append((c, rstd, ws))
    torch.cuda.synchronize()
    for c, rstd, ws in bufs:
        dx, dw = cake.cake_rmsnorm_bwd(c["dy"], c["x"], rstd, c["w"], deterministic=True, workspace=ws)
        torch.cuda.synchronize()
        outs_alone.append((dx, dw))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for rep in range(3):
        res = []
        for (c, rstd, ws), s in zip(bufs, streams):
            with torch.cuda.stream(s):
                res.append(cake.cake_rmsnorm_bwd(c["dy"], c["x"], rstd, c["w"], deterministic=True, workspace=ws))
        torch.cuda.synchronize()
        for (dx, dw), (dxa, dwa) in zip(res, outs_alone):
            assert torch.equal(dx, dxa) and torch.equal(dw, dwa)
