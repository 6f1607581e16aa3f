"""The pages' own constants (tests/golden/pages_constants.txt, each line cited)
against the synthetic workloads and the tolerances the parity tests use."""
import os

import torch

import cake_inputs
from tests import tolerances

HERE = os.path.dirname(os.path.abspath(__file__))


def _golden():
    out = {}
    with open(os.path.join(HERE, "golden", "pages_constants.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = (s.strip() for s in line.split("=", 1))
                out[k] = v
    return out


def test_tolerances_are_the_pages():
    g = _golden()
    assert float(g["eps"]) == cake_inputs.EPS
    assert float(g["dw_atol"]) == tolerances.DW_ATOL
    assert float(g["dw_rtol"]) == tolerances.DW_RTOL
    assert int(g["accuracy_inputs_per_family"]) == cake_inputs.SWEEP_SEEDS


def test_per_head_views_have_the_pages_strides():
    g = _golden()
    nh, d = (int(v) for v in g["query_view_shape"].split(","))
    strides = tuple(int(v) for v in g["query_view_strides"].split(","))
    case = cake_inputs.heads_case(3, nh, strided=True, seed=0)
    assert tuple(case["x"].shape[1:]) == (nh, d)
    assert case["x"].stride() == strides
    assert case["w"].shape == (int(g["head_dim"]),)
    knh, kd = (int(v) for v in g["key_view_shape"].split(","))
    kcase = cake_inputs.heads_case(3, knh, strided=False, seed=0)
    assert tuple(kcase["x"].shape[1:]) == (knh, kd) and kcase["x"].is_contiguous()


def test_workload_shapes():
    g = _golden()
    hidden = {int(v) for v in g["hidden_sizes"].split(",")}
    for name, spec in cake_inputs.WORKLOADS.items():
        if spec["kind"] in ("plain", "res"):
            assert spec["H"] in hidden, name
    assert cake_inputs.WORKLOADS["h6144_t131072_res"]["H"] == int(g["residual_hidden"])


def test_outlier_family_scales_one_percent_of_rows():
    c = cake_inputs.plain_case(1000, 64, family="outlier", seed=3)
    rms = c["x"].float().pow(2).mean(dim=1).sqrt()
    assert int((rms > 10).sum()) == 10
    c2 = cake_inputs.plain_case(1000, 64, family="outlier", seed=3)
    assert torch.equal(c["x"], c2["x"])
