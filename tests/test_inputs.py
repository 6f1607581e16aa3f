"""The seeded input generators (shared by the oracle tests and the GPU
tests; they hold none of the method's arithmetic): each family has the
statistics its recipe states and the same seed gives the same bits."""
import torch

import cake_inputs


def test_rowmean_family_recipe():
    """Per-row random mean: each row centred on its own 3 + N(0, 1)."""
    g = torch.Generator().manual_seed(4)
    x = cake_inputs.rows_input(2000, 512, "rowmean", g)
    xf = x.float()
    m = xf.mean(dim=1)
    assert abs(float(m.mean()) - 3.0) < 0.1 and abs(float(m.std()) - 1.0) < 0.1
    assert abs(float((xf - m[:, None]).std()) - 1.0) < 0.02
    assert torch.equal(cake_inputs.rows_input(2000, 512, "rowmean", torch.Generator().manual_seed(4)), x)


def test_offset_and_outlier_recipes():
    x = cake_inputs.rows_input(3000, 256, "offset", torch.Generator().manual_seed(1)).float()
    assert abs(float(x.mean()) - 3.0) < 0.01 and abs(float(x.std()) - 1.0) < 0.01
    x = cake_inputs.rows_input(3000, 256, "outlier", torch.Generator().manual_seed(1)).float()
    big = (x.abs().amax(dim=1) > 20).sum()
    assert int(big) == 30  # ceil(1 % of 3000) rows scaled by 30
