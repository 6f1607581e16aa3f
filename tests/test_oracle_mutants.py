"""The oracle's pins catch plausible mistakes.

Each case below plants one mistake in a copy of ``oracle/cake_oracle.c`` (a
dropped term, a wrong sign, a wrong index or stride, a skipped rounding),
builds the copy, points the oracle module at it and runs every pin in
``tests/test_oracle.py``: at least one pin must fail.  The unchanged source
run through the same harness must pass them all.  Everything here runs on the
CPU; the mutants never leave the test's temporary directory.
"""
import inspect
import itertools
import os
import subprocess

import pytest

import oracle
from tests import test_oracle as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "cake_oracle.c")

# name: (text in the oracle source, replacement)
MUTANTS = {
    "mean square without 1/H": ("double ms = ss / (double)H;", "double ms = ss;"),
    "eps outside the root": ("return 1.0 / sqrt(ms + eps);", "return 1.0 / sqrt(ms) + eps;"),
    "dx sign flip": ("dx[j] = rs * (g - xh * c)", "dx[j] = rs * (g + xh * c)"),
    "row dot without 1/H": ("    c /= (double)H;\n", "\n"),
    "dx without the leading rstd": ("dx[j] = rs * (g - xh * c)", "dx[j] = (g - xh * c)"),
    "dh dropped": ("+ (dh ? dh[j] : 0.0)", "+ 0.0"),
    "y without w": ("y[j] = h[j] * rs * w[j];", "y[j] = h[j] * rs;"),
    "y ignores the given rstd": ("row_y(h, wd, H, rstd_in ? (double)rstd_in[r] : r64, y + i * H);",
                                "row_y(h, wd, H, r64, y + i * H);"),
    "w read at one index": ("wd[j] = weight_at(w, w_is_f32, j);\n    for (int64_t i = 0; i < nrows; ++i) {\n"
                            "        int64_t r = rows ? rows[i] : i;\n        if (r < 0 || r >= T * nh)\n"
                            "            return 2;\n        load_row(dy",
                            "wd[j] = weight_at(w, w_is_f32, 0);\n    for (int64_t i = 0; i < nrows; ++i) {\n"
                            "        int64_t r = rows ? rows[i] : i;\n        if (r < 0 || r >= T * nh)\n"
                            "            return 2;\n        load_row(dy"),
    "dw without rstd (BF16 views)": ("dw[i] += bf16_to_f64(dyr[j]) * bf16_to_f64(hr[j]) * rs;",
                                     "dw[i] += bf16_to_f64(dyr[j]) * bf16_to_f64(hr[j]);"),
    "dw without rstd (FP64 rows)": ("s += dy[r * H + j] * h[r * H + j] * rstd[r];", "s += dy[r * H + j] * h[r * H + j];"),
    "dw with dx's w": ("s += dy[r * H + j] * h[r * H + j] * rstd[r];", "s += dy[r * H + j] * w[j] * h[r * H + j] * rstd[r];"),
    "head and token strides swapped": ("return t * st + k * sh;", "return t * sh + k * st;"),
    "BF16 rounding truncates": ("double r = nearbyint(ldexp(a, -q));", "double r = trunc(ldexp(a, -q));"),
    "residual sum not rounded to BF16": ("h[j] = bf16_to_f64(b);", "h[j] = h[j] + tmp[j];"),
}


def _cases(fn):
    """Every argument combination of a (possibly parametrized) pin."""
    marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
    combos = [{}]
    for m in marks:
        names = [n.strip() for n in m.args[0].split(",")] if isinstance(m.args[0], str) else list(m.args[0])
        new = []
        for c, v in itertools.product(combos, m.args[1]):
            v = v if len(names) > 1 else (v,)
            new.append({**c, **dict(zip(names, v))})
        combos = new
    return combos


def _run_pins():
    """Run every pin; return the names of those that failed."""
    failed = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        for kw in _cases(fn):
            try:
                fn(**kw)
            except Exception:  # an assertion, or an error the mistake provoked
                failed.append(name)
                break
    return failed


def _build(src_text, tmp_path, tag):
    c = tmp_path / f"oracle_{tag}.c"
    so = tmp_path / f"liboracle_{tag}.so"
    c.write_text(src_text)
    subprocess.check_call(["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-std=c99", "-fPIC", "-shared",
                           "-o", str(so), str(c), "-lm"])
    return str(so)


def _use(monkeypatch, path):
    monkeypatch.setattr(oracle, "build", lambda force=False: path)
    monkeypatch.setattr(oracle, "_lib", None)


def test_unchanged_source_passes_every_pin(tmp_path, monkeypatch):
    _use(monkeypatch, _build(open(SRC).read(), tmp_path, "same"))
    assert _run_pins() == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) >= 1, f"the oracle source no longer contains the text this case mutates: {old!r}"
    _use(monkeypatch, _build(text.replace(old, new, 1), tmp_path, "m"))
    failed = _run_pins()
    assert failed, f"no pin caught the planted mistake: {name}"
