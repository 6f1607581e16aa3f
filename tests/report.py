"""Per-case accuracy records of the GPU parity tests.

Every parity check records what it measured against the oracle -- the dx
counts of ``tolerances.dx_report`` (strict 1-ulp violations, those beyond the
FP32-evaluation allowance, those off cancellation, the largest distance in
BF16 steps) and the worst dw element as a fraction of its budget -- so that a
passing run still shows how close each case came to its bar.  The session
prints them as a table at the end and, when CAKE_PARITY_REPORT names a file,
writes them there as JSON.
"""
from __future__ import annotations

import os

RECORDS: list[dict] = []


def record(case: str, **fields):
    """Add one case's measurements (plain numbers and strings)."""
    RECORDS.append({"case": case, **fields})


def write(path: str | None = None):
    import json

    path = path or os.environ.get("CAKE_PARITY_REPORT")
    if not path or not RECORDS:
        return None
    with open(path, "w") as f:
        json.dump(RECORDS, f, indent=1)
    return path


def summary_lines() -> list[str]:
    if not RECORDS:
        return []
    lines = [f"{'case':60} {'dx n':>11} {'max_ulp':>7} {'strict':>7} {'bounded':>7} {'off_canc':>8} {'dw/budget':>9}"]
    for r in RECORDS:
        dx = r.get("dx", {})
        lines.append(f"{r['case'][:60]:60} {dx.get('n', 0):>11} {dx.get('max_ulp', 0):>7} {dx.get('strict', 0):>7} "
                     f"{dx.get('bounded', 0):>7} {dx.get('off_cancellation', 0):>8} {r.get('dw_worst', 0.0):>9.4f}")
    return lines
