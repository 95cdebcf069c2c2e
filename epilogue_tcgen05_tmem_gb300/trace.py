"""Summaries of the per-CTA timelines the kernel records (eg_plan_set_trace).

Each CTA writes EG_TRACE_POINTS %globaltimer stamps (ns): start, setup done,
first TMA issued (after any wait on the previous kernel), first UMMA
operands ready, last UMMA committed, first accumulator ready in the
epilogue, epilogue done, end; then the first weight loads issued (before
the wait on the previous kernel), the last load issued, and for the CTA's
last work unit the accumulator final, the split-K partial stored or sent,
the arrival counted or partials received, and the start of the output
stores.  Unwritten points stay at the buffer's fill value (0).
"""
from __future__ import annotations

import numpy as np

from . import TRACE_POINT_NAMES


def summarize(trace: np.ndarray, t0: int | None = None) -> dict:
    """Percentiles (in microseconds, relative to t0 or the earliest CTA
    start) of every trace point over the CTAs that recorded it."""
    t = np.asarray(trace, dtype=np.int64)
    starts = t[:, 0][t[:, 0] > 0]
    if starts.size == 0:
        return {}
    base = int(starts.min()) if t0 is None else int(t0)
    out = {}
    for i, name in enumerate(TRACE_POINT_NAMES):
        col = t[:, i]
        col = col[col > 0]
        if col.size:
            rel = (col - base) / 1e3
            out[name] = {"p0": round(float(rel.min()), 3), "p50": round(float(np.median(rel)), 3),
                         "p100": round(float(rel.max()), 3), "ctas": int(col.size)}
    return out


def ordered(trace: np.ndarray) -> bool:
    """Every CTA's recorded points are non-decreasing in pipeline order
    (start <= setup <= first TMA <= first operands <= last commit, and
    first accumulator <= epilogue done <= end)."""
    t = np.asarray(trace, dtype=np.int64)
    for row in t:
        if row[0] == 0:
            continue
        chain1 = [row[i] for i in (0, 1, 2, 3, 4) if row[i] > 0]
        chain2 = [row[i] for i in (1, 5, 6, 7) if row[i] > 0]
        if any(b < a for a, b in zip(chain1, chain1[1:])) or \
           any(b < a for a, b in zip(chain2, chain2[1:])):
            return False
    return True
