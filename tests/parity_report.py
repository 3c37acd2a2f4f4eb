"""Error statistics of every GPU-vs-oracle comparison, recorded per case.

The evaluation page lists what a parity report keeps for each case
("MetaX-TileLang工具链", §2.4: max_abs_err, max_rel_err, num_failed,
element_pass_rate; §2.10: the failing index of a failing case).  Each
comparison made through ``compare`` appends one record; the session prints
them as a table at the end (tests/conftest.py) and, when the environment
variable MOE_PARITY_REPORT names a file, writes them there as JSON.
"""
from __future__ import annotations

import numpy as np

RECORDS: list[dict] = []

# fp16-step distance buckets of the histogram: 0, 1, 2, 3-4, 5-8, 9-16, > 16
ULP_EDGES = (0, 1, 2, 4, 8, 16)
REL_FLOOR = 2.0 ** -10      # relative errors are taken where |oracle| >= this


def _ulp_key(b):
    b = b.astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)


def ulp_histogram(got_bits, ref_bits) -> dict:
    d = np.abs(_ulp_key(np.asarray(got_bits, np.uint16)) - _ulp_key(np.asarray(ref_bits, np.uint16)))
    out, lo = {}, -1
    for hi in ULP_EDGES:
        out[str(hi) if lo + 1 == hi else f"{lo + 1}-{hi}"] = int(np.count_nonzero((d > lo) & (d <= hi)))
        lo = hi
    out[f">{lo}"] = int(np.count_nonzero(d > lo))
    return out


def compare(case: str, what: str, got_bits, ref_bits, atol: float, rtol: float) -> np.ndarray:
    """Elementwise |got - ref| <= atol + rtol·|ref| (and got finite) on fp16 bit
    arrays; records the case's statistics and returns the pass mask."""
    gb = np.ascontiguousarray(got_bits, dtype=np.uint16)
    rb = np.ascontiguousarray(ref_bits, dtype=np.uint16)
    g = gb.view(np.float16).astype(np.float64)
    r = rb.view(np.float16).astype(np.float64)
    err = np.abs(g - r)
    ok = (err <= atol + rtol * np.abs(r)) & np.isfinite(g)
    big = np.abs(r) >= REL_FLOOR
    n = ok.size
    bad = np.flatnonzero(~ok.reshape(-1))
    rec = {
        "case": case, "what": what, "elements": int(n),
        "max_abs_err": float(np.nanmax(err)) if n else 0.0,
        "max_rel_err": float(np.max(err[big] / np.abs(r[big]))) if big.any() else 0.0,
        "median_abs_ref": float(np.median(np.abs(r))) if n else 0.0,
        "num_failed": int(bad.size),
        "element_pass_rate": float(ok.mean()) if n else 1.0,
        "first_failed_index": [int(i) for i in np.unravel_index(bad[0], ok.shape)] if bad.size else None,
        "ulp_histogram": ulp_histogram(gb, rb),
        "atol": atol, "rtol": rtol,
    }
    RECORDS.append(rec)
    return ok
