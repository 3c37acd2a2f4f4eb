import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a GB300 (sm_103a) and the compiled CUDA library")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


def pytest_terminal_summary(terminalreporter):
    """Print the parity statistics the GPU tests recorded (and write them as
    JSON to $MOE_PARITY_REPORT when that is set)."""
    import json

    import parity_report
    recs = parity_report.RECORDS
    if not recs:
        return
    path = os.environ.get("MOE_PARITY_REPORT")
    if path:
        with open(path, "w") as f:
            json.dump(recs, f, indent=1)
    tr = terminalreporter
    tr.write_sep("-", f"parity: {len(recs)} comparisons against the oracle")
    for r in recs:
        h = r["ulp_histogram"]
        tr.write_line(f"{r['case'][:44]:44s} {r['what']:9s} n={r['elements']:<10d} "
                      f"max_abs={r['max_abs_err']:.2e} max_rel={r['max_rel_err']:.2e} "
                      f"failed={r['num_failed']} pass={r['element_pass_rate']:.6f} "
                      f"ulp<=1:{(h['0'] + h['1']) / max(1, r['elements']):.4f}")
