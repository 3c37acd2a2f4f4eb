"""The MOE_DEBUG build, the stand-in for a sanitizer where none can run: its kernels
also check their own tile indices, TMA coordinates, store bounds, table
invariants and a shared-memory canary, and report a failed check as
MOE_DEV_DEBUG_CHECK.  On every case of debug_build_cases.py it raises no check
and produces, bit for bit, the release build's tables, packing, forward (both
launch forms), combine and router outputs."""
import os
import subprocess
import sys

import numpy as np
import pytest

import routed_grouped_gemm_dispatch_gb300 as moe

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_debug_build_matches_release_and_raises_no_check(tmp_path):
    import debug_build_cases
    moe.build(debug=True)
    out = tmp_path / "debug.npz"
    env = dict(os.environ, MOE_GB300_DEBUG="1",
               PYTHONPATH=os.pathsep.join([ROOT, HERE, os.environ.get("PYTHONPATH", "")]))
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_build_cases.py"), str(out)], cwd=HERE,
                       env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    dbg = np.load(out)
    rel = debug_build_cases.run_cases()
    assert set(dbg.files) == set(rel)
    for key in sorted(rel):
        if key.endswith("/status"):
            assert not np.any(dbg[key]), (key, dbg[key])
            assert not np.any(rel[key]), (key, rel[key])
        else:
            assert np.array_equal(dbg[key], rel[key]), key
