"""Failure detection without a GPU fault: a bounded wait that runs out.

With MOE_TEST_DROP_SIGNAL, phase 1's MMA issuer withholds its first
"accumulator ready" signal, so the epilogue's wait on it (bounded at 2 s) runs
out.  The kernel must then stop by itself: drain its copies and MMAs, free
its tensor memory, report MOE_DEV_TIMEOUT in the status word — and leave the
context usable, so that the next ordinary call is correct.
"""
import numpy as np
import pytest
import torch

import routed_grouped_gemm_dispatch_gb300 as moe
from gpu_side import bits, gpu_prepare, run_forward, sentinel
from moe_cases import raw_inputs, small_workload

pytestmark = pytest.mark.gpu


def test_timed_out_wait_reports_and_context_survives():
    w = small_workload(tokens=300, top_k=2, experts=3, hidden=256, intermediate=384)
    side = gpu_prepare(raw_inputs(w, seed=9))
    ul_ref, out_ref = run_forward(side, w.intermediate)
    torch.cuda.synchronize()

    t = side.tables
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ul = sentinel(side.rows_total, w.intermediate)
    out = sentinel(side.rows_total, w.hidden)
    moe.fused_forward(side.x_packed, side.gate, side.up, side.down, side.rw, t["group_sizes"],
                      t["group_offsets"], t["group_padded_offsets"], t["group_idx_for_bx"], ul, out,
                      status=status,
                      flags=moe.MOE_RUN_PHASE1 | moe.MOE_RUN_PHASE2 | moe.MOE_TEST_DROP_SIGNAL)
    torch.cuda.synchronize()                     # returns: no hang, no fault
    assert int(status.item()) & moe.MOE_DEV_TIMEOUT

    status.zero_()
    ul2, out2 = run_forward(side, w.intermediate, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(bits(out2), bits(out_ref))
    assert np.array_equal(bits(ul2), bits(ul_ref))
