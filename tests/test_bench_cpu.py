"""The roofline inputs bench.py derives for each workload, on CPU: FLOPs over
valid rows (6·P·H·I), touched-expert weight bytes and activation bytes, against
the per-config figures derived independently from the shapes (P·(2H read +
2H written + 4 + 2I written + 2I read) activation bytes, 6·H·I bytes per
touched expert), with the routing drawn by the workload generator and the
tables from the oracle."""
import numpy as np
import pytest

import bench
import oracle
import workloads

# (pairs, FLOPs, touched weight GB, activation GB, touched experts or None)
EXPECTED = {
    "tiny": (128, 1.007e8, 3.15e-3, 0.39e-3, 4),
    "dsv2_lite": (24576, 4.252e11, 1.107, 0.340, 64),
    "mixtral": (16384, 5.772e12, 2.819, 1.208, 8),
    "dsv3": (131072, 1.1545e13, 22.55, 4.83, 256),
}


@pytest.mark.parametrize("name", sorted(EXPECTED))
def test_roofline_inputs(name):
    w = workloads.WORKLOADS[name]
    pairs, flops, wgb, agb, touched_e = EXPECTED[name]
    assert w.pairs == pairs
    assert w.flops() == pytest.approx(flops, rel=1e-3)
    ids, _ = workloads.routing(w, 0)
    sizes = oracle.build_dispatch(ids, w.experts)["group_sizes"]
    wbytes, act, touched = bench.touched_bytes(w, sizes)
    assert touched == touched_e
    assert wbytes / 1e9 == pytest.approx(wgb, rel=2e-3)
    assert act / 1e9 == pytest.approx(agb, rel=1e-2)


def test_decode_touches_a_subset_of_experts():
    w = workloads.WORKLOADS["decode_skewed"]
    ids, _ = workloads.routing(w, 0)
    sizes = oracle.build_dispatch(ids, w.experts)["group_sizes"]
    wbytes, act, touched = bench.touched_bytes(w, sizes)
    assert touched == int(np.count_nonzero(sizes)) and 40 < touched < w.experts
    assert wbytes == 6.0 * w.hidden * w.intermediate * touched
    assert act == pytest.approx(2.9e6, rel=5e-2)
