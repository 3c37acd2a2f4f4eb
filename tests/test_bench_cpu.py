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


def test_default_workload_is_the_largest():
    args = bench.parse_args([])
    assert args.workload == "dsv3"
    big = max(workloads.WORKLOADS.values(), key=lambda w: w.flops())
    assert big.name == args.workload


def test_padding_statistics_by_hand():
    """Three experts with 0, 128 and 300 rows: the "+1" rule pads them to 128,
    256 and 384 rows; their active blocks are 0, 1 and 3; the 2-SM tiles are
    0, 1 (a lone block, 128 rows) and 2 (a pair, 256 rows, plus a lone block)."""
    w = workloads.Workload("hand", 107, 4, 3, 256, 512)
    assert w.pairs == 428
    s = bench.work_stats(w, np.array([0, 128, 300]))
    assert s["padded_rows"] == 128 + 256 + 384
    assert s["active_blocks"] == 4 and s["tile_units"] == 3
    assert s["executed_mma_rows"] == 128 + 256 + 128
    assert s["alloc_rows"] == (4 + 3) * 128
    assert s["padding_waste_rows"] == 7 * 128 - 428
    assert s["padded_minus_valid_rows"] == 768 - 428
    assert s["touched_experts"] == 2
    assert s["flops_phase1"] + s["flops_phase2"] == w.flops()
    assert s["activation_bytes"] == s["activation_bytes_phase1"] + s["activation_bytes_phase2"]
    assert s["activation_bytes"] - s["activation_bytes_no_up_logits"] == 428 * 4 * 512


@pytest.mark.parametrize("name,bound1", [("dsv3", "tensor"), ("mixtral", "tensor"), ("decode_skewed", "hbm")])
def test_kernel_bound_follows_its_own_times(name, bound1):
    """Phase 1's bound is the larger of its FLOP time and byte time at the
    peaks: the compute-heavy shapes are tensor-bound, the decode shape (a few
    rows per expert, every touched expert's weights streamed once) HBM-bound,
    and the fraction is then reported in GB/s against the HBM peak."""
    w = workloads.WORKLOADS[name]
    ids, _ = workloads.routing(w, 0)
    s = bench.work_stats(w, oracle.build_dispatch(ids, w.experts)["group_sizes"])
    r = bench.kernel_roofline("p1", s["flops_phase1"], s["weight_bytes_phase1"] + s["activation_bytes_phase1"],
                              1.0, 1700.0, 6700.0, "test")
    assert r["bound"] == bound1
    if bound1 == "hbm":
        assert r["unit"] == "GB/s" and r["achieved"] == pytest.approx(r["algorithmic_bytes_per_launch"] / 1e6)
    else:
        assert r["unit"] == "TFLOP/s" and r["achieved"] == pytest.approx(s["flops_phase1"] / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])
