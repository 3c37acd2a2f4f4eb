"""GPU dispatch-table builder against the oracle: bit-exact.

Tables per "moe_dispatch_contract.py" (TileLang tutorial, ch. 18), built by
``moe_build_dispatch`` on the device and compared entry by entry with the
oracle's tables for the same topk_ids.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import routed_grouped_gemm_dispatch_gb300 as moe
import workloads

pytestmark = pytest.mark.gpu

KEYS = ("group_sizes", "group_offsets", "group_padded_offsets", "group_idx_for_bx")


def _gpu_tables(ids_np, E, status=None):
    ids = torch.from_numpy(np.ascontiguousarray(ids_np, dtype=np.int32)).cuda()
    t = moe.build_dispatch(ids, E, status=status)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in t.items()}


def _assert_equal(ids_np, E):
    g = _gpu_tables(ids_np, E)
    o = oracle.build_dispatch(ids_np, E)
    for k in KEYS:
        assert np.array_equal(g[k], o[k]), k


def test_golden_cases(golden_dir):
    with open(os.path.join(golden_dir, "dispatch_tables.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        if "topk_ids" in case:
            ids = np.array(case["topk_ids"], np.int32)
        else:
            ids = np.array(sum(([e] * n for e, n in case["topk_ids_runs"]), []), np.int32).reshape(-1, 1)
        g = _gpu_tables(ids, case["n_experts"])
        for k in KEYS:
            assert g[k].tolist() == case[k], (case["name"], k)


@pytest.mark.parametrize("name", list(workloads.WORKLOADS))
def test_workload_routing_bit_exact(name):
    w = workloads.WORKLOADS[name]
    ids, _ = workloads.routing(w, seed=0)
    _assert_equal(ids, w.experts)


@pytest.mark.parametrize("seed", range(6))
def test_random_shapes_bit_exact(seed):
    rng = np.random.default_rng(100 + seed)
    E = int(rng.integers(1, 300))
    k = int(rng.integers(1, min(E, 8) + 1))
    T = int(rng.integers(0, 5000))
    keys = rng.random((T, E))
    ids = np.argsort(keys, axis=1)[:, :k].astype(np.int32)
    _assert_equal(ids, E)


def test_edge_cases_bit_exact():
    _assert_equal(np.zeros((0, 4), np.int32), 7)                  # no tokens
    _assert_equal(np.zeros((1, 1), np.int32), 1)                  # one pair, one expert
    _assert_equal(np.zeros((1280, 1), np.int32), 4)               # 10 full blocks -> +1 rule
    _assert_equal(np.full((127, 1), 3, np.int32), 4)              # count+1 == 128
    ids = np.arange(1024 * 3, dtype=np.int32).reshape(-1, 1) % 1024
    _assert_equal(ids, 1024)                                      # maximum experts
    rng = np.random.default_rng(9)
    big = rng.integers(0, 256, size=(200_000, 8)).astype(np.int32)  # 1.6M pairs (not distinct: counted anyway)
    _assert_equal(big, 256)


def test_out_of_range_ids_flagged():
    ids = np.array([[0, 1], [5, 2], [-1, 3]], np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = _gpu_tables(ids, 4, status=status)
    assert int(status.item()) & moe.MOE_DEV_BAD_EXPERT_ID
    assert g["group_sizes"].tolist() == [1, 1, 1, 1]


def test_host_validation():
    ids = torch.zeros((4, 2), dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError):
        moe.build_dispatch(ids, 4, block_token=64)
    with pytest.raises(moe.MoeError):
        moe.build_dispatch(ids, 4096)
