"""Pins for the oracle's dispatch tables.

Pinned against (a) hand-derived examples in tests/golden/dispatch_tables.json,
(b) the three invariants that "moe_dispatch_contract.py" (TileLang tutorial,
ch. 18) checks — every (token, expert) pair exactly once, each padded range
covers its compact range, the kernel's m_start / actual_rows stay inside the
compact range — plus closed forms of the padding rule, and (c) a token-by-token
brute force on random small inputs.
"""
import bisect
import json
import math
import os

import numpy as np
import pytest

import oracle
import workloads

BT = 128


def _ids_from_case(case):
    if "topk_ids" in case:
        return np.array(case["topk_ids"], np.int32)
    ids = []
    for e, n in case["topk_ids_runs"]:
        ids += [e] * n
    return np.array(ids, np.int32).reshape(-1, 1)


def _actual_rows(t, bx):
    e = t["group_idx_for_bx"][bx]
    off = bx * BT - t["group_padded_offsets"][e]
    return max(0, min(BT, int(t["group_sizes"][e]) - off))


def _golden_cases(golden_dir):
    with open(os.path.join(golden_dir, "dispatch_tables.json")) as f:
        return json.load(f)["cases"]


def test_golden_cases(golden_dir):
    for case in _golden_cases(golden_dir):
        ids = _ids_from_case(case)
        t = oracle.build_dispatch(ids, case["n_experts"])
        for k in ("group_sizes", "group_offsets", "group_padded_offsets", "group_idx_for_bx"):
            assert t[k].tolist() == case[k], (case["name"], k)
        assert t["num_blocks_m"] == case["num_blocks_m"]
        assert [_actual_rows(t, bx) for bx in range(t["num_blocks_m"])] == case["actual_rows"]
        if "pair_rows" in case:
            rows = oracle.pair_padded_rows(ids, case["n_experts"], t["group_padded_offsets"])
            assert rows.tolist() == case["pair_rows"]


def _brute_force(ids, E):
    """Token-by-token recount; bisect for the block map; a Python stable sort
    for the pair order."""
    flat = [int(v) for v in ids.reshape(-1)]
    counts = [0] * E
    for e in flat:
        counts[e] += 1
    offsets = [sum(counts[:e]) for e in range(E + 1)]
    steps = [((c + 1 + BT - 1) // BT) * BT for c in counts]
    padded = [sum(steps[:e]) for e in range(E + 1)]
    m = -(-len(flat) // BT) + E
    gidx = [bisect.bisect_right(padded[:E], bx * BT) - 1 for bx in range(m)]
    order = sorted(range(len(flat)), key=lambda f: flat[f])
    rows = [0] * len(flat)
    seen = [0] * E
    for f in order:
        e = flat[f]
        rows[f] = padded[e] + seen[e]
        seen[e] += 1
    return counts, offsets, padded, m, gidx, rows


@pytest.mark.parametrize("seed", range(12))
def test_against_brute_force(seed):
    rng = np.random.default_rng(seed)
    E = int(rng.integers(1, 40))
    k = int(rng.integers(1, min(E, 8) + 1))
    T = int(rng.integers(0, 300))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32) \
        if T else np.zeros((0, k), np.int32)
    t = oracle.build_dispatch(ids, E)
    counts, offsets, padded, m, gidx, rows = _brute_force(ids, E)
    assert t["group_sizes"].tolist() == counts
    assert t["group_offsets"].tolist() == offsets
    assert t["group_padded_offsets"].tolist() == padded
    assert t["num_blocks_m"] == m
    assert t["group_idx_for_bx"].tolist() == gidx
    got_rows = oracle.pair_padded_rows(ids, E, t["group_padded_offsets"])
    assert got_rows.reshape(-1).tolist() == rows


def _check_contract_invariants(ids, E, t, rows):
    """The three checks of moe_dispatch_contract.py, plus closed forms."""
    P = ids.size
    sizes, offs, padded, gidx = (t["group_sizes"], t["group_offsets"],
                                 t["group_padded_offsets"], t["group_idx_for_bx"])
    flat = ids.reshape(-1)
    # 1) each (token, expert) pair exactly once; sum of sizes = pairs
    assert int(sizes.sum()) == P
    pairs = {(f // ids.shape[1], int(flat[f])) for f in range(P)}
    assert len(pairs) == P
    rl = rows.reshape(-1)
    assert len(set(rl.tolist())) == P
    for f in range(P):
        e = flat[f]
        assert padded[e] <= rl[f] < padded[e] + sizes[e]
    # 2) padded range covers compact range, closed form of the step
    for e in range(E):
        step = int(padded[e + 1] - padded[e])
        assert step == math.ceil((int(sizes[e]) + 1) / BT) * BT
        assert step >= sizes[e] + 1 and step % BT == 0
        assert offs[e + 1] - offs[e] == sizes[e]
    assert offs[0] == 0 and padded[0] == 0 and offs[E] == P
    assert t["num_blocks_m"] * BT >= padded[E]
    # 3) m_start / actual_rows in bounds for every block
    covered = np.zeros(P, np.int32)
    for bx, g in enumerate(gidx):
        assert 0 <= g < E
        start = bx * BT
        assert start >= padded[g]
        if g < E - 1:
            assert start < padded[g + 1]
        m_start = start - padded[g] + offs[g]
        ar = _actual_rows(t, bx)
        if ar > 0:
            assert m_start >= offs[g]
            assert m_start + ar <= offs[g] + sizes[g]
            covered[m_start:m_start + ar] += 1
    # every compact row is reached by exactly one block
    assert np.all(covered == 1)


@pytest.mark.parametrize("name", ["tiny", "dsv2_lite", "decode_skewed", "mixtral"])
def test_invariants_on_workload_routing(name):
    w = workloads.WORKLOADS[name]
    ids, _ = workloads.routing(w, seed=0)
    t = oracle.build_dispatch(ids, w.experts)
    rows = oracle.pair_padded_rows(ids, w.experts, t["group_padded_offsets"])
    _check_contract_invariants(ids, w.experts, t, rows)


def test_invariants_degenerate():
    # no tokens at all: every expert owns one empty block
    ids = np.zeros((0, 2), np.int32)
    t = oracle.build_dispatch(ids, 5)
    assert t["num_blocks_m"] == 5
    assert t["group_padded_offsets"].tolist() == [0, 128, 256, 384, 512, 640]
    assert t["group_idx_for_bx"].tolist() == [0, 1, 2, 3, 4]
    # one expert takes everything
    ids = np.zeros((1000, 1), np.int32)
    t = oracle.build_dispatch(ids, 3)
    assert t["group_sizes"].tolist() == [1000, 0, 0]
    assert t["group_padded_offsets"].tolist() == [0, 1024, 1152, 1280]
    rows = oracle.pair_padded_rows(ids, 3, t["group_padded_offsets"])
    _check_contract_invariants(ids, 3, t, rows)


def test_rejects_out_of_range_ids():
    with pytest.raises(ValueError):
        oracle.build_dispatch(np.array([[0, 4]], np.int32), 4)
    with pytest.raises(ValueError):
        oracle.build_dispatch(np.array([[-1, 0]], np.int32), 4)
