"""Pack and combine on the GPU against the oracle, bit for bit.

Pack ("moe_dispatch_contract.py" build_contract: stable sort by expert;
"Fused MoE GEMM 提交说明" §实现要点: padded rows for x, compact rows for the
routed weights): every pair's padded row, the packed activation rows and the
compact routed weights must equal the oracle's exactly, and padding rows of the
packed array stay as the caller filled them.  Combine: an fp32 sum of a
token's k expert rows in j order with one fp16 rounding on both sides, so the
token outputs must also match exactly (same synthetic expert rows on both
sides, drawn by the input generator).
"""
import numpy as np
import pytest
import torch

import oracle
import routed_grouped_gemm_dispatch_gb300 as moe
import workloads
from moe_cases import SENTINEL, small_workload

pytestmark = pytest.mark.gpu


def _pack_both(w, hidden=None, seed=0):
    ids, tw = workloads.routing(w, seed)
    H = hidden or w.hidden
    x = workloads.tokens(w, seed, n_tokens=w.tokens) if hidden is None else \
        np.random.default_rng(seed).standard_normal((w.tokens, H), dtype=np.float32).astype(np.float16)
    tab = oracle.build_dispatch(ids, w.experts)
    prow = oracle.pair_padded_rows(ids, w.experts, tab["group_padded_offsets"])
    rows_total = tab["num_blocks_m"] * 128
    xo, rwo = oracle.pack(x, ids, tw, prow, tab, rows_total, pad_bits=SENTINEL)

    dev = torch.device("cuda")
    ids_d = torch.from_numpy(ids).to(dev)
    t = moe.build_dispatch(ids_d, w.experts)
    stacked = torch.full((rows_total, H), SENTINEL, dtype=torch.int16, device=dev).view(torch.float16)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    pk = moe.pack_routed(ids_d, torch.from_numpy(tw).to(dev), torch.from_numpy(x).to(dev), t,
                         rows_total, stacked=stacked, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return (ids, tw, x, tab, prow, xo, rwo, rows_total,
            pk["pair_padded_rows"].cpu().numpy(),
            pk["stacked_expert_tokens"].view(torch.int16).cpu().numpy().view(np.uint16),
            pk["routed_expert_weights"].cpu().numpy())


@pytest.mark.parametrize("name,hidden", [("tiny", None), ("dsv2_lite", None), ("decode_skewed", None),
                                         ("mixtral", 128), ("dsv3", 128)])
def test_pack_bit_exact(name, hidden):
    w = workloads.WORKLOADS[name]
    ids, tw, x, tab, prow, xo, rwo, rows_total, prow_g, xg, rwg = _pack_both(w, hidden)
    assert np.array_equal(prow_g, prow)
    assert np.array_equal(xg, xo)              # valid rows copied, padding rows untouched
    assert np.array_equal(rwg.view(np.uint32), rwo.view(np.uint32))


@pytest.mark.parametrize("seed", range(4))
def test_pack_random_shapes_bit_exact(seed):
    rng = np.random.default_rng(50 + seed)
    E = int(rng.integers(1, 300))
    k = int(rng.integers(1, min(E, 8) + 1))
    T = int(rng.integers(1, 9000))            # several 4096-pair chunks, ragged tail
    w = small_workload(tokens=T, top_k=k, experts=E, hidden=128, intermediate=128)
    ids, tw, x, tab, prow, xo, rwo, rows_total, prow_g, xg, rwg = _pack_both(w, seed=seed)
    assert np.array_equal(prow_g, prow)
    assert np.array_equal(xg, xo)
    assert np.array_equal(rwg.view(np.uint32), rwo.view(np.uint32))


def test_pack_one_expert_takes_all():
    w = small_workload(tokens=5000, top_k=1, experts=3, hidden=256, intermediate=128)
    ids = np.zeros((5000, 1), np.int32)
    tab = oracle.build_dispatch(ids, 3)
    prow = oracle.pair_padded_rows(ids, 3, tab["group_padded_offsets"])
    ids_d = torch.from_numpy(ids).cuda()
    t = moe.build_dispatch(ids_d, 3)
    pk = moe.pack_routed(ids_d, None, None, t)
    torch.cuda.synchronize()
    assert np.array_equal(pk["pair_padded_rows"].cpu().numpy(), prow)


@pytest.mark.parametrize("name,hidden", [("tiny", None), ("dsv2_lite", None), ("dsv3", 256)])
def test_combine_bit_exact(name, hidden):
    w = workloads.WORKLOADS[name]
    ids, _ = workloads.routing(w, 0)
    tab = oracle.build_dispatch(ids, w.experts)
    prow = oracle.pair_padded_rows(ids, w.experts, tab["group_padded_offsets"])
    rows_total = tab["num_blocks_m"] * 128
    H = hidden or w.hidden
    out = (np.random.default_rng(3).standard_normal((rows_total, H), dtype=np.float32) * 0.3).astype(np.float16)
    y_o = oracle.combine(out, prow, w.tokens, w.top_k)
    y_g = moe.combine_routed(torch.from_numpy(out).cuda(), torch.from_numpy(prow).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(y_g.view(torch.int16).cpu().numpy().view(np.uint16), y_o)


def test_pack_flags_bad_ids_and_checks_workspace():
    ids = torch.tensor([[0, 1], [7, 2]], dtype=torch.int32, device="cuda")
    good = torch.tensor([[0, 1], [3, 2]], dtype=torch.int32, device="cuda")
    t = moe.build_dispatch(good, 4)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pk = moe.pack_routed(ids, None, None, t, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & moe.MOE_DEV_BAD_EXPERT_ID
    assert int(pk["pair_padded_rows"][1, 0].item()) == -1
    small = torch.empty(8, dtype=torch.uint8, device="cuda")
    with pytest.raises(moe.MoeError):
        moe.pack_routed(good, None, None, t, workspace=small)
