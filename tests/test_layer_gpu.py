"""The whole MoE layer on the GPU against the oracle chain: router -> dispatch
tables -> pack -> fused forward -> combine ("MetaX-TileLang工具链" §2.4 for
the router and the layer; "Fused MoE GEMM 提交说明" for the forward).

The GPU router's choices feed both chains, so a near-tie that the two routers
break differently cannot make the chains diverge; the routers themselves are
compared where the k-th and (k+1)-th logits are clearly apart.  A token's
output is the fp32 sum of its k expert rows, each within 2e-2 + 2e-2·|oracle|,
so y is compared within k·2e-2 + 2e-2·Σ_j |oracle row j|."""
import numpy as np
import pytest
import torch

import oracle
import routed_grouped_gemm_dispatch_gb300 as moe
import workloads
from moe_cases import small_workload

pytestmark = pytest.mark.gpu


def _f16(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


@pytest.mark.parametrize("w", [
    workloads.WORKLOADS["tiny"],
    small_workload(tokens=300, top_k=6, experts=40, hidden=256, intermediate=384),
    small_workload(tokens=129, top_k=1, experts=8, hidden=384, intermediate=256),
], ids=["tiny", "e40_k6", "e8_k1"])
def test_router_to_combine_matches_oracle(w):
    x = workloads.tokens(w, 7)
    wg = workloads.router_weights(w, 7)
    gate, up, down = workloads.expert_weights(w, 7, device="cpu")
    gate, up, down = gate.numpy(), up.numpy(), down.numpy()
    dev = torch.device("cuda")

    # router: GPU vs oracle on the clear cases
    x_d = torch.from_numpy(x).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ids_d, tw_d = moe.router_topk(x_d, torch.from_numpy(wg).to(dev), w.top_k, status=status)
    ids_g, tw_g = ids_d.cpu().numpy(), tw_d.cpu().numpy()
    ids_o, tw_o = oracle.router(x, wg, w.top_k)
    lg = x.astype(np.float64) @ wg.astype(np.float64).T
    srt = -np.sort(-lg, axis=1)
    clear = np.ones(w.tokens, bool) if w.top_k == w.experts else \
        (srt[:, w.top_k - 1] - srt[:, w.top_k]) > 1e-3
    assert clear.mean() > 0.9
    assert np.array_equal(ids_g[clear], ids_o[clear])
    assert np.allclose(tw_g[clear], tw_o[clear], rtol=5e-5, atol=1e-7)

    # the GPU chain
    t = moe.build_dispatch(ids_d, w.experts, status=status)
    rows_total = t["group_idx_for_bx"].numel() * 128
    pk = moe.pack_routed(ids_d, tw_d, x_d, t, rows_total, status=status)
    ul = torch.zeros((rows_total, w.intermediate), dtype=torch.float16, device=dev)
    out = torch.zeros((rows_total, w.hidden), dtype=torch.float16, device=dev)
    g_d, u_d, d_d = (torch.from_numpy(a).to(dev) for a in (gate, up, down))
    moe.fused_forward(pk["stacked_expert_tokens"], g_d, u_d, d_d, pk["routed_expert_weights"],
                      t["group_sizes"], t["group_offsets"], t["group_padded_offsets"],
                      t["group_idx_for_bx"], ul, out, status=status)
    y_g = moe.combine_routed(out, pk["pair_padded_rows"])
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    y_g = y_g.view(torch.int16).cpu().numpy().view(np.uint16)

    # the oracle chain on the same routing
    tab = oracle.build_dispatch(ids_g, w.experts)
    prow = oracle.pair_padded_rows(ids_g, w.experts, tab["group_padded_offsets"])
    xo, rwo = oracle.pack(x, ids_g, tw_g, prow, tab, tab["num_blocks_m"] * 128)
    _, out_o = oracle.fused_forward(xo, gate, up, down, rwo, tab)
    y_o = oracle.combine(out_o, prow, w.tokens, w.top_k)

    assert np.array_equal(pk["pair_padded_rows"].cpu().numpy(), prow)
    rows_abs = np.abs(_f16(out_o))[prow.reshape(-1)].reshape(w.tokens, w.top_k, w.hidden).sum(axis=1)
    err = np.abs(_f16(y_g) - _f16(y_o))
    assert np.all(np.isfinite(_f16(y_g)))
    assert np.all(err <= w.top_k * 2e-2 + 2e-2 * rows_abs + 1e-3 * np.abs(_f16(y_o)))
