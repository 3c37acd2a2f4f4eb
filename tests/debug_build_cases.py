"""Cases that tests/test_debug_build_gpu.py runs twice: in the test process with
the release library, and in a child process started with MOE_GB300_DEBUG=1,
which loads the MOE_DEBUG build (kernels that also check their own indices,
coordinates and shared-memory canary and report MOE_DEV_DEBUG_CHECK).  Every
output and every status word goes into one .npz per run.

    python debug_build_cases.py OUT.npz
"""
import sys

import numpy as np
import torch

import routed_grouped_gemm_dispatch_gb300 as moe
import workloads
from gpu_side import bits, sentinel
from moe_cases import BT, raw_inputs, small_workload

CASES = [
    ("tiny", None),
    ("small_ragged", dict(tokens=300, top_k=2, experts=3, hidden=256, intermediate=384)),
    ("small_zipf", dict(tokens=32, top_k=8, experts=128, hidden=256, intermediate=256, routing="zipf",
                        zipf_s=1.2)),
    ("one_expert", dict(tokens=700, top_k=1, experts=2, hidden=512, intermediate=640, routing="zipf",
                        zipf_s=1.2)),
    ("decode_skewed", None),
    ("dsv2_lite", None),
]


def run_cases():
    res = {}
    for name, kw in CASES:
        w = workloads.WORKLOADS[name] if kw is None else small_workload(**kw)
        raw = raw_inputs(w, seed=3)
        st = torch.zeros(4, dtype=torch.int32, device="cuda")   # dispatch, pack, forward, single launch
        ids = torch.from_numpy(np.ascontiguousarray(raw.topk_ids)).cuda()
        t = moe.build_dispatch(ids, w.experts, status=st[0:1])
        x = torch.from_numpy(np.ascontiguousarray(raw.x_tokens)).cuda()
        tw = torch.from_numpy(np.ascontiguousarray(raw.topk_weights)).cuda()
        rows_total = t["group_idx_for_bx"].numel() * BT
        pk = moe.pack_routed(ids, tw, x, t, rows_total, status=st[1:2])
        g, u, d = (torch.from_numpy(a).cuda() for a in (raw.gate, raw.up, raw.down))
        outs = []
        for i, single in enumerate((None, torch.empty(
                moe.single_launch_workspace_bytes(t["group_idx_for_bx"].numel()), dtype=torch.uint8,
                device="cuda"))):
            ul = sentinel(rows_total, w.intermediate)
            out = sentinel(rows_total, w.hidden)
            moe.fused_forward(pk["stacked_expert_tokens"], g, u, d, pk["routed_expert_weights"],
                              t["group_sizes"], t["group_offsets"], t["group_padded_offsets"],
                              t["group_idx_for_bx"], ul, out, status=st[2 + i:3 + i],
                              single_launch_workspace=single)
            outs.append((ul, out))
        y = moe.combine_routed(outs[0][1], pk["pair_padded_rows"])
        torch.cuda.synchronize()
        for key, val in t.items():
            res[f"{name}/{key}"] = val.cpu().numpy()
        res[f"{name}/pair_rows"] = pk["pair_padded_rows"].cpu().numpy()
        res[f"{name}/x_packed"] = bits(pk["stacked_expert_tokens"])
        res[f"{name}/ul"] = bits(outs[0][0])
        res[f"{name}/out"] = bits(outs[0][1])
        res[f"{name}/ul_single"] = bits(outs[1][0])
        res[f"{name}/out_single"] = bits(outs[1][1])
        res[f"{name}/y"] = bits(y)
        res[f"{name}/status"] = st.cpu().numpy()
    # the router on two workloads' tokens
    for name in ("tiny", "dsv2_lite"):
        w = workloads.WORKLOADS[name]
        x = torch.from_numpy(workloads.tokens(w, 4)).cuda()
        wg = torch.from_numpy(workloads.router_weights(w, 4)).cuda()
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        ids, wts = moe.router_topk(x, wg, w.top_k, status=st)
        torch.cuda.synchronize()
        res[f"router_{name}/ids"] = ids.cpu().numpy()
        res[f"router_{name}/weights"] = wts.cpu().numpy()
        res[f"router_{name}/status"] = st.cpu().numpy()
    return res


if __name__ == "__main__":
    np.savez(sys.argv[1], **run_cases())
