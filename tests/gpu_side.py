"""GPU-side preparation of a case: device tensors, tables from the CUDA
library, and the grouped/padded packing of tokens.

Shares nothing with the oracle side: the tables come from
``moe_build_dispatch``; the packing is plain PyTorch indexing on the device
(a stable sort by expert, each pair's rank within its expert), written from the
contract's description, not from the oracle.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

import routed_grouped_gemm_dispatch_gb300 as moe
from moe_cases import BT, SENTINEL, Raw


@dataclass
class GpuSide:
    ids: torch.Tensor
    tables: dict
    pair_rows: torch.Tensor       # int64 [T, k]
    rows_total: int
    x_packed: torch.Tensor        # fp16 [rows_total, H]
    rw: torch.Tensor              # fp32 [P]
    gate: torch.Tensor
    up: torch.Tensor
    down: torch.Tensor


def to_device_weights(raw: Raw, device="cuda"):
    return (torch.from_numpy(raw.gate).to(device), torch.from_numpy(raw.up).to(device),
            torch.from_numpy(raw.down).to(device))


def gpu_prepare(raw: Raw, weights=None, device="cuda") -> GpuSide:
    T, k = raw.topk_ids.shape
    E, H = raw.w.experts, raw.w.hidden
    ids = torch.from_numpy(np.ascontiguousarray(raw.topk_ids)).to(device)
    t = moe.build_dispatch(ids, E)
    flat = ids.reshape(-1).long()
    P = flat.numel()
    order = torch.sort(flat, stable=True).indices
    e_sorted = flat[order]
    rank = torch.arange(P, device=device) - t["group_offsets"].long()[e_sorted]
    rows = torch.empty(P, dtype=torch.long, device=device)
    rows[order] = t["group_padded_offsets"].long()[e_sorted] + rank
    rows_total = t["group_idx_for_bx"].numel() * BT
    x = torch.from_numpy(raw.x_tokens).to(device)
    xp = torch.full((rows_total, H), float("nan"), dtype=torch.float16, device=device)
    if P:
        xp[rows] = x[torch.arange(P, device=device) // k]
    tw = torch.from_numpy(raw.topk_weights).to(device).reshape(-1)
    rw = tw[order].contiguous()                 # compact index of sorted position i is i
    g, u, d = weights if weights is not None else to_device_weights(raw, device)
    return GpuSide(ids, t, rows.reshape(T, k), rows_total, xp, rw, g, u, d)


def sentinel(rows: int, cols: int, device="cuda") -> torch.Tensor:
    return torch.full((rows, cols), SENTINEL, dtype=torch.int16, device=device).view(torch.float16)


def run_forward(side: GpuSide, intermediate: int, status=None):
    ul = sentinel(side.rows_total, intermediate)
    out = sentinel(side.rows_total, side.x_packed.shape[1])
    t = side.tables
    moe.fused_forward(side.x_packed, side.gate, side.up, side.down, side.rw,
                      t["group_sizes"], t["group_offsets"], t["group_padded_offsets"],
                      t["group_idx_for_bx"], ul, out, status=status)
    return ul, out


def bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)
