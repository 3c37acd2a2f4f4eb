"""GPU-side preparation of a case: device tensors, tables from the CUDA
library, and the grouped/padded packing of tokens.

Shares nothing with the oracle side: the tables come from
``moe_build_dispatch`` and the packing from ``moe_pack_routed``, both CUDA
kernels of the library.
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
    pair_rows: torch.Tensor       # int32 [T, k]
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
    """Tables from moe_build_dispatch, packing from moe_pack_routed."""
    E = raw.w.experts
    ids = torch.from_numpy(np.ascontiguousarray(raw.topk_ids)).to(device)
    t = moe.build_dispatch(ids, E)
    x = torch.from_numpy(np.ascontiguousarray(raw.x_tokens)).to(device)
    tw = torch.from_numpy(np.ascontiguousarray(raw.topk_weights)).to(device)
    rows_total = t["group_idx_for_bx"].numel() * BT
    pk = moe.pack_routed(ids, tw, x, t, rows_total)
    g, u, d = weights if weights is not None else to_device_weights(raw, device)
    return GpuSide(ids, t, pk["pair_padded_rows"], rows_total, pk["stacked_expert_tokens"],
                   pk["routed_expert_weights"], g, u, d)


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
