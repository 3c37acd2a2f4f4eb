"""Test helpers: raw seeded inputs and their oracle-side preparation.

Raw inputs come from ``workloads`` (routing, tokens, expert weights).  The
oracle-side tables, pair rows and packed arrays come from ``oracle`` only; the
GPU side builds its own from the same raw inputs with the CUDA library.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

import oracle
import workloads

BT = 128
PAD_BITS = 0x7E00         # fp16 NaN: padding rows of the packed x
SENTINEL = 0x7D5A         # fp16 NaN with a payload: pre-fill of up_logits / out


@dataclass
class Raw:
    w: workloads.Workload
    topk_ids: np.ndarray
    topk_weights: np.ndarray
    x_tokens: np.ndarray          # fp16 [T, H]
    gate: np.ndarray              # fp16 [E, I, H]
    up: np.ndarray
    down: np.ndarray              # fp16 [E, H, I]
    extra: dict = field(default_factory=dict)


def raw_inputs(w: workloads.Workload, seed: int = 0) -> Raw:
    ids, tw = workloads.routing(w, seed)
    x = workloads.tokens(w, seed)
    g, u, d = workloads.expert_weights(w, seed, device="cpu")
    return Raw(w, ids, tw, x, g.numpy(), u.numpy(), d.numpy())


def small_workload(name="small", tokens=40, top_k=2, experts=4, hidden=256,
                   intermediate=384, routing="uniform", zipf_s=0.0):
    return workloads.Workload(name, tokens, top_k, experts, hidden, intermediate,
                              routing, zipf_s)


@dataclass
class OracleSide:
    tables: dict
    pair_rows: np.ndarray
    rows_total: int
    x_packed: np.ndarray          # uint16 bits [rows_total, H]
    rw: np.ndarray                # fp32 compact


def oracle_prepare(raw: Raw) -> OracleSide:
    E = raw.w.experts
    t = oracle.build_dispatch(raw.topk_ids, E)
    rows = oracle.pair_padded_rows(raw.topk_ids, E, t["group_padded_offsets"])
    rows_total = t["num_blocks_m"] * BT
    xp, rw = oracle.pack(raw.x_tokens, raw.topk_ids, raw.topk_weights, rows, t,
                         rows_total, PAD_BITS)
    return OracleSide(t, rows, rows_total, xp, rw)


def ulp_diff(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in representable fp16 steps between two arrays of finite halves."""
    def key(b):
        b = b.astype(np.int32)
        return np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(key(a_bits) - key(b_bits))


def within_tol(got_bits, ref_bits, atol=2e-2, rtol=2e-2):
    """Elementwise |got - ref| <= atol + rtol * |ref| on fp16 bit arrays."""
    g = np.asarray(got_bits, np.uint16).view(np.float16).astype(np.float64)
    r = np.asarray(ref_bits, np.uint16).view(np.float16).astype(np.float64)
    ok = np.abs(g - r) <= atol + rtol * np.abs(r)
    return ok & np.isfinite(g)
