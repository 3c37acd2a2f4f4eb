"""Seeded synthetic inputs for the routed fused-MoE expert GEMM.

This module serves both the CUDA path and the CPU oracle, so it holds none of
the method's arithmetic: no dispatch tables, no packing, no GEMM.  It draws
routing choices, routed weights, token activations and expert weights with the
shapes and distributions of the workloads below, and nothing else.

Workloads (model-shaped; no dataset or trained weights are involved):
  tiny            64 tokens, top-2 of 4 experts, hidden 256, intermediate 512,
                  uniform distinct picks, all weights ~N(0, 1/hidden)
  dsv2_lite       DeepSeek-V2-Lite-shaped: 4096 tokens, top-6 of 64, 2048 / 1408, uniform
  mixtral         Mixtral-shaped: 8192 tokens, top-2 of 8, 4096 / 14336, uniform
  decode_skewed   32 tokens, top-8 of 128, 2048 / 768, Zipf(s=1.2) popularity
  dsv3            DeepSeek-V3-shaped: 16384 tokens, top-8 of 256, 7168 / 2048, Zipf(s=1.0)
  dsv3_slice      a small case of the DeepSeek-V3-shaped kernels for profiler captures
                  (a few GB on the device): 2048 tokens, top-8 of 32, 7168 / 2048, Zipf(s=1.0)

Distributions: x ~ N(0, 1) fp16; gate/up ~ N(0, 1/hidden), down ~ N(0, 1/intermediate)
fp16 (tiny: all three ~ N(0, 1/hidden)); routed weights = softmax over the k
chosen experts of N(0, 1) logits, fp32.  Zipf popularity p_e ∝ (e+1)^-s with
no shuffle of ranks; each token takes k distinct experts without replacement
∝ p (Gumbel-top-k).  Uniform: k distinct experts, uniformly.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

__all__ = ["Workload", "WORKLOADS", "routing", "tokens", "expert_weights", "router_weights"]


@dataclass(frozen=True)
class Workload:
    name: str
    tokens: int
    top_k: int
    experts: int
    hidden: int
    intermediate: int
    routing: str = "uniform"      # "uniform" | "zipf"
    zipf_s: float = 0.0
    weight_std: str = "fan_in"    # "fan_in" | "hidden"

    @property
    def pairs(self) -> int:
        return self.tokens * self.top_k

    def flops(self) -> float:
        """2 * pairs * 3 * hidden * intermediate (valid rows only)."""
        return 6.0 * self.pairs * self.hidden * self.intermediate


WORKLOADS = {
    "tiny": Workload("tiny", 64, 2, 4, 256, 512, "uniform", 0.0, "hidden"),
    "dsv2_lite": Workload("dsv2_lite", 4096, 6, 64, 2048, 1408, "uniform"),
    "mixtral": Workload("mixtral", 8192, 2, 8, 4096, 14336, "uniform"),
    "decode_skewed": Workload("decode_skewed", 32, 8, 128, 2048, 768, "zipf", 1.2),
    "dsv3": Workload("dsv3", 16384, 8, 256, 7168, 2048, "zipf", 1.0),
    "dsv3_slice": Workload("dsv3_slice", 2048, 8, 32, 7168, 2048, "zipf", 1.0),
}


def routing(w: Workload, seed: int = 0):
    """topk_ids int32 [T, k] (distinct per token) and topk_weights fp32 [T, k]."""
    rng = np.random.default_rng(seed)
    T, k, E = w.tokens, w.top_k, w.experts
    if w.routing == "uniform":
        keys = rng.random((T, E))
    elif w.routing == "zipf":
        logp = -w.zipf_s * np.log(np.arange(1, E + 1, dtype=np.float64))
        keys = logp[None, :] + rng.gumbel(size=(T, E))
    else:
        raise ValueError(w.routing)
    # the k largest keys per token, distinct by construction
    ids = np.argsort(-keys, axis=1, kind="stable")[:, :k].astype(np.int32)
    logits = rng.standard_normal((T, k))
    z = np.exp(logits - logits.max(axis=1, keepdims=True))
    weights = (z / z.sum(axis=1, keepdims=True)).astype(np.float32)
    return np.ascontiguousarray(ids), np.ascontiguousarray(weights)


def _std(w: Workload):
    if w.weight_std == "hidden":
        s = 1.0 / np.sqrt(w.hidden)
        return s, s, s
    return 1.0 / np.sqrt(w.hidden), 1.0 / np.sqrt(w.hidden), 1.0 / np.sqrt(w.intermediate)


def tokens(w: Workload, seed: int = 0, n_tokens: int | None = None) -> np.ndarray:
    """x ~ N(0, 1), fp16 [T, H] (numpy, host)."""
    rng = np.random.default_rng(seed + 1_000_003)
    T = w.tokens if n_tokens is None else n_tokens
    return rng.standard_normal((T, w.hidden), dtype=np.float32).astype(np.float16)


def expert_weights(w: Workload, seed: int = 0, device: str = "cpu", experts=None):
    """gate_w, up_w [E, I, H] and down_w [E, H, I], fp16, as torch tensors.

    Drawn with a seeded torch.Generator on ``device`` (the 22.5 GB DSV3-shaped
    set is drawn on the GPU).  Values depend on the device's generator, so a
    test draws once and hands the same tensors to both sides.  ``experts``
    limits the draw to the first n experts (for small parity cases).
    """
    import torch

    E = w.experts if experts is None else experts
    g = torch.Generator(device=device)
    g.manual_seed(seed + 7)
    sg, su, sd = _std(w)

    def draw(shape, std):
        t = torch.empty(shape, dtype=torch.float16, device=device)
        # chunk over experts to bound the fp32 temporary
        for e in range(shape[0]):
            t[e].copy_(torch.randn(shape[1:], generator=g, device=device,
                                   dtype=torch.float32).mul_(std))
        return t

    gate = draw((E, w.intermediate, w.hidden), sg)
    up = draw((E, w.intermediate, w.hidden), su)
    down = draw((E, w.hidden, w.intermediate), sd)
    return gate, up, down


def router_weights(w: Workload, seed: int = 0) -> np.ndarray:
    """Router weight W_g [E, H] ~ N(0, 1/H), fp16 (numpy, host)."""
    rng = np.random.default_rng(seed + 2_000_003)
    return (rng.standard_normal((w.experts, w.hidden), dtype=np.float32)
            / np.float32(np.sqrt(w.hidden))).astype(np.float16)
