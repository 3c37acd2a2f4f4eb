"""Router on the GPU against the oracle ("MetaX-TileLang工具链" §2.4).

Both sides accumulate the logits in fp32 but in different orders, so the top-k
decision is compared where it is not a near tie: for every token whose k-th
and (k+1)-th logits differ by more than 1e-3 (float64 reference), the chosen
experts must be the oracle's, in the same descending order wherever adjacent
chosen logits also differ by more than 1e-3; everywhere, the GPU's choice must
be a valid top-k (no unchosen logit above a chosen one by more than 1e-3) and
its weights the softmax probabilities within 5e-5 relative: a probability's
relative error is about its logit's absolute error, and an fp32 logit summed
over up to 7168 products of unit-scale terms is off by a few 1e-6 against the
float64 reference (measured 6e-6 at hidden 4096).
"""
import numpy as np
import pytest
import torch

import oracle
import routed_grouped_gemm_dispatch_gb300 as moe
import workloads
from moe_cases import small_workload

pytestmark = pytest.mark.gpu

GAP = 1e-3


def _check(x, wg, k):
    ids_o, w_o = oracle.router(x, wg, k)
    ids_g, w_g = moe.router_topk(torch.from_numpy(x).cuda(), torch.from_numpy(wg).cuda(), k)
    torch.cuda.synchronize()
    ids_g, w_g = ids_g.cpu().numpy(), w_g.cpu().numpy()
    lg = x.astype(np.float64) @ wg.astype(np.float64).T
    srt = -np.sort(-lg, axis=1)
    E = lg.shape[1]
    cut = srt[:, k - 1] - (srt[:, k] if k < E else -np.inf)
    clear = cut > GAP
    assert clear.mean() > 0.95
    assert np.array_equal(np.sort(ids_g[clear], axis=1), np.sort(ids_o[clear], axis=1))
    chosen = np.take_along_axis(lg, ids_g.astype(np.int64), axis=1)
    gaps = chosen[:, :-1] - chosen[:, 1:]
    ordered = np.all(gaps > GAP, axis=1) & clear
    assert np.array_equal(ids_g[ordered], ids_o[ordered])
    assert np.all(gaps > -GAP)                                  # descending
    kth = chosen[:, -1]
    mask = np.ones_like(lg, bool)
    np.put_along_axis(mask, ids_g.astype(np.int64), False, axis=1)
    assert np.all(np.where(mask, lg, -np.inf).max(axis=1) <= kth + GAP)   # a valid top-k
    p = np.exp(lg - lg.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    ref = np.take_along_axis(p, ids_g.astype(np.int64), axis=1)
    assert np.allclose(w_g, ref, rtol=5e-5, atol=1e-7)


@pytest.mark.parametrize("name,tokens", [("tiny", None), ("dsv2_lite", None), ("decode_skewed", None),
                                         ("mixtral", 1000), ("dsv3", 1000), ("dsv3", None)])
def test_router_workloads(name, tokens):
    w = workloads.WORKLOADS[name]
    T = tokens or w.tokens
    x = workloads.tokens(w, seed=4, n_tokens=T)
    wg = workloads.router_weights(w, seed=4)
    _check(x, wg, w.top_k)


@pytest.mark.parametrize("T,E,k,H", [(1, 40, 5, 128), (333, 40, 1, 256), (257, 200, 16, 384), (130, 16, 16, 128)])
def test_router_odd_shapes(T, E, k, H):
    w = small_workload(tokens=T, top_k=k, experts=E, hidden=H, intermediate=128)
    x = workloads.tokens(w, seed=T)
    wg = workloads.router_weights(w, seed=T)
    _check(x, wg, k)


def test_router_host_validation():
    x = torch.zeros((4, 128), dtype=torch.float16, device="cuda")
    with pytest.raises(moe.MoeError):
        moe.router_topk(x, torch.zeros((300, 128), dtype=torch.float16, device="cuda"), 2)
    with pytest.raises(moe.MoeError):
        moe.router_topk(x, torch.zeros((8, 128), dtype=torch.float16, device="cuda"), 9)


def _exact_case(T, E, H, seed, zero_w=False):
    """Inputs whose fp32 logits are exact integers (entries in {-1, 0, 1}), so
    that every summation order gives the same logits and equal logits are
    exact ties: the chosen experts, ties to the lower index, must be the
    oracle's exactly."""
    rng = np.random.default_rng(seed)
    x = rng.integers(-1, 2, size=(T, H)).astype(np.float16)
    wg = np.zeros((E, H), np.float16) if zero_w else rng.integers(-1, 2, size=(E, H)).astype(np.float16)
    return x, wg


@pytest.mark.parametrize("T,E,k,H,zero_w", [
    (300, 64, 6, 128, False), (200, 256, 8, 256, False), (130, 16, 16, 128, False), (64, 40, 5, 128, False),
    (33, 128, 8, 2048, False),                       # one ragged tile, the hidden split over the cluster
    (9800, 64, 6, 128, False), (9800, 256, 8, 256, False),   # more tiles than half the SMs: 2-SM pairs, a spare CTA
    (9800, 256, 8, 128, True),
    (100, 64, 6, 128, True), (100, 256, 8, 128, True), (100, 16, 4, 128, True), (20, 128, 8, 1024, True)])
def test_router_exact_ties(T, E, k, H, zero_w):
    x, wg = _exact_case(T, E, H, seed=T + E, zero_w=zero_w)
    ids_o, w_o = oracle.router(x, wg, k)
    ids_g, w_g = moe.router_topk(torch.from_numpy(x).cuda(), torch.from_numpy(wg).cuda(), k)
    torch.cuda.synchronize()
    ids_g, w_g = ids_g.cpu().numpy(), w_g.cpu().numpy()
    assert np.array_equal(ids_g, ids_o)
    assert np.allclose(w_g, w_o, rtol=2e-5, atol=1e-8)
    if zero_w:
        assert np.array_equal(ids_g, np.broadcast_to(np.arange(k, dtype=np.int32), (T, k)))


@pytest.mark.parametrize("T,E,k,H", [(10000, 256, 8, 512), (19000, 96, 4, 256), (19000, 200, 16, 128)])
def test_router_pairs(T, E, k, H):
    """Token counts whose tiles outnumber half the SMs: no K split, tiles paired
    on 2-SM MMAs that split W_g's rows (odd tile counts leave a spare CTA)."""
    w = small_workload(tokens=T, top_k=k, experts=E, hidden=H, intermediate=128)
    x = workloads.tokens(w, seed=T)
    wg = workloads.router_weights(w, seed=T)
    _check(x, wg, k)
