"""Pins for the oracle's router ("MetaX-TileLang工具链" §2.4: logits = W_g(x),
scores = softmax(logits), top-k of the scores).

  * one-hot weights W_g[e] = onehot(e) make every logit one of the token's own
    values exactly, so the top-k and the softmax reduce to numpy's argsort and
    a float64 softmax of those values;
  * a float64 brute force on random inputs: the same experts wherever the
    k-th and (k+1)-th logits are not a near tie, the same probabilities;
  * tie-breaking (equal logits: the lower expert index first) and ordering.
"""
import numpy as np

import oracle
import workloads
from moe_cases import small_workload


def _softmax64(v):
    z = np.exp(v - v.max(axis=-1, keepdims=True))
    return z / z.sum(axis=-1, keepdims=True)


def test_one_hot_router_closed_form():
    T, H, E, k = 200, 128, 40, 6
    rng = np.random.default_rng(0)
    x = rng.standard_normal((T, H)).astype(np.float16)
    wg = np.zeros((E, H), np.float16)
    wg[np.arange(E), np.arange(E)] = 1.0            # logit[t, e] = x[t, e] exactly
    ids, wts = oracle.router(x, wg, k)
    lg = x[:, :E].astype(np.float64)
    ref_ids = np.argsort(-lg, axis=1, kind="stable")[:, :k]
    assert np.array_equal(ids, ref_ids)
    p = _softmax64(lg)
    ref_w = np.take_along_axis(p, ref_ids, axis=1)
    assert np.allclose(wts, ref_w, rtol=2e-6, atol=1e-7)


def test_ties_go_to_the_lower_index_and_order_is_descending():
    H, E, k = 128, 8, 4
    x = np.zeros((1, H), np.float16)
    x[0, :E] = [0.5, 2.0, 2.0, -1.0, 0.5, 3.0, 0.5, 0.0]
    wg = np.zeros((E, H), np.float16)
    wg[np.arange(E), np.arange(E)] = 1.0
    ids, wts = oracle.router(x, wg, k)
    assert ids.tolist() == [[5, 1, 2, 0]]
    assert np.all(np.diff(wts[0]) <= 0)
    assert wts[0, 1] == wts[0, 2]


def test_brute_force_float64():
    w = small_workload(tokens=300, top_k=6, experts=64, hidden=256, intermediate=128)
    x = workloads.tokens(w, seed=3)
    wg = workloads.router_weights(w, seed=3)
    ids, wts = oracle.router(x, wg, w.top_k)
    lg = x.astype(np.float64) @ wg.astype(np.float64).T
    order = np.argsort(-lg, axis=1, kind="stable")
    p = _softmax64(lg)
    srt = np.take_along_axis(lg, order, axis=1)
    clear = (srt[:, w.top_k - 1] - srt[:, w.top_k]) > 1e-4     # no near tie at the cut
    assert clear.mean() > 0.95
    assert np.array_equal(ids[clear], order[clear, :w.top_k])
    ref_w = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    assert np.allclose(wts, ref_w, rtol=1e-5, atol=1e-7)
    assert np.all(wts.sum(axis=1) <= 1.0 + 1e-6)
