"""Pins for the oracle's fused forward.

The semantics come from "Fused MoE GEMM 提交说明" (§算子来源: gate = x·gate_wᵀ,
up = x·up_wᵀ, hidden = silu(gate)·up, out = hidden·down_wᵀ · routed weight;
§实现要点: padded rows for x / up_logits / out, compact rows for the routed
weights, padding rows neither computed nor written) and "MetaX-TileLang工具链"
§2.4 (the same expert MLP).

Pins, none of which re-types the oracle's loops:
  * closed forms — zero gate, zero routed weight, and one-hot weight matrices
    for which every dot product has a single term, so the result reduces to
    elementwise silu / products that numpy evaluates directly;
  * a brute force over (token, expert) pairs in token order with no tables and
    no padding, in float64 with numpy's own fp16 casts; it must agree bit for
    bit with the oracle's fp64 mode and within 1 fp16 step with its fp32 mode;
  * thread-count determinism, padding rows untouched, the row-subset entry.
"""
import numpy as np
import pytest

import oracle
from moe_cases import (BT, PAD_BITS, SENTINEL, oracle_prepare, raw_inputs,
                       small_workload, ulp_diff)


def _silu(v):
    return v / (1.0 + np.exp(-v))


def _run(raw, side, **kw):
    rows = side.rows_total
    up0 = np.full((rows, raw.w.intermediate), SENTINEL, np.uint16)
    out0 = np.full((rows, raw.w.hidden), SENTINEL, np.uint16)
    return oracle.fused_forward(side.x_packed, raw.gate, raw.up, raw.down, side.rw,
                                side.tables, up0, out0, **kw)


def _valid_mask(side):
    mask = np.zeros(side.rows_total, bool)
    mask[side.pair_rows.reshape(-1)] = True
    return mask


@pytest.fixture(scope="module")
def small():
    raw = raw_inputs(small_workload(tokens=300, top_k=2, experts=3), seed=3)
    return raw, oracle_prepare(raw)


def _brute_force(raw):
    """out for every (token, j) pair, in token order, float64, numpy fp16 casts."""
    T, k = raw.topk_ids.shape
    x = raw.x_tokens.astype(np.float64)
    G = raw.gate.astype(np.float64)
    U = raw.up.astype(np.float64)
    D = raw.down.astype(np.float64)
    up = np.zeros((T, k, raw.w.intermediate), np.float16)
    out = np.zeros((T, k, raw.w.hidden), np.float16)
    for t in range(T):
        for j in range(k):
            e = raw.topk_ids[t, j]
            g = G[e] @ x[t]
            u = U[e] @ x[t]
            up[t, j] = (_silu(g) * u).astype(np.float16)
            a = D[e] @ up[t, j].astype(np.float64)
            out[t, j] = (a * np.float64(raw.topk_weights[t, j])).astype(np.float16)
    return up.view(np.uint16), out.view(np.uint16)


def test_brute_force_fp64_mode_bit_exact(small):
    raw, side = small
    up_ref, out_ref = _brute_force(raw)
    up, out = _run(raw, side, acc_f64=True)
    r = side.pair_rows
    assert np.array_equal(up[r], up_ref)
    assert np.array_equal(out[r], out_ref)


def test_brute_force_fp32_mode_close(small):
    """fp32 accumulation differs from fp64 only by fp32 rounding.  up_logits:
    one fp16 step away from zero, an absolute 1e-5 near zero where the sum
    cancels (fp32 error of ~256 unit-size terms).  out: the same plus what a
    one-step change of some up_logits entries moves through the down
    projection (384 terms of |down| ~ 0.05, a few flipped)."""
    raw, side = small
    up_ref, out_ref = _brute_force(raw)
    up, out = _run(raw, side)
    r = side.pair_rows
    for got, ref, atol, rtol in ((up[r], up_ref, 1e-5, 2.0 ** -10),
                                 (out[r], out_ref, 1e-3, 2.0 ** -9)):
        g = got.view(np.float16).astype(np.float64)
        f = ref.view(np.float16).astype(np.float64)
        assert np.all(np.abs(g - f) <= atol + rtol * np.abs(f))
        assert (got == ref).mean() > 0.98


def test_padding_rows_untouched(small):
    raw, side = small
    up, out = _run(raw, side)
    pad = ~_valid_mask(side)
    assert pad.sum() > 0
    assert np.all(up[pad] == SENTINEL) and np.all(out[pad] == SENTINEL)
    valid = ~pad
    assert not np.any(up[valid] == SENTINEL) and not np.any(out[valid] == SENTINEL)


def test_padding_rows_of_x_do_not_leak(small):
    raw, side = small
    # padding rows of x are NaN (PAD_BITS); no valid output may be NaN
    assert np.all(side.x_packed[~_valid_mask(side)] == PAD_BITS)
    up, out = _run(raw, side)
    v = _valid_mask(side)
    assert np.all(np.isfinite(up[v].view(np.float16)))
    assert np.all(np.isfinite(out[v].view(np.float16)))


def test_zero_gate_gives_zero(small):
    raw, side = small
    raw0 = type(raw)(**{**raw.__dict__, "gate": np.zeros_like(raw.gate)})
    up, out = _run(raw0, side)
    v = _valid_mask(side)
    assert np.all((up[v] & 0x7FFF) == 0)
    assert np.all((out[v] & 0x7FFF) == 0)


def test_zero_routed_weight_gives_zero(small):
    raw, side = small
    side0 = type(side)(**{**side.__dict__, "rw": np.zeros_like(side.rw)})
    up_ref, _ = _run(raw, side)
    up, out = _run(raw, side0)
    v = _valid_mask(side)
    assert np.array_equal(up[v], up_ref[v])
    assert np.all((out[v] & 0x7FFF) == 0)


def test_one_hot_weights_closed_form():
    """gate_w[e][j] = a_e·onehot(σ_e(j)), up_w[e][j] = b_e·onehot(τ_e(j)),
    down_w[e][c] = d_e·onehot(ρ_e(c)): every dot product has one term, so
    up[p, j] = fp16(silu(a·x[σ(j)]) · b·x[τ(j)]) and out[p, c] =
    fp16(d·up[p, ρ(c)] · w).  H != I, so a transposed operand cannot even
    index; distinct σ, τ, scales per expert catch a swapped gate/up or a
    wrong expert."""
    w = small_workload(tokens=150, top_k=2, experts=3, hidden=256, intermediate=384)
    raw = raw_inputs(w, seed=11)
    rng = np.random.default_rng(5)
    E, I, H = w.experts, w.intermediate, w.hidden
    G = np.zeros((E, I, H), np.float16)
    U = np.zeros((E, I, H), np.float16)
    D = np.zeros((E, H, I), np.float16)
    params = []
    for e in range(E):
        a, b, d = (float(v) for v in rng.choice([0.5, 1.0, 2.0, -1.0], 3))
        sig = rng.integers(0, H, I)
        tau = rng.integers(0, H, I)
        rho = rng.integers(0, I, H)
        G[e, np.arange(I), sig] = a
        U[e, np.arange(I), tau] = b
        D[e, np.arange(H), rho] = d
        params.append((a, b, d, sig, tau, rho))
    raw = type(raw)(**{**raw.__dict__, "gate": G, "up": U, "down": D})
    side = oracle_prepare(raw)
    up32, out32 = _run(raw, side)
    up64, out64 = _run(raw, side, acc_f64=True)
    T, k = raw.topk_ids.shape
    for t in range(T):
        xt = raw.x_tokens[t].astype(np.float64)
        for j in range(k):
            e = raw.topk_ids[t, j]
            a, b, d, sig, tau, rho = params[e]
            p = side.pair_rows[t, j]
            up_ref = (_silu(a * xt[sig]) * (b * xt[tau])).astype(np.float16)
            out_ref = ((d * up_ref.astype(np.float64)[rho])
                       * np.float64(raw.topk_weights[t, j])).astype(np.float16)
            ub, ob = up_ref.view(np.uint16), out_ref.view(np.uint16)
            assert np.array_equal(up64[p], ub)
            assert np.array_equal(out64[p], ob)
            # one-term dot products are exact in fp32 too; only silu's fp32
            # evaluation and the fp32 products can move a result by one step
            assert ulp_diff(up32[p], ub).max() <= 1
            assert ulp_diff(out32[p], ob).max() <= 1


def test_silu_textbook_values():
    """One expert, gate = up = identity (H = I): up = fp16(silu(x)·x); with
    down = identity and w = 1, out = up.  silu(1) = e/(1+e), silu(-1) =
    -1/(1+e), silu(0) = 0, silu(x) -> x for large x."""
    H = I = 128
    w = small_workload(tokens=1, top_k=1, experts=1, hidden=H, intermediate=I)
    raw = raw_inputs(w, seed=0)
    x = np.zeros((1, H), np.float16)
    x[0, :4] = [1.0, -1.0, 0.0, 12.0]
    eye = np.eye(H, dtype=np.float16)[None]
    raw = type(raw)(**{**raw.__dict__, "x_tokens": x, "gate": eye, "up": eye,
                       "down": eye.copy(), "topk_weights": np.ones((1, 1), np.float32)})
    side = oracle_prepare(raw)
    up, out = _run(raw, side, acc_f64=True)
    e = np.e
    expect = np.array([e / (1 + e) * 1.0, -1 / (1 + e) * -1.0, 0.0,
                       12.0 / (1 + np.exp(-12.0)) * 12.0]).astype(np.float16).view(np.uint16)
    assert np.array_equal(up[0, :4], expect)
    assert np.array_equal(out[0, :4], expect)


def test_thread_count_determinism(small):
    raw, side = small
    a = _run(raw, side, n_threads=1)
    b = _run(raw, side, n_threads=4)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_forward_rows_matches_full(small):
    raw, side = small
    up, out = _run(raw, side)
    pick = np.array([0, 1, BT - 1, BT, side.pair_rows[7, 1], side.rows_total - 1], np.int64)
    upr, outr, valid = oracle.forward_rows(side.x_packed, raw.gate, raw.up, raw.down,
                                           side.rw, side.tables, pick)
    vm = _valid_mask(side)
    assert np.array_equal(valid, vm[pick])
    for n, p in enumerate(pick):
        if valid[n]:
            assert np.array_equal(upr[n], up[p]) and np.array_equal(outr[n], out[p])


def test_pack_and_combine_closed_forms(small):
    raw, side = small
    T, k = raw.topk_ids.shape
    xb = raw.x_tokens.view(np.uint16)
    for t in range(T):
        for j in range(k):
            p = side.pair_rows[t, j]
            assert np.array_equal(side.x_packed[p], xb[t])
            e = raw.topk_ids[t, j]
            compact = side.tables["group_offsets"][e] + (p - side.tables["group_padded_offsets"][e])
            assert side.rw[compact] == raw.topk_weights[t, j]
    # combine: out rows holding 0.25 * (j + 1) sum to 0.25 * k(k+1)/2 per token
    out = np.zeros((side.rows_total, raw.w.hidden), np.float16)
    for t in range(T):
        for j in range(k):
            out[side.pair_rows[t, j]] = 0.25 * (j + 1)
    y = oracle.combine(out.view(np.uint16), side.pair_rows, T, k).view(np.float16)
    assert np.all(y == np.float16(0.25 * k * (k + 1) / 2))


def _combine_case(T, k, H, rng, values):
    """Pair rows scattered over a padded array: token t's j-th row holds
    values[t, j] (fp16 [T, k, H]); every other row is NaN."""
    rows_total = 4 * T * k + 7
    pr = rng.permutation(rows_total)[:T * k].astype(np.int32).reshape(T, k)
    out = np.full((rows_total, H), np.nan, np.float16)
    for t in range(T):
        for j in range(k):
            out[pr[t, j]] = values[t, j]
    return out, pr


def test_combine_pinned_by_exact_sums():
    """oracle.combine against the exact sum rounded once to fp16 (numpy's
    float64 sum, then numpy's RNE cast): "MetaX-TileLang工具链" §2.7 sums a
    token's expert rows with scatter_reduce; the reading is an fp32 sum in j
    order with one rounding.  The row values are distinct per (token, j) and
    are multiples of 2^-6 below 2^5 in magnitude, so every partial sum of up
    to 8 of them is exact in fp32 and the exact sum is the reference: a
    combine that reads another token's rows or another j, drops a row, or
    rounds a partial sum to fp16 fails."""
    rng = np.random.default_rng(11)
    T, k, H = 37, 6, 64
    vals = (rng.integers(-2047, 2048, size=(T, k, H)) / 64.0).astype(np.float16)
    assert np.all(vals.astype(np.float64) * 64 == np.round(vals.astype(np.float64) * 64))
    out, pr = _combine_case(T, k, H, rng, vals)
    y = oracle.combine(out.view(np.uint16), pr, T, k).view(np.float16)
    expect = vals.astype(np.float64).sum(axis=1).astype(np.float16)
    assert np.array_equal(y.view(np.uint16), expect.view(np.uint16))
    # the values really tell tokens and rows apart (the pin would catch a mix-up)
    swapped = vals[::-1].astype(np.float64).sum(axis=1).astype(np.float16)
    assert not np.array_equal(swapped, expect)
    fewer = vals[:, :-1].astype(np.float64).sum(axis=1).astype(np.float16)
    assert np.count_nonzero(fewer != expect) > 0.9 * expect.size


def test_combine_special_sums():
    """Cancellation to +0, a sum an fp16 accumulator would get wrong
    (2048 + 1 + 1: fp16 steps are 2 above 2048, so rounding each partial sum
    gives 2048, the fp32 sum gives 2050), and overflow: a sum at or above
    65520 rounds to +inf under round-to-nearest-even, 65519 to 65504."""
    rng = np.random.default_rng(12)
    cases = [
        ([1000.5, -1000.5, 3.25, -3.25], 0.0),
        ([2048.0, 1.0, 1.0, 0.0], 2050.0),
        ([30000.0, 30000.0, 5520.0, 0.0], np.inf),
        ([-30000.0, -30000.0, -5520.0, 0.0], -np.inf),
        ([30000.0, 30000.0, 5504.0, 15.0], 65504.0),
    ]
    T, k, H = len(cases), 4, 8
    vals = np.zeros((T, k, H), np.float16)
    for t, (v, _) in enumerate(cases):
        vals[t] = np.array(v, np.float16)[:, None]
    out, pr = _combine_case(T, k, H, rng, vals)
    y = oracle.combine(out.view(np.uint16), pr, T, k).view(np.float16)
    for t, (_, want) in enumerate(cases):
        assert np.all(y[t] == np.float16(want)), (t, y[t], want)
    assert np.all(np.signbit(y[0]) == False)  # noqa: E712  (x + -x is +0 in round-to-nearest)
