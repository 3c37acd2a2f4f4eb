"""Fused forward on the GPU against the CPU oracle.

Bar ("Fused MoE GEMM 提交说明", §实现要点 and §完整算子代码): every valid row of
out and up_logits within |gpu − oracle| <= 2e-2 + 2e-2·|oracle| elementwise;
every padding row of out and up_logits left bit-for-bit as the caller filled it.
Small cases compare every element; the full-size workloads compare at least
one valid row of every active block (so both CTAs of every 2-SM tile and every
N slice are checked; the oracle computes the rows one by one), every valid row
of the decode shape, plus the whole padding/valid structure.  Every comparison
records its error statistics (tests/parity_report.py).
"""
import numpy as np
import pytest
import torch

import oracle
import routed_grouped_gemm_dispatch_gb300 as moe
import workloads
from gpu_side import bits, gpu_prepare, run_forward
from moe_cases import BT, SENTINEL, Raw, oracle_prepare, raw_inputs, small_workload
from parity_report import compare

pytestmark = pytest.mark.gpu

ATOL = 2e-2
RTOL = 2e-2


def _valid_mask(pair_rows, rows_total):
    m = np.zeros(rows_total, bool)
    m[np.asarray(pair_rows).reshape(-1)] = True
    return m


def _case(raw, tag=""):
    w = raw.w
    return (f"{w.name}{tag} T{w.tokens} k{w.top_k} E{w.experts} H{w.hidden} I{w.intermediate}")


def _full_parity(raw, tag=""):
    side_o = oracle_prepare(raw)
    up_o = np.full((side_o.rows_total, raw.w.intermediate), SENTINEL, np.uint16)
    out_o = np.full((side_o.rows_total, raw.w.hidden), SENTINEL, np.uint16)
    oracle.fused_forward(side_o.x_packed, raw.gate, raw.up, raw.down, side_o.rw, side_o.tables,
                         up_o, out_o)
    side_g = gpu_prepare(raw)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ul, out = run_forward(side_g, raw.w.intermediate, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # the GPU harness placed every pair where the oracle did
    assert np.array_equal(side_g.pair_rows.cpu().numpy(), side_o.pair_rows)
    assert np.array_equal(bits(side_g.x_packed), side_o.x_packed)
    up_g, out_g = bits(ul), bits(out)
    v = _valid_mask(side_o.pair_rows, side_o.rows_total)
    # padding rows untouched, bit for bit
    assert np.array_equal(up_g[~v], up_o[~v])
    assert np.array_equal(out_g[~v], out_o[~v])
    ok_u = compare(_case(raw, tag), "up_logits", up_g[v], up_o[v], ATOL, RTOL)
    ok_o = compare(_case(raw, tag), "out", out_g[v], out_o[v], ATOL, RTOL)
    assert ok_u.all(), f"up_logits: {np.count_nonzero(~ok_u)} of {ok_u.size} outside tolerance"
    assert ok_o.all(), f"out: {np.count_nonzero(~ok_o)} of {ok_o.size} outside tolerance"
    return up_g, out_g, up_o, out_o


def test_tiny_workload_full_parity():
    raw = raw_inputs(workloads.WORKLOADS["tiny"], seed=0)
    _full_parity(raw)


@pytest.mark.parametrize("shape", [
    # tokens, top_k, experts, hidden, intermediate, routing
    (300, 2, 3, 256, 384, "uniform"),     # 2 blocks per expert, ragged tails
    (500, 4, 40, 384, 256, "uniform"),    # > 16 active blocks (several panels); H = 256 + 128
    (40, 2, 4, 128, 128, "uniform"),      # smallest shape: one slice each, half-empty N tile
    (32, 8, 128, 256, 256, "zipf"),       # decode-like: many empty experts
    (700, 1, 2, 512, 640, "zipf"),        # one expert holds most rows (> 4 blocks)
])
def test_small_shapes_full_parity(shape):
    T, k, E, H, I, routing = shape
    w = small_workload(tokens=T, top_k=k, experts=E, hidden=H, intermediate=I,
                       routing=routing, zipf_s=1.2 if routing == "zipf" else 0.0)
    _full_parity(raw_inputs(w, seed=1))


@pytest.mark.parametrize("seed", range(10))
def test_random_shapes_full_parity(seed):
    """Seeded random shapes: 1-64 experts, top-1..8, 1-600 tokens, H and I in
    128..640, uniform or Zipf routing; every element against the oracle."""
    rng = np.random.default_rng(1000 + seed)
    E = int(rng.choice([1, 2, 3, 5, 8, 16, 40, 64]))
    k = int(rng.integers(1, min(8, E) + 1))
    T = int(rng.choice([1, 7, 64, 129, 255, 600]))
    H = int(rng.choice([128, 256, 384, 640]))
    I = int(rng.choice([128, 256, 512, 640]))
    routing = "zipf" if rng.random() < 0.5 else "uniform"
    w = small_workload(tokens=T, top_k=k, experts=E, hidden=H, intermediate=I, routing=routing,
                       zipf_s=1.1 if routing == "zipf" else 0.0)
    _full_parity(raw_inputs(w, seed=seed), tag=f" seed{seed}")


def test_exact_multiple_of_block():
    """An expert with exactly 128 rows: the +1 rule gives it a second block,
    which is empty and must be skipped."""
    w = small_workload(tokens=128, top_k=1, experts=2, hidden=256, intermediate=256)
    raw = raw_inputs(w, seed=2)
    raw.topk_ids[:] = 0
    _full_parity(raw)


def test_no_tokens_writes_nothing():
    w = small_workload(tokens=0, top_k=2, experts=3, hidden=256, intermediate=256)
    raw = raw_inputs(w, seed=0)
    side = gpu_prepare(raw)
    ul, out = run_forward(side, w.intermediate)
    torch.cuda.synchronize()
    assert np.all(bits(ul) == SENTINEL) and np.all(bits(out) == SENTINEL)


def test_bad_table_entry_is_flagged_not_fatal():
    w = small_workload(tokens=64, top_k=2, experts=4, hidden=256, intermediate=256)
    raw = raw_inputs(w, seed=0)
    side = gpu_prepare(raw)
    side.tables["group_idx_for_bx"][1] = 99          # out of range expert
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ul, out = run_forward(side, w.intermediate, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & moe.MOE_DEV_BAD_TABLE
    # block 1's rows were skipped, not written
    assert np.all(bits(out)[BT:2 * BT] == SENTINEL)


def test_host_validation_rejects_bad_shapes():
    w = small_workload(tokens=16, top_k=1, experts=2, hidden=256, intermediate=256)
    raw = raw_inputs(w, seed=0)
    side = gpu_prepare(raw)
    t = side.tables
    ul = torch.empty((side.rows_total, 256), dtype=torch.float16, device="cuda")
    short = torch.empty((side.rows_total - BT, 256), dtype=torch.float16, device="cuda")
    with pytest.raises(ValueError):
        moe.fused_forward(side.x_packed, side.gate, side.up, side.down, side.rw,
                          t["group_sizes"], t["group_offsets"], t["group_padded_offsets"],
                          t["group_idx_for_bx"], ul, short)
    with pytest.raises(moe.MoeError):
        moe.fused_forward(side.x_packed[:-BT], side.gate, side.up, side.down, side.rw,
                          t["group_sizes"], t["group_offsets"], t["group_padded_offsets"],
                          t["group_idx_for_bx"], ul[:-BT], short)


def test_repeated_calls_identical():
    raw = raw_inputs(small_workload(tokens=300, top_k=2, experts=3), seed=4)
    side = gpu_prepare(raw)
    a = [bits(t) for t in run_forward(side, raw.w.intermediate)]
    b = [bits(t) for t in run_forward(side, raw.w.intermediate)]
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_phases_run_separately_match_the_fused_call():
    """moe_fused_forward_ex: phase 1 alone, then phase 2 alone (with and without
    programmatic dependent launch), reproduces the two-phase call bit for bit."""
    raw = raw_inputs(small_workload(tokens=500, top_k=4, experts=40, hidden=384, intermediate=256), seed=6)
    side = gpu_prepare(raw)
    ref = [bits(t) for t in run_forward(side, raw.w.intermediate)]
    from gpu_side import sentinel
    t = side.tables
    for p2_flags in (moe.MOE_RUN_PHASE2, moe.MOE_RUN_PHASE2 | moe.MOE_NO_PDL):
        ul = sentinel(side.rows_total, raw.w.intermediate)
        out = sentinel(side.rows_total, raw.w.hidden)
        for flags in (moe.MOE_RUN_PHASE1, p2_flags):
            moe.fused_forward(side.x_packed, side.gate, side.up, side.down, side.rw, t["group_sizes"],
                              t["group_offsets"], t["group_padded_offsets"], t["group_idx_for_bx"], ul, out,
                              flags=flags)
        torch.cuda.synchronize()
        assert np.array_equal(bits(ul), ref[0]) and np.array_equal(bits(out), ref[1])


def test_side_stream_and_concurrent_calls():
    """The whole chain on a caller's stream, and two independent forwards on two
    streams at once, give the default-stream result bit for bit."""
    raw1 = raw_inputs(small_workload(tokens=300, top_k=2, experts=3), seed=4)
    raw2 = raw_inputs(small_workload(tokens=200, top_k=4, experts=16, hidden=384, intermediate=256), seed=5)
    side1, side2 = gpu_prepare(raw1), gpu_prepare(raw2)
    ref1 = [bits(t) for t in run_forward(side1, raw1.w.intermediate)]
    ref2 = [bits(t) for t in run_forward(side2, raw2.w.intermediate)]
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s1):
        got1 = run_forward(side1, raw1.w.intermediate)
    with torch.cuda.stream(s2):
        got2 = run_forward(side2, raw2.w.intermediate)
    torch.cuda.synchronize()
    assert all(np.array_equal(bits(g), r) for g, r in zip(got1, ref1))
    assert all(np.array_equal(bits(g), r) for g, r in zip(got2, ref2))


# --------------------------------------------------------------------------
# full-size workloads: a row of every active block
# --------------------------------------------------------------------------

def _rows_every_block(tables, rng, per_block=1):
    """Padded rows to check: `per_block` random valid rows of every active
    block (each row runs through every N slice of its tile, so every (tile,
    slice) and both CTAs of every pair are covered), plus the first and last
    valid rows of every block of the three largest experts."""
    sizes = np.asarray(tables["group_sizes"])
    padded = np.asarray(tables["group_padded_offsets"])
    picks = []
    big = set(np.argsort(-sizes)[:3].tolist())
    for e in np.nonzero(sizes)[0]:
        c = int(sizes[e])
        for lo in range(0, c, BT):
            hi = min(c, lo + BT)
            picks += list(rng.choice(np.arange(lo, hi), size=min(per_block, hi - lo), replace=False) + padded[e])
            if e in big:
                picks += [padded[e] + lo, padded[e] + hi - 1]
    return np.array(sorted(set(int(p) for p in picks)), np.int64)


def _check_rows(case, up_g, out_g, up_r, out_r):
    ok_u = compare(case, "up_logits", up_g, up_r, ATOL, RTOL)
    ok_o = compare(case, "out", out_g, out_r, ATOL, RTOL)
    assert ok_u.all(), f"{np.count_nonzero(~ok_u)} up_logits entries outside tolerance"
    assert ok_o.all(), f"{np.count_nonzero(~ok_o)} out entries outside tolerance"


def _full_size_rows(raw, rows_of, tag=""):
    w = raw.w
    side_o = oracle_prepare(raw)
    side_g = gpu_prepare(raw)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ul, out = run_forward(side_g, w.intermediate, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    up_g, out_g = bits(ul), bits(out)
    v = _valid_mask(side_o.pair_rows, side_o.rows_total)
    assert np.all(up_g[~v] == SENTINEL) and np.all(out_g[~v] == SENTINEL)
    assert np.all(np.isfinite(out_g[v].view(np.float16)))
    assert np.all(np.isfinite(up_g[v].view(np.float16)))
    rows = rows_of(side_o)
    up_r, out_r, valid = oracle.forward_rows(side_o.x_packed, raw.gate, raw.up, raw.down,
                                             side_o.rw, side_o.tables, rows)
    assert valid.all()
    _check_rows(_case(raw, tag) + f" ({rows.size} rows)", up_g[rows], out_g[rows], up_r, out_r)
    return rows


@pytest.mark.parametrize("name", ["dsv2_lite", "mixtral"])
def test_full_size_every_active_block(name):
    w = workloads.WORKLOADS[name]
    raw = raw_inputs(w, seed=0)
    rows = _full_size_rows(raw, lambda so: _rows_every_block(so.tables, np.random.default_rng(0)))
    sizes = oracle.build_dispatch(raw.topk_ids, w.experts)["group_sizes"]
    assert rows.size >= int(np.sum(-(-sizes // BT)))


def test_full_size_decode_every_valid_row():
    w = workloads.WORKLOADS["decode_skewed"]
    raw = raw_inputs(w, seed=0)
    rows = _full_size_rows(raw, lambda so: np.sort(so.pair_rows.reshape(-1)).astype(np.int64))
    assert rows.size == w.pairs


def test_full_size_top1_unit_routed_weight():
    """DeepSeek-V2-Lite-shaped experts with top-1 routing: the routed weight is
    softmax over one logit, exactly 1.0, so out keeps the full scale of
    h·down_wᵀ (typical |out| about 0.4 rather than 0.04) and the tolerance is
    tested where it is tight relative to the values.  Every expert has one
    block of about 64 rows (every tile a lone block)."""
    w = workloads.Workload("dsv2_lite_top1", 4096, 1, 64, 2048, 1408, "uniform")
    raw = raw_inputs(w, seed=3)
    assert np.all(raw.topk_weights == 1.0)
    _full_size_rows(raw, lambda so: _rows_every_block(so.tables, np.random.default_rng(3), per_block=4))


def test_dsv3_full_size_every_active_block():
    """DeepSeek-V3-shaped (22.5 GB of expert weights, drawn on the GPU): the
    oracle recomputes a valid row of every active block.  Its host weight
    arrays are filled a few experts at a time (the rest stay unallocated zero
    pages), so host memory stays near one batch of experts."""
    w = workloads.WORKLOADS["dsv3"]
    ids, tw = workloads.routing(w, seed=0)
    x = workloads.tokens(w, seed=0)
    gate, up, down = workloads.expert_weights(w, seed=0, device="cuda")
    raw = Raw(w, ids, tw, x, None, None, None)
    side_g = gpu_prepare(raw, weights=(gate, up, down))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ul, out = run_forward(side_g, w.intermediate, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0

    tab = oracle.build_dispatch(ids, w.experts)
    for key in ("group_sizes", "group_offsets", "group_padded_offsets", "group_idx_for_bx"):
        assert np.array_equal(side_g.tables[key].cpu().numpy(), tab[key])
    prow = oracle.pair_padded_rows(ids, w.experts, tab["group_padded_offsets"])
    assert np.array_equal(side_g.pair_rows.cpu().numpy(), prow)
    rows_total = tab["num_blocks_m"] * BT
    xo, rwo = oracle.pack(x, ids, tw, prow, tab, rows_total)
    rows = _rows_every_block(tab, np.random.default_rng(1))
    row_e = tab["group_idx_for_bx"][rows // BT]
    E, I, H = w.experts, w.intermediate, w.hidden
    idx = torch.from_numpy(rows).cuda()
    up_all = ul.view(torch.int16)[idx].cpu().numpy().view(np.uint16)
    out_all = out.view(torch.int16)[idx].cpu().numpy().view(np.uint16)
    up_r = np.zeros_like(up_all)
    out_r = np.zeros_like(out_all)
    experts = np.unique(row_e)
    for b in range(0, experts.size, 16):
        batch = experts[b:b + 16]
        g_np = np.zeros((E, I, H), np.float16)
        u_np = np.zeros((E, I, H), np.float16)
        d_np = np.zeros((E, H, I), np.float16)
        for e in batch:
            g_np[e] = gate[e].cpu().numpy()
            u_np[e] = up[e].cpu().numpy()
            d_np[e] = down[e].cpu().numpy()
        sel = np.isin(row_e, batch)
        ur, orr, valid = oracle.forward_rows(xo, g_np, u_np, d_np, rwo, tab, rows[sel])
        assert valid.all()
        up_r[sel], out_r[sel] = ur, orr
        del g_np, u_np, d_np
    _check_rows(f"dsv3 T{w.tokens} k{w.top_k} E{E} H{H} I{I} ({rows.size} rows)", up_all, out_all, up_r, out_r)
    assert rows.size >= int(np.sum(-(-tab["group_sizes"] // BT)))
    # every padding row of out is untouched (checked on the device)
    valid_mask = torch.zeros(rows_total, dtype=torch.bool, device="cuda")
    valid_mask[side_g.pair_rows.reshape(-1).long()] = True
    pad_rows = out.view(torch.int16)[~valid_mask]
    assert bool((pad_rows == SENTINEL).all())


def test_run_kernel_page_signature():
    """run_kernel keeps the submission page's argument list ("Fused MoE GEMM
    提交说明", §提交文件): no up_logits argument (a cached workspace is used),
    out written in place, nothing returned; checked against the oracle, twice
    in a row on the same cached workspace."""
    raw = raw_inputs(small_workload(tokens=300, top_k=2, experts=3, hidden=256, intermediate=384), seed=8)
    side_o = oracle_prepare(raw)
    up_o = np.full((side_o.rows_total, raw.w.intermediate), SENTINEL, np.uint16)
    out_o = np.full((side_o.rows_total, raw.w.hidden), SENTINEL, np.uint16)
    oracle.fused_forward(side_o.x_packed, raw.gate, raw.up, raw.down, side_o.rw, side_o.tables, up_o, out_o)
    side = gpu_prepare(raw)
    t = side.tables
    from gpu_side import sentinel
    v = _valid_mask(side_o.pair_rows, side_o.rows_total)
    for call in range(2):
        out = sentinel(side.rows_total, raw.w.hidden)
        r = moe.run_kernel(side.x_packed, side.gate, side.up, side.down, side.rw, t["group_sizes"],
                           t["group_offsets"], t["group_padded_offsets"], t["group_idx_for_bx"], out)
        assert r is None
        torch.cuda.synchronize()
        got = bits(out)
        assert np.array_equal(got[~v], out_o[~v])
        ok = compare(_case(raw, f" run_kernel call{call}"), "out", got[v], out_o[v], ATOL, RTOL)
        assert ok.all()


def test_forward_at_block_and_expert_limits():
    """num_blocks_m = MOE_MAX_BLOCKS and n_experts = MOE_MAX_EXPERTS (H = I = 128,
    top-8 uniform routing over 245,760 tokens): the largest active-block list
    and unit list the kernels keep in shared memory.  A valid row of every
    active block against the oracle; every padding row untouched (checked on
    the device)."""
    E, k = moe.MAX_EXPERTS, 8
    T = (moe.MAX_BLOCKS - E) * BT // k
    w = small_workload(tokens=T, top_k=k, experts=E, hidden=128, intermediate=128)
    raw = raw_inputs(w, seed=5)
    side_o = oracle_prepare(raw)
    assert side_o.tables["num_blocks_m"] == moe.MAX_BLOCKS
    side_g = gpu_prepare(raw)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ul, out = run_forward(side_g, w.intermediate, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rows = _rows_every_block(side_o.tables, np.random.default_rng(2))
    up_r, out_r, valid = oracle.forward_rows(side_o.x_packed, raw.gate, raw.up, raw.down,
                                             side_o.rw, side_o.tables, rows)
    assert valid.all()
    idx = torch.from_numpy(rows).cuda()
    up_g = ul.view(torch.int16)[idx].cpu().numpy().view(np.uint16)
    out_g = out.view(torch.int16)[idx].cpu().numpy().view(np.uint16)
    _check_rows(_case(raw, f" limits ({rows.size} rows)"), up_g, out_g, up_r, out_r)
    valid_mask = torch.zeros(side_o.rows_total, dtype=torch.bool, device="cuda")
    valid_mask[side_g.pair_rows.reshape(-1).long()] = True
    assert bool((out.view(torch.int16)[~valid_mask] == SENTINEL).all())
    assert bool((ul.view(torch.int16)[~valid_mask] == SENTINEL).all())
    assert bool((out.view(torch.int16)[valid_mask] != SENTINEL).all())


# --------------------------------------------------------------------------
# both phases in one persistent launch
# --------------------------------------------------------------------------

def _run_single_launch(side, intermediate, status=None):
    from gpu_side import sentinel
    ul = sentinel(side.rows_total, intermediate)
    out = sentinel(side.rows_total, side.x_packed.shape[1])
    t = side.tables
    ws = torch.empty(moe.single_launch_workspace_bytes(t["group_idx_for_bx"].numel()), dtype=torch.uint8,
                     device="cuda")
    ws.fill_(0x5A)      # the call must zero its own counters
    moe.fused_forward(side.x_packed, side.gate, side.up, side.down, side.rw, t["group_sizes"],
                      t["group_offsets"], t["group_padded_offsets"], t["group_idx_for_bx"], ul, out,
                      status=status, single_launch_workspace=ws)
    return ul, out


@pytest.mark.parametrize("shape", [
    (300, 2, 3, 256, 384, "uniform"),
    (500, 4, 40, 384, 256, "uniform"),
    (32, 8, 128, 256, 256, "zipf"),
    (700, 1, 2, 512, 640, "zipf"),
])
def test_single_launch_matches_two_launches_bit_for_bit(shape):
    """Each tile is computed identically (same k order, same epilogue), so
    the one-launch forward must reproduce the two-launch forward exactly —
    including untouched padding rows — and stay within the oracle tolerance."""
    T, k, E, H, I, routing = shape
    w = small_workload(tokens=T, top_k=k, experts=E, hidden=H, intermediate=I,
                       routing=routing, zipf_s=1.2 if routing == "zipf" else 0.0)
    raw = raw_inputs(w, seed=6)
    side = gpu_prepare(raw)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ul2, out2 = run_forward(side, I)
    ul1, out1 = _run_single_launch(side, I, status=status)
    ul1b, out1b = _run_single_launch(side, I, status=status)     # twice: counters re-zeroed per call
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for a, b in ((ul1, ul2), (out1, out2), (ul1b, ul2), (out1b, out2)):
        assert np.array_equal(bits(a), bits(b))
    side_o = oracle_prepare(raw)
    up_o = np.full((side_o.rows_total, I), SENTINEL, np.uint16)
    out_o = np.full((side_o.rows_total, H), SENTINEL, np.uint16)
    oracle.fused_forward(side_o.x_packed, raw.gate, raw.up, raw.down, side_o.rw, side_o.tables, up_o, out_o)
    v = _valid_mask(side_o.pair_rows, side_o.rows_total)
    assert compare(_case(raw, " single launch"), "out", bits(out1)[v], out_o[v], ATOL, RTOL).all()


@pytest.mark.parametrize("name", ["dsv2_lite", "decode_skewed"])
def test_single_launch_full_size_matches_two_launches(name):
    w = workloads.WORKLOADS[name]
    raw = raw_inputs(w, seed=0)
    side = gpu_prepare(raw)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ul2, out2 = run_forward(side, w.intermediate)
    ul1, out1 = _run_single_launch(side, w.intermediate, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(bits(out1), bits(out2))
    assert np.array_equal(bits(ul1), bits(ul2))
