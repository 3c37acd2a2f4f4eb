#!/usr/bin/env python3
"""Benchmark of the routed fused-MoE expert GEMM on GB300.

One step = one pass of the whole hot path over one batch of synthetic routed
input already resident in HBM: the dispatch tables built on the GPU from
topk_ids (moe_build_dispatch), then phase 1 + phase 2 (moe_fused_forward).

Metric: fused MoE forward TFLOP/s over valid rows, 2·pairs·3·hidden·intermediate
per step ÷ step time, and the fraction of the roofline
max(FLOPs / tensor peak, bytes / HBM peak).  Default workload: the largest one,
DeepSeek-V3-shaped (16384 tokens, top-8 of 256 experts with Zipf(1.0)
popularity, hidden 7168, intermediate 2048; 22.5 GB of expert weights).  Every
non-tiny working set is far larger than the 129 MB L2, so back-to-back steps do
not reuse L2 between iterations.

Timing ("MetaX-TileLang工具链" §2.5: warm-up, then repeats; §2.5.2: mean,
median, p90, p99, std): W warm-up steps (continued until --settle-s seconds of
steps have run, so the power-capped clock has settled), then exactly K steps
between synchronisations, timed with CUDA events on the launching stream.  A
separate loop times steps one by one for the latency distribution, and another
times the dispatch builder, phase 1 and phase 2 apart for the per-kernel
rooflines.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle
instead (the reference arm: the pages' own kernel targets a MetaX C500 and
cannot run on this GPU).

Multi-GPU: the path does not shard inside one forward on one GPU; N ranks run
independent replicas of the workload ("replicas only"), value = units of all
ranks ÷ the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused MoE forward TFLOP/s (valid rows) and % of roofline on 1 GB300"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "dsv3"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CPU_SAMPLE_EXPERTS = 8      # the oracle samples rows of at most this many experts (bounded host memory)


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=800)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--settle-s", type=float, default=3.0,
                    help="warm-up continues until this many seconds of steps have run")
    ap.add_argument("--phase-steps", type=int, default=500,
                    help="steps of the per-kernel loop (outside the timed region)")
    ap.add_argument("--latency-steps", type=int, default=200,
                    help="steps timed one by one for the latency distribution")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle sample (cpu_baseline)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--eager", action="store_true",
                    help="launch every step from Python instead of replaying a captured CUDA graph")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# peaks, clocks, profiles, host
# ---------------------------------------------------------------------------

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in r.stdout.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, every 100 ms."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.rows = []
        self.proc = None
        self.thread = None
        self.t_begin = None
        self.t_end = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def mark_begin(self):
        self.t_begin = time.time()

    def mark_end(self):
        self.t_end = time.time()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        inside = [r for t, r in self.rows if self.t_begin and self.t_end and self.t_begin <= t <= self.t_end]
        used = inside
        if len(used) < 3 and self.t_begin and self.t_end:
            # a timed region shorter than a few sampling periods: take the
            # last second of the (settled) warm-up as well
            used = [r for t, r in self.rows if self.t_begin - 1.0 <= t <= self.t_end]
        if not used:
            used = [r for _, r in self.rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        sm, smax, pw = [], [], []
        for r in used:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
                pw.append(float(r[3]))
            except (ValueError, IndexError):
                continue
            for i, n in enumerate(names):
                if len(r) > 5 + i and r[5 + i].lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": sorted(reasons), "samples": len(used),
                "samples_in_timed_region": len(inside),
                "window": "timed region" if used is inside else "timed region and the second before it"}


def kernel_source_hash():
    """Hash of the GEMM kernels' code (comments and layout stripped), so that
    the DRAM traffic in profiles/ is only used for the kernel it was taken on."""
    import re
    h = hashlib.sha256()
    for rel in ("routed_grouped_gemm_dispatch_gb300/csrc/grouped_gemm.cu",
                "routed_grouped_gemm_dispatch_gb300/csrc/sm103_ptx.cuh"):
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def profile_traffic(workload: str, phase: int):
    """DRAM bytes per launch of one GEMM phase from the committed ncu summary,
    if it was taken on the current kernel source (else None)."""
    stem = "phase1_gate_up" if phase == 1 else "phase2_down"
    path = os.path.join(ROOT, "profiles", f"{stem}_{workload}.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha") != kernel_source_hash():
            return None
        return float(kv["dram_bytes_per_launch_full_size"])
    except (OSError, KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# algorithmic work (host arithmetic on the group sizes)
# ---------------------------------------------------------------------------

def work_stats(w, sizes) -> dict:
    """Algorithmic FLOPs and bytes per phase, and the padding statistics of the
    grouped layout, from the workload's shape and its group sizes.

    Bytes count every touched expert's weights once, every valid row's
    activations once (x read, up_logits written and read back, out written,
    routed weight read) and nothing for padding rows or re-reads.  Padding:
    the allocated rows (num_blocks_m·128), the rows the page's "+1" rule pads
    the groups to (Σ ceil((c+1)/128)·128) and the rows the kernels' 2-SM tiles
    execute (each pair of an expert's active blocks is one 256-row MMA tile,
    each lone active block one 128-row tile)."""
    import numpy as np
    sizes = np.asarray(sizes, np.int64)
    P, H, I, E = w.pairs, w.hidden, w.intermediate, w.experts
    touched = int(np.count_nonzero(sizes))
    active = -(-sizes // 128)
    units = active // 2 + active % 2
    m_blocks = -(-P // 128) + E
    padded = int(np.sum(-(-(sizes + 1) // 128) * 128))
    executed = int(256 * (active // 2).sum() + 128 * (active % 2).sum())
    return {
        "pairs": P, "touched_experts": touched, "active_blocks": int(active.sum()),
        "tile_units": int(units.sum()), "alloc_rows": int(m_blocks * 128), "padded_rows": padded,
        "padding_waste_rows": int(m_blocks * 128 - P), "padded_minus_valid_rows": padded - P,
        "executed_mma_rows": executed, "executed_row_ratio": executed / P if P else 0.0,
        "flops": 6.0 * P * H * I, "flops_phase1": 4.0 * P * H * I, "flops_phase2": 2.0 * P * H * I,
        "weight_bytes": 6.0 * H * I * touched,
        "weight_bytes_phase1": 4.0 * H * I * touched, "weight_bytes_phase2": 2.0 * H * I * touched,
        "activation_bytes": P * (2.0 * H + 2.0 * H + 4.0 + 4.0 * I),
        "activation_bytes_no_up_logits": P * (2.0 * H + 2.0 * H + 4.0),
        "activation_bytes_phase1": P * (2.0 * H + 2.0 * I),
        "activation_bytes_phase2": P * (2.0 * I + 2.0 * H + 4.0),
    }


def touched_bytes(w, sizes):
    """(touched-expert weight bytes, activation bytes, touched experts)."""
    s = work_stats(w, sizes)
    return s["weight_bytes"], s["activation_bytes"], s["touched_experts"]


def kernel_roofline(name, flops, nbytes, ms, tc_peak, hbm_peak, tc_label, traffic=None, extra=None):
    """Roofline of one kernel: bound = whichever of FLOP time and byte time is
    larger; achieved in that resource's unit ÷ its peak."""
    t_flop = flops / (tc_peak * 1e12)
    t_byte = nbytes / (hbm_peak * 1e9)
    if t_flop >= t_byte:
        r = {"kernel": name, "bound": "tensor", "achieved": flops / (ms * 1e-3) / 1e12, "peak": tc_peak,
             "unit": "TFLOP/s"}
    else:
        r = {"kernel": name, "bound": "hbm", "achieved": nbytes / (ms * 1e-3) / 1e9, "peak": hbm_peak,
             "unit": "GB/s"}
    r["frac"] = r["achieved"] / r["peak"]
    r.update({"traffic": traffic, "launch_ms": ms, "algorithmic_flops_per_launch": flops,
              "algorithmic_bytes_per_launch": nbytes, "t_flop_ms": 1e3 * t_flop, "t_byte_ms": 1e3 * t_byte,
              "tensor_peak_kind": tc_label})
    if extra:
        r.update(extra)
    return r


def graph_time(fn, dev, per_graph=20, replays=10):
    """Device time of one call of `fn` (its kernels back to back): `per_graph`
    calls captured in a CUDA graph, replayed `replays` times after one warm
    replay, timed with CUDA events on the capturing stream; the mean per call."""
    import torch
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for _ in range(2):
            fn()
    torch.cuda.current_stream(dev).wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(per_graph):
            fn()
    g.replay()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(replays):
        g.replay()
    b.record()
    torch.cuda.synchronize(dev)
    return a.elapsed_time(b) / (replays * per_graph)


def latency_stats(ms_list):
    import numpy as np
    a = np.asarray(ms_list, np.float64)
    return {"n": int(a.size), "mean": float(a.mean()), "median": float(np.median(a)),
            "p90": float(np.percentile(a, 90)), "p99": float(np.percentile(a, 99)),
            "std": float(a.std(ddof=1)) if a.size > 1 else 0.0, "min": float(a.min()), "max": float(a.max())}


# ---------------------------------------------------------------------------
# workload preparation
# ---------------------------------------------------------------------------

def prepare_device(w, seed, dev):
    """Routing, tokens and expert weights; GPU tables and packing."""
    import torch

    import routed_grouped_gemm_dispatch_gb300 as moe
    import workloads

    ids_np, tw_np = workloads.routing(w, seed)
    x_np = workloads.tokens(w, seed)
    gate, up, down = workloads.expert_weights(w, seed, device=str(dev))
    ids = torch.from_numpy(ids_np).to(dev)
    tables = moe.build_dispatch(ids, w.experts)
    rows_total = tables["group_idx_for_bx"].numel() * moe.BLOCK_TOKEN
    x_tok = torch.from_numpy(x_np).to(dev)
    tw = torch.from_numpy(tw_np).to(dev)
    pk = moe.pack_routed(ids, tw, x_tok, tables, rows_total)
    xp, rw, rows = pk["stacked_expert_tokens"], pk["routed_expert_weights"], pk["pair_padded_rows"]
    ul = torch.zeros((rows_total, w.intermediate), dtype=torch.float16, device=dev)
    out = torch.zeros((rows_total, w.hidden), dtype=torch.float16, device=dev)
    torch.cuda.synchronize(dev)
    return dict(ids=ids, tables=tables, xp=xp, rw=rw, ul=ul, out=out, gate=gate, up=up, down=down,
                ids_np=ids_np, tw_np=tw_np, x_np=x_np, rows_total=rows_total, pair_rows=rows,
                x_tok=x_tok, tw=tw)


# ---------------------------------------------------------------------------
# oracle timing (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------

class OracleSample:
    """A bounded sample of the workload for the CPU oracle: valid rows of at
    most CPU_SAMPLE_EXPERTS experts, with host copies of those experts'
    weights only (the other experts' slices are never read and stay
    unallocated zero pages).  Every valid row costs the oracle the same
    6·H·I FLOPs whatever its expert, so the rate is that of the workload."""

    def __init__(self, w, seed, weights_of, experts_from_front=False):
        import numpy as np

        import oracle
        import workloads
        self.w = w
        ids_np, tw_np = workloads.routing(w, seed)
        x_np = workloads.tokens(w, seed)
        self.tab = oracle.build_dispatch(ids_np, w.experts)
        prow = oracle.pair_padded_rows(ids_np, w.experts, self.tab["group_padded_offsets"])
        rows_total = self.tab["num_blocks_m"] * oracle.BLOCK_TOKEN
        self.xo, self.rwo = oracle.pack(x_np, ids_np, tw_np, prow, self.tab, rows_total)
        sizes = self.tab["group_sizes"]
        nonempty = np.nonzero(sizes)[0]
        rng = np.random.default_rng(seed + 17)
        n_e = min(CPU_SAMPLE_EXPERTS, nonempty.size)
        if experts_from_front:
            chosen = nonempty[:n_e]
        else:
            chosen = np.sort(rng.choice(nonempty, size=n_e, replace=False))
        self.how = "first non-empty" if experts_from_front else "randomly chosen"
        self.experts = [int(e) for e in chosen]
        E, I, H = w.experts, w.intermediate, w.hidden
        self.g = np.zeros((E, I, H), np.float16)
        self.u = np.zeros((E, I, H), np.float16)
        self.d = np.zeros((E, H, I), np.float16)
        for e, (ge, ue, de) in zip(self.experts, weights_of(self.experts)):
            self.g[e], self.u[e], self.d[e] = ge, ue, de
        ex = np.zeros(E, bool)
        ex[self.experts] = True
        flat = prow.reshape(-1)
        self.valid = flat[ex[ids_np.reshape(-1)]]
        self.n_valid_total = flat.size
        self.threads = len(os.sched_getaffinity(0))
        self.rng = np.random.default_rng(seed)
        self.per_row_flops = 6.0 * H * I

    def run(self, n, n_threads=None):
        import oracle
        rows = self.rng.choice(self.valid, size=min(n, self.valid.size), replace=False)
        t0 = time.perf_counter()
        oracle.forward_rows(self.xo, self.g, self.u, self.d, self.rwo, self.tab, rows,
                            n_threads=self.threads if n_threads is None else n_threads)
        return rows.size, time.perf_counter() - t0

    def describe(self, n):
        return (f"{n} randomly chosen valid rows (of the {self.valid.size} rows of {len(self.experts)} "
                f"{self.how} experts; {self.n_valid_total} valid rows in all), each row's full "
                f"phase 1 and phase 2 with fp32 accumulation, {self.threads} OpenMP threads")

    def rate(self, target_s):
        """(TFLOP/s, rows, seconds) of a sample sized to take about target_s."""
        n0 = min(self.valid.size, max(self.threads, 8))
        _, t0 = self.run(n0)
        n = int(min(self.valid.size, max(n0, round(n0 * target_s / max(t0, 1e-6)))))
        n, dt = self.run(n)
        return n * self.per_row_flops / dt / 1e12, n, dt


def tiny_single_thread():
    """The oracle's whole forward on the tiny workload with one thread:
    (TFLOP/s, seconds per forward, best of 3)."""
    import numpy as np

    import oracle
    import workloads
    w = workloads.WORKLOADS["tiny"]
    ids, tw = workloads.routing(w, 0)
    x = workloads.tokens(w, 0)
    g, u, d = (t.numpy() for t in workloads.expert_weights(w, 0, device="cpu"))
    tab = oracle.build_dispatch(ids, w.experts)
    prow = oracle.pair_padded_rows(ids, w.experts, tab["group_padded_offsets"])
    xo, rwo = oracle.pack(x, ids, tw, prow, tab, tab["num_blocks_m"] * oracle.BLOCK_TOKEN)
    best = np.inf
    for _ in range(3):
        t0 = time.perf_counter()
        oracle.fused_forward(xo, g, u, d, rwo, tab, n_threads=1)
        best = min(best, time.perf_counter() - t0)
    return w.flops() / best / 1e12, best


def _cpu_weights_front(w, seed):
    """Weights for the reference arm, drawn on the host for the first experts only."""
    import workloads

    def weights_of(experts):
        n = max(experts) + 1
        g, u, d = workloads.expert_weights(w, seed, device="cpu", experts=n)
        return [(g[e].numpy(), u[e].numpy(), d[e].numpy()) for e in experts]
    return weights_of


def reference_arm(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    # size each step so that warmup + steps finish within ~3 minutes
    budget = 180.0 / max(1, args.steps + args.warmup)
    per_step_target = max(0.2, min(3.0, budget))
    smp = OracleSample(w, args.seed, _cpu_weights_front(w, args.seed), experts_from_front=True)
    rate0, _, _ = smp.rate(per_step_target)
    n = max(1, int(rate0 * 1e12 * per_step_target / smp.per_row_flops))
    n = min(n, smp.valid.size)
    times = []
    for i in range(args.warmup + args.steps):
        n_done, dt = smp.run(n)
        if i >= args.warmup:
            times.append(dt)
    ms = 1e3 * sum(times) / len(times)
    value = n_done * smp.per_row_flops / (ms / 1e3) / 1e12
    sample = "per step " + smp.describe(n_done)
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": config_of(w, "host cores; bounded sample per step"),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": smp.threads, "kind": "oracle",
                             "sample": sample, "cpu_model": cpu_model()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "latency_ms": latency_stats([1e3 * t for t in times]),
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def max_over_ranks(ms, dist, device):
    """The job's step time: the slowest rank's (one all-reduce; identity on one rank)."""
    if dist is None:
        return ms
    import torch
    tt = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def job_value(world, flops_per_rank, ms):
    """Whole-job TFLOP/s: every rank runs its own replica of the workload
    (weak scaling), so the job does world x the per-rank FLOPs per step."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


def config_of(w, l2):
    return {"workload": w.name, "tokens": w.tokens, "top_k": w.top_k, "experts": w.experts,
            "hidden": w.hidden, "intermediate": w.intermediate, "pairs": w.pairs,
            "routing": w.routing + (f"(s={w.zipf_s})" if w.routing == "zipf" else ""),
            "block_token": 128, "l2": l2}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def main(argv=None):
    args = parse_args(argv)
    import workloads
    w = workloads.WORKLOADS[args.workload]
    if args.impl == "reference":
        reference_arm(args, w)
        return

    import numpy as np
    import torch

    import routed_grouped_gemm_dispatch_gb300 as moe
    moe.lib()  # fail loudly if the library is missing

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    def barrier():
        if dist is not None:
            dist.barrier()

    d = prepare_device(w, args.seed + rank, dev)
    t = d["tables"]
    E = w.experts

    def step():
        moe.build_dispatch(d["ids"], E, out=t)
        moe.fused_forward(d["xp"], d["gate"], d["up"], d["down"], d["rw"], t["group_sizes"],
                          t["group_offsets"], t["group_padded_offsets"], t["group_idx_for_bx"],
                          d["ul"], d["out"])

    props = torch.cuda.get_device_properties(dev)
    gpu_id = str(getattr(props, "uuid", local))
    if gpu_id and not gpu_id.startswith("GPU-") and len(gpu_id) > 8:
        gpu_id = "GPU-" + gpu_id
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.3)

    status = torch.zeros(1, dtype=torch.int32, device=dev)
    run_step = step
    run_one = step
    per_replay = 1          # steps per launch of run_step
    if not args.eager:
        # S consecutive steps (each: dispatch tables, phase 1, phase 2 with its
        # programmatic dependency) captured as one CUDA graph, replayed
        # steps / S times; S = 8 when it divides the step count, which spreads
        # the graph-launch gap (~3 us) over 8 steps.  A one-step graph serves
        # the latency loop.
        per_replay = 8 if args.steps % 8 == 0 else 1
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            for _ in range(3):
                step()
        torch.cuda.current_stream(dev).wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(per_replay):
                step()
        run_step = graph.replay
        graph1 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph1):
            step()
        run_one = graph1.replay

    # warm-up: at least W steps (and 3), continued until settle_s seconds of
    # steps have run so that the timed region sees the settled clock
    warm_launches = 0
    t_settle = time.perf_counter()
    while True:
        run_step()
        warm_launches += 1
        if warm_launches * per_replay >= max(3, args.warmup):
            torch.cuda.synchronize(dev)
            if time.perf_counter() - t_settle >= args.settle_s:
                break
    warmup_steps = warm_launches * per_replay
    torch.cuda.synchronize(dev)
    barrier()
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    sampler.mark_begin()
    ev0.record()
    for _ in range(args.steps // per_replay):
        run_step()
    ev1.record()
    torch.cuda.synchronize(dev)
    sampler.mark_end()
    barrier()
    ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, dist, dev)
    sampler.stop()
    flops = w.flops()
    value = job_value(world, flops, ms)

    # ---- latency distribution: steps timed one by one ----------------------
    n_lat = max(10, args.latency_steps)
    lat_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_lat)]
    for a_, b_ in lat_ev:
        a_.record()
        run_one()
        b_.record()
    torch.cuda.synchronize(dev)
    latency = latency_stats([a_.elapsed_time(b_) for a_, b_ in lat_ev])

    # ---- per-kernel durations (same stream, CUDA events) -------------------
    # a fixed number of steps whatever --steps is, so the power-capped clock
    # settles as in the timed loop; the second half is averaged
    n_ph = max(6, args.phase_steps)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_ph)]
    for i in range(n_ph):
        e = evs[i]
        e[0].record()
        moe.build_dispatch(d["ids"], E, out=t)
        e[1].record()
        moe.fused_forward(d["xp"], d["gate"], d["up"], d["down"], d["rw"], t["group_sizes"],
                          t["group_offsets"], t["group_padded_offsets"], t["group_idx_for_bx"],
                          d["ul"], d["out"], status=status, flags=moe.MOE_RUN_PHASE1)
        e[2].record()
        moe.fused_forward(d["xp"], d["gate"], d["up"], d["down"], d["rw"], t["group_sizes"],
                          t["group_offsets"], t["group_padded_offsets"], t["group_idx_for_bx"],
                          d["ul"], d["out"], status=status, flags=moe.MOE_RUN_PHASE2 | moe.MOE_NO_PDL)
        e[3].record()
    torch.cuda.synchronize(dev)
    steady = evs[n_ph // 2:]
    dispatch_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in steady)
    p1_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in steady)
    p2_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in steady)
    dev_status = int(status.item())

    # ---- end to end through the public API with host buffers ---------------
    # token-major inputs in pinned host memory -> H2D -> dispatch tables ->
    # pack -> phase 1 + phase 2 -> combine -> D2H of the token outputs, every
    # step.  Pipelined the way a serving loop runs it: two slots of device
    # staging buffers; step i's H2D runs on its own stream while step i-1
    # computes, and its D2H on a third stream while step i+1 computes.  The
    # serial form (everything on one stream) is timed too.
    e2e = None
    pack_ms = combine_ms = None
    if not args.no_e2e:
        h_ids = d["ids"].cpu().pin_memory()
        h_x = d["x_tok"].cpu().pin_memory()
        h_tw = d["tw"].cpu().pin_memory()
        T = h_x.shape[0]
        h_y = [torch.empty((T, w.hidden), dtype=torch.float16).pin_memory() for _ in range(2)]
        d_ids = [torch.empty_like(d["ids"]) for _ in range(2)]
        d_x = [torch.empty_like(d["x_tok"]) for _ in range(2)]
        d_tw = [torch.empty_like(d["tw"]) for _ in range(2)]
        d_y = [torch.empty((T, w.hidden), dtype=torch.float16, device=dev) for _ in range(2)]
        ws = torch.empty(max(16, int(moe.lib().moe_pack_workspace_bytes(w.pairs, E))), dtype=torch.uint8,
                         device=dev)
        prows = torch.empty((T, w.top_k), dtype=torch.int32, device=dev)
        n_e2e = max(5, min(args.steps, 100))
        comp = torch.cuda.current_stream(dev)
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]      # the slot's inputs have landed
        ev_used = [torch.cuda.Event() for _ in range(2)]    # pack has read the slot's inputs
        ev_y = [torch.cuda.Event() for _ in range(2)]       # the slot's token outputs are ready
        ev_out = [torch.cuda.Event() for _ in range(2)]     # the slot's outputs have left
        for e_ in ev_used + ev_out:
            e_.record(comp)

        def pack(ids_, x_, tw_):
            moe.pack_routed(ids_, tw_, x_, t, d["rows_total"], stacked=d["xp"], routed_weights=d["rw"],
                            pair_rows=prows, workspace=ws)

        def compute(ids_, x_, tw_, y_):
            moe.build_dispatch(ids_, E, out=t)
            pack(ids_, x_, tw_)
            return lambda: (moe.fused_forward(d["xp"], d["gate"], d["up"], d["down"], d["rw"],
                                              t["group_sizes"], t["group_offsets"], t["group_padded_offsets"],
                                              t["group_idx_for_bx"], d["ul"], d["out"]),
                            moe.combine_routed(d["out"], prows, y=y_))

        def e2e_step(i):
            sl = i % 2
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_used[sl])
                d_ids[sl].copy_(h_ids, non_blocking=True)
                d_x[sl].copy_(h_x, non_blocking=True)
                d_tw[sl].copy_(h_tw, non_blocking=True)
                ev_in[sl].record(s_in)
            comp.wait_event(ev_in[sl])
            rest = compute(d_ids[sl], d_x[sl], d_tw[sl], d_y[sl])
            ev_used[sl].record(comp)
            comp.wait_event(ev_out[sl])
            rest()
            ev_y[sl].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_y[sl])
                h_y[sl].copy_(d_y[sl], non_blocking=True)
                ev_out[sl].record(s_out)

        def e2e_step_serial():
            d_ids[0].copy_(h_ids, non_blocking=True)
            d_x[0].copy_(h_x, non_blocking=True)
            d_tw[0].copy_(h_tw, non_blocking=True)
            compute(d_ids[0], d_x[0], d_tw[0], d_y[0])()
            h_y[0].copy_(d_y[0], non_blocking=True)

        for i in range(4):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(comp)
        s_in.wait_event(a)
        for i in range(n_e2e):
            e2e_step(i)
        comp.wait_stream(s_out)
        b.record(comp)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(a.elapsed_time(b) / n_e2e, dist, dev)
        for _ in range(3):
            e2e_step_serial()
        torch.cuda.synchronize(dev)
        a.record(comp)
        for _ in range(n_e2e):
            e2e_step_serial()
        b.record(comp)
        torch.cuda.synchronize(dev)
        serial_ms = max_over_ranks(a.elapsed_time(b) / n_e2e, dist, dev)
        y_ok = bool(torch.equal(h_y[0].to(dev), d_y[0]))
        h2d = h_ids.numel() * 4 + h_x.numel() * 2 + h_tw.numel() * 4
        d2h = h_y[0].numel() * 2
        e2e = {"value": job_value(world, flops, e2e_ms), "unit": UNIT, "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "steps": n_e2e, "gpu_launches_per_step": 7, "pipelined": True,
               "serial_ms_per_step": serial_ms,
               "serial_value": job_value(world, flops, serial_ms),
               "host_copy_matches_device": y_ok,
               "path": "pinned host tokens [T,H] + topk_ids + topk weights -> H2D -> moe_build_dispatch -> "
                       "moe_pack_routed -> moe_fused_forward -> moe_combine_routed -> D2H token outputs [T,H]; "
                       "copies on two side streams with double-buffered staging, overlapping the "
                       "neighbouring steps' compute"}

        # pack (three launches) and combine timed apart from graph replays
        # (no host launch overhead between kernels)
        pack_ms = graph_time(lambda: pack(d["ids"], d["x_tok"], d["tw"]), dev)
        combine_ms = graph_time(lambda: moe.combine_routed(d["out"], prows, y=d_y[0]), dev)

    # ---- timing scopes of the evaluation page: the whole MoE layer ---------
    # cached_e2e: router -> dispatch -> pack -> forward -> combine on tokens
    # already on the device, all buffers reused (routing from a random router,
    # so it is near-uniform whatever the workload's own routing is);
    # e2e_host: the same with the tokens copied in and the outputs copied out.
    scopes = None
    router_ms = None
    if not args.no_e2e and E <= moe.ROUTER_MAX_EXPERTS:
        wg = torch.from_numpy(workloads.router_weights(w, args.seed + rank)).to(dev)
        ids_l = torch.empty_like(d["ids"])
        tw_l = torch.empty_like(d["tw"])
        prows_l = torch.empty((w.tokens, w.top_k), dtype=torch.int32, device=dev)
        ws_l = torch.empty(max(16, int(moe.lib().moe_pack_workspace_bytes(w.pairs, E))), dtype=torch.uint8,
                           device=dev)
        y_l = torch.empty((w.tokens, w.hidden), dtype=torch.float16, device=dev)
        h_xl = d["x_tok"].cpu().pin_memory()
        h_yl = torch.empty((w.tokens, w.hidden), dtype=torch.float16).pin_memory()
        x_l = torch.empty_like(d["x_tok"])
        x_l.copy_(d["x_tok"])
        t_l = {key: torch.empty_like(val) for key, val in t.items()}   # the layer's own tables

        def layer(x_in):
            moe.router_topk(x_in, wg, w.top_k, topk_ids=ids_l, topk_weights=tw_l)
            moe.build_dispatch(ids_l, E, out=t_l)
            moe.pack_routed(ids_l, tw_l, x_in, t_l, d["rows_total"], stacked=d["xp"], routed_weights=d["rw"],
                            pair_rows=prows_l, workspace=ws_l)
            moe.fused_forward(d["xp"], d["gate"], d["up"], d["down"], d["rw"], t_l["group_sizes"],
                              t_l["group_offsets"], t_l["group_padded_offsets"], t_l["group_idx_for_bx"],
                              d["ul"], d["out"])
            moe.combine_routed(d["out"], prows_l, y=y_l)

        def layer_host():
            x_l.copy_(h_xl, non_blocking=True)
            layer(x_l)
            h_yl.copy_(y_l, non_blocking=True)

        def time_fn(fn, n):
            for _ in range(3):
                fn()
            torch.cuda.synchronize(dev)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(n):
                fn()
            b.record()
            torch.cuda.synchronize(dev)
            return a.elapsed_time(b) / n

        n_sc = max(5, min(args.steps, 100))
        cached_ms = max_over_ranks(time_fn(lambda: layer(x_l), n_sc), dist, dev)
        host_ms = max_over_ranks(time_fn(layer_host, n_sc), dist, dev)
        router_ms = graph_time(lambda: moe.router_topk(x_l, wg, w.top_k, topk_ids=ids_l, topk_weights=tw_l), dev)
        router_flops = 2.0 * w.tokens * w.hidden * w.experts
        scopes = {"routed_kernel_only_ms": ms, "cached_e2e_ms": cached_ms, "e2e_host_ms": host_ms,
                  "cached_e2e_tflops": job_value(world, flops + router_flops, cached_ms),
                  "e2e_host_tflops": job_value(world, flops + router_flops, host_ms),
                  "flops_note": "expert FLOPs 6*P*H*I plus router 2*T*H*E; routing from a random "
                                "router (near-uniform), not the workload's own routing",
                  "launches_per_layer": 8}

    # ---- rooflines ---------------------------------------------------------------
    peaks, src = load_peaks()
    ws_ = work_stats(w, t["group_sizes"].cpu().numpy())
    tc_burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    tc_sust = float(peaks.get("bf16_tflops_sustained", tc_burst))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    # the per-kernel loop runs hundreds of back-to-back steps under the power
    # cap, so its kernels are held against the sustained dense peak (the burst
    # fraction is given beside it)
    tc_label = f"{src} bf16 dense sustained (fp16 dense rate is the same on this part)"
    H, I = w.hidden, w.intermediate
    k1 = kernel_roofline("grouped_gemm_kernel<1> (phase 1: gate+up GEMM, SiLU·up epilogue)",
                         ws_["flops_phase1"], ws_["weight_bytes_phase1"] + ws_["activation_bytes_phase1"],
                         p1_ms, tc_sust, hbm, tc_label, traffic=profile_traffic(w.name, 1))
    k2 = kernel_roofline("grouped_gemm_kernel<2> (phase 2: down GEMM, routed-weight epilogue)",
                         ws_["flops_phase2"], ws_["weight_bytes_phase2"] + ws_["activation_bytes_phase2"],
                         p2_ms, tc_sust, hbm, tc_label, traffic=profile_traffic(w.name, 2))
    for k in (k1, k2):
        if k["bound"] == "tensor":
            k["frac_vs_burst_peak"] = k["achieved"] / tc_burst
            k["burst_peak"] = tc_burst
    kd = kernel_roofline("build_dispatch_kernel", 0.0, 4.0 * w.pairs + 4.0 * (3 * E + 2 + ws_["alloc_rows"] // 128),
                         dispatch_ms, tc_sust, hbm, tc_label)
    kernels = [k1, k2, kd]
    if pack_ms is not None:
        kernels.append(kernel_roofline(
            "pack (rank_chunks_kernel + scan_chunks_kernel + place_pairs_kernel)", 0.0,
            w.tokens * 2.0 * H + w.pairs * (2.0 * H + 4 + 4 + 4 + 4) + 4.0 * w.pairs, pack_ms, tc_sust, hbm,
            tc_label,
            extra={"bytes_note": "per token: its row read once 2H; per pair: packed row written 2H + id, "
                                 "weight, compact weight, padded row; ids read once more for the ranks"}))
        kernels.append(kernel_roofline(
            "combine_kernel", 0.0, w.pairs * (2.0 * H + 4) + w.tokens * 2.0 * H, combine_ms, tc_sust, hbm,
            tc_label, extra={"bytes_note": "per pair: expert row read 2H + its padded row 4; per token: "
                                           "output row written 2H"}))
    if router_ms is not None:
        kernels.append(kernel_roofline(
            "router_kernel", 2.0 * w.tokens * H * E, 2.0 * w.tokens * H + 2.0 * E * H + 8.0 * w.pairs,
            router_ms, tc_sust, hbm, tc_label))
    roof = max((k1, k2), key=lambda k: k["launch_ms"])     # the dominant kernel of the step

    t_flop = ws_["flops"] / (tc_burst * 1e12)
    t_flop_s = ws_["flops"] / (tc_sust * 1e12)
    t_byte = (ws_["weight_bytes"] + ws_["activation_bytes"]) / (hbm * 1e9)
    t_byte_nul = (ws_["weight_bytes"] + ws_["activation_bytes_no_up_logits"]) / (hbm * 1e9)
    forward_roofline = {
        "t_roof_ms": 1e3 * max(t_flop, t_byte), "t_flop_ms": 1e3 * t_flop, "t_byte_ms": 1e3 * t_byte,
        "t_byte_ms_without_up_logits": 1e3 * t_byte_nul,
        "bound": "tensor" if t_flop >= t_byte else "hbm",
        "frac_of_step": 1e3 * max(t_flop, t_byte) / ms,
        "frac_of_step_vs_sustained_peak": 1e3 * max(t_flop_s, t_byte) / ms,
        "phase1_ms": p1_ms, "phase2_ms": p2_ms, "dispatch_ms": dispatch_ms, "step_ms": ms,
        "peaks": f"{src}: {tc_burst} TFLOP/s burst, {tc_sust} TFLOP/s sustained "
                 f"(power-capped back-to-back GEMMs), {hbm} GB/s"}
    work = {k: ws_[k] for k in ("pairs", "touched_experts", "active_blocks", "tile_units", "alloc_rows",
                                "padded_rows", "padding_waste_rows", "padded_minus_valid_rows",
                                "executed_mma_rows", "executed_row_ratio", "weight_bytes", "activation_bytes",
                                "activation_bytes_no_up_logits")}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        def weights_of(experts):
            return [(d["gate"][e].cpu().numpy(), d["up"][e].cpu().numpy(), d["down"][e].cpu().numpy())
                    for e in experts]
        smp = OracleSample(w, args.seed, weights_of)
        rate, n, secs = smp.rate(args.cpu_seconds)
        tiny_rate, tiny_s = tiny_single_thread()
        cpu = {"value": rate, "unit": UNIT, "cores": smp.threads, "kind": "oracle", "sample": smp.describe(n),
               "seconds": secs, "cpu_model": cpu_model(),
               "tiny_single_thread": {"value": tiny_rate, "unit": UNIT, "seconds_per_forward": tiny_s,
                                      "threads": 1, "sample": "the whole tiny forward (128 valid rows)"}}

    if rank == 0:
        clocks = sampler.summary()
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": warmup_steps, "ms_per_step": ms, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
                "config": config_of(w, "working set larger than L2 (no flush needed)"),
                "parallelism": "replicas only" if world > 1 else "single GPU",
                "roofline": roof, "forward_roofline": forward_roofline, "kernels": kernels,
                "latency_ms": latency, "work": work,
                "cpu_baseline": cpu, "e2e": e2e, "scopes": scopes, "clocks": clocks,
                "gpu_launches": 3 * args.steps, "device_status": dev_status,
                "launch_mode": "eager" if args.eager else
                f"cuda_graph ({per_replay} step(s) captured per graph, replayed steps/{per_replay} times)",
                "warmup_note": f"at least {max(3, args.warmup)} warm-up steps, continued for "
                               f"{args.settle_s:g} s so the timed region runs at the settled clock",
                "kernel_source_sha": kernel_source_hash()}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
