"""The multi-rank host logic of bench.py, on CPU with the gloo backend at world
size 2: the job's step time is the slowest rank's (one all-reduce), the job
value counts every rank's replica (weak scaling: replicas only, no data-path
collective), and the reference arm runs on rank 0 alone while the other ranks
exit 0 without output."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, ms_by_rank, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = bench.max_over_ranks(ms_by_rank[rank], dist, "cpu")
    out_q.put((rank, ms, bench.job_value(world, 2.0e12, ms)))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_job_value_with_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    ms_by_rank = [1.25, 4.0]
    procs = [ctx.Process(target=_worker, args=(r, world, port, ms_by_rank, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _ in res] == [0, 1]
    for _, ms, value in res:
        assert ms == 4.0                                   # the slowest rank
        assert abs(value - world * 2.0e12 / 4.0e-3 / 1e12) < 1e-9


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert abs(bench.job_value(1, 1.0e12, 1.0) - 1.0e3) < 1e-9


def _reference_arm(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--workload", "tiny", "--steps", "1", "--warmup", "0", "--gpus", "2"],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_other_ranks_exit_quietly():
    r = _reference_arm(1)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_rank0_prints_one_line():
    r = _reference_arm(0)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
