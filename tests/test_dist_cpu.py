"""bench.py's multi-rank host logic on the CPU, two ranks over gloo.

With several GPUs every rank runs the whole workload on its own device (the
(b, hq) problems need no exchange, so no collective touches the data path);
the ranks meet only at barriers around the timed region and in a max over
ranks of the timings.  These tests run that host logic with world size 2 on
the CPU: the max-reduction and barrier helpers over gloo, and the reference
arm launched the way a multi-GPU run launches it (rank 0 alone prints one
line, the other ranks exit 0 without work).
"""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, ws: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    got_ws, got_rank, _ = bench.dist_info()
    bench.init_dist(got_ws, "gloo")
    bench.barrier(got_ws)
    m = bench.reduce_max(1.5 * (got_rank + 1), got_ws)
    bench.barrier(got_ws)
    q.put((got_rank, got_ws, m))
    torch.distributed.destroy_process_group()


def test_reduce_max_and_barrier_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        results = sorted(q.get(timeout=120) for _ in range(2))
    finally:
        for p in procs:
            p.join(timeout=60)
    assert results == [(0, 2, 3.0), (1, 2, 3.0)]
    assert all(p.exitcode == 0 for p in procs)


def test_single_rank_helpers_are_noops():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(2.5, 1) == 2.5
    bench.barrier(1)  # no process group needed


def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    env = dict(os.environ, OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--workload", "selfattn_b1_h1_n128_d64", "--steps", "2", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
