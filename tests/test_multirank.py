"""The N > 1 host path of bench.py on the CPU with two gloo ranks.

Each GPU runs an independent replica (the forward has no exchange step), so
what multi-rank adds is host logic: the process-group setup, the barrier
around the timed region, the maximum of the ranks' times, and rank 0 alone
printing the JSON line.  These run here on CPU processes.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _helpers_rank(rank: int, world: int, port: int, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench

    dist, w, r, local = bench.dist_setup(world)
    bench.barrier(dist)
    m = bench.max_over_ranks(dist, 10.0 * rank + 1.5, torch.device("cpu"))
    bench.barrier(dist)
    out.put((r, w, m))
    dist.destroy_process_group()


def test_dist_helpers_two_gloo_ranks():
    world, port = 2, free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_helpers_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(world))
    # every rank sees the maximum over ranks (rank 1's 11.5)
    assert got == [(0, 2, 11.5), (1, 2, 11.5)]


def test_single_process_needs_no_process_group(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    sys.path.insert(0, ROOT)
    import bench

    dist, w, r, local = bench.dist_setup(1)
    assert dist is None and (w, r, local) == (1, 0, 0)
    assert bench.max_over_ranks(None, 3.0, torch.device("cpu")) == 3.0


@pytest.mark.timeout(300)
def test_reference_arm_under_torchrun_two_ranks():
    """The launch the benchmark driver uses for N = 2: rank 0 alone runs the
    reference arm and prints one JSON line; the other rank exits 0 silently."""
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "3", "--workload", "mha_l256_d64"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=280, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
