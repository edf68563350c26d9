"""The N > 1 path on the CPU: two gloo ranks (no GPU).

Every output element is independent, so multi-GPU runs are replicas: each rank
runs its own copy, and the only cross-rank steps are a barrier and the maximum
of the ranks' times.  These tests run that host logic as world-size-2 process
groups over gloo, and the reference arm under torchrun.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    try:
        d.barrier()
        slowest = d.max(1.5 + rank)                 # rank r "took" 1.5 + r seconds
        value = bench.aggregate(3.0e9, d.world, slowest)
        q.put((rank, d.world, slowest, value))
    finally:
        d.close()


def test_dist_barrier_and_max_over_two_gloo_ranks():
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the slowest time; the job value counts both ranks' bytes
    assert [g[:3] for g in got] == [(0, 2, 2.5), (1, 2, 2.5)]
    assert all(abs(g[3] - 2 * 3.0e9 / 2.5 / 1e9) < 1e-9 for g in got)


def test_reference_arm_prints_once_under_torchrun():
    """Under torchrun the reference arm runs on rank 0 alone; the other rank
    exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["n_gpus"] == 2 and out["value"] > 0
    assert out["e2e"]["h2d_bytes_per_step"] == 0 and out["cpu_baseline"]["kind"] == "oracle"
