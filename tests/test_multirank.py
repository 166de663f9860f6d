"""The bench's multi-rank path on the CPU (gloo, world size 2): the op has no
data-path collective (ranks are independent replicas), so what N > 1 adds is
the timing reduction (max over ranks), the weak-scaling rate and the
reference arm's rank handling."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [12.5, 14.25][rank]  # the second rank is the slower one
        m = bench.max_over_ranks(local_ms, dist, "cpu")
        rate = bench.whole_job_rate(world, 1.0e9, 3, m)
        out.put((rank, m, rate))
    finally:
        dist.destroy_process_group()


def test_timing_reduction_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, rate in res:
        assert m == 14.25  # every rank sees the slowest rank's time
        assert rate == pytest.approx(2 * 1.0e9 * 3 / 14.25e-3)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.0, None, "cpu") == 7.0
    assert bench.whole_job_rate(1, 10.0, 2, 1000.0) == pytest.approx(20.0)


def test_reference_arm_under_torchrun_prints_once():
    """`bench.py --impl reference` launched like the driver's N = 2 run: rank
    0 alone times the oracle and prints one JSON line; rank 1 exits 0."""
    env = dict(os.environ, SMQA_REF_TOKENS_PER_STEP="2", OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--seq", "192"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
