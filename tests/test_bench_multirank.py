"""bench.py's host logic for N > 1 ranks, on CPU with the gloo backend: the
max-over-ranks timing, the barrier, the whole-job aggregate, and the
reference arm under torchrun (rank 0 alone works and prints one line)."""
import json
import multiprocessing as mp
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, local = bench.dist_setup()
    # each rank reports a different "timed total"; every rank must see the max
    got = bench.max_over_ranks(10.0 * (rank + 1), w)
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()
    out.put((r, w, local, got))


def test_max_over_ranks_and_barrier_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[:3] for r in res] == [(0, 2, 0), (1, 2, 1)]
    assert all(r[3] == 20.0 for r in res)  # the slower rank's time, on both


def test_job_value_counts_every_rank_in_the_slowest_time():
    sys.path.insert(0, ROOT)
    import bench
    flops = 2.0 * 4096 ** 3
    one = bench.job_value(1, flops, 100, 10.0)
    assert one == pytest.approx(flops * 100 / 10e-3 / 1e12)
    # weak scaling: two replicas in the same slowest time double the total
    assert bench.job_value(2, flops, 100, 10.0) == pytest.approx(2 * one)
    assert bench.job_value(2, flops, 100, 20.0) == pytest.approx(one)


def test_reference_arm_under_torchrun_world2():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="4")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout  # rank 0 alone prints
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 1
    assert line["value"] > 0 and line["unit"] == "TFLOP/s"
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
