"""The benchmark's multi-GPU mode is replicas only: every rank runs the whole
path on its own inputs, with a barrier around the timed region and the
maximum time over ranks.  These CPU tests run its rank plumbing as two gloo
processes (no GPU, no data-path collective)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    g = bench.Group(w, r, local, use_cuda=False)
    try:
        g.barrier()
        out[rank] = (g.max(1.5 + rank), g.max(10.0 - rank))
        g.barrier()
    finally:
        g.close()


def test_two_gloo_ranks_barrier_and_max():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    assert dict(out) == {0: (2.5, 10.0), 1: (2.5, 10.0)}


def test_job_throughput_is_sum_over_ranks_at_the_slowest_time():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.job_tops(1, 4.0e12, 10, 20.0)          # 40e12 ops in 20 ms
    assert one == pytest.approx(2000.0)
    assert bench.job_tops(4, 4.0e12, 10, 20.0) == pytest.approx(4 * one)
    assert bench.job_tops(2, 4.0e12, 10, 40.0) == pytest.approx(one)   # slower rank halves it


def test_single_process_group_is_a_no_op():
    sys.path.insert(0, ROOT)
    import bench
    g = bench.Group(1, 0, 0, use_cuda=False)
    g.barrier()
    assert g.max(3.25) == 3.25
    g.close()


def test_bench_gpus_2_starts_two_ranks_itself():
    """`bench.py --gpus 2`, run directly (no torchrun), starts its own two
    rank processes; in the CPU self-test mode they meet over gloo and rank 0
    prints n_gpus = 2 and the maximum over the ranks' times."""
    import json
    import subprocess
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--launcher-selftest"],
                         capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    rec = json.loads(lines[0])
    assert rec["n_gpus"] == 2 and rec["ms_max"] == 11.0
