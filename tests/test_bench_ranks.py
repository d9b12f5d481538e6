"""bench.py's multi-replica host logic on CPU: two gloo ranks, no GPU.

The path has no exchange step, so N GPUs run N independent replicas; what the
ranks share is the timing: every rank's step time is reduced with MAX (the
job is as slow as its slowest replica), the whole-job rate counts all
replicas' work, and only rank 0 prints. The reference arm runs on rank 0
alone; the other ranks exit without work.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, step_ms, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench

    dist, r, w = bench._dist("gloo")
    ms = bench.max_over_ranks(step_ms[rank], dist, "cpu")
    out.put((r, w, ms, bench.whole_job_rate(w, 1000.0, ms)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_replica_and_the_whole_job_rate():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    step_ms = [3.0, 5.0]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, step_ms, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the slowest replica's 5 ms; 2 replicas x 1000 units / 5 ms
    assert got == [(0, 2, 5.0, 2 * 1000.0 / 5e-3), (1, 2, 5.0, 2 * 1000.0 / 5e-3)]


def test_one_replica_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(7.5, None) == 7.5
    assert bench.whole_job_rate(1, 300.0, 2.0) == 300.0 / 2e-3


def test_reference_arm_on_a_non_zero_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
