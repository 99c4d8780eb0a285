"""The benchmark's multi-rank logic on CPU: two `gloo` ranks (world size 2) on 127.0.0.1.

Every rank runs its own replica (weak scaling); the job's time is the maximum over ranks and the
whole-job value counts the work of every rank. Under the reference arm only rank 0 works and prints.
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


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        local = [10.0 + 5.0 * rank, 3.0 - rank]  # rank 1 slower in the first figure, faster in the second
        got = bench.max_over_ranks(local, dist, "cpu")
        value = bench.whole_job_tflops(2.0e12, 4, world, got[0])
        q.put((rank, got, value))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, got, value in res:
        assert got == [15.0, 3.0]  # the maximum of every figure over both ranks
        # 2 ranks x 4 steps x 2 TFLOP in 15 ms
        assert value == pytest.approx(2 * 4 * 2.0 / 15e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert bench.whole_job_tflops(1e12, 10, 1, 1000.0) == pytest.approx(10.0)


def test_reference_arm_non_zero_rank_exits_without_output():
    """Under torchrun the reference arm runs on rank 0 only; another rank exits 0 and prints nothing."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
