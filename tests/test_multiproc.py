"""The multi-GPU path is replicas only (every operator is independent per row /
token, there is no exchange step): each rank runs its own copy of the step and
the ranks meet only to time it. These CPU tests run that host logic on two
gloo ranks: the max-over-ranks step time, the whole-job weak-scaling value and
the reference arm's rank-0-only rule."""
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [0.5, 0.8][rank]
        ms = bench.reduce_max(local_ms, torch.device("cpu"))
        value = bench.weak_value(1_000_000_000, ms, world)
        dist.barrier()
        q.put((rank, ms, value))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, value in got:
        assert ms == 0.8                                   # the slowest rank's time, on every rank
        assert value == pytest.approx(2 * 1e9 / 0.8e-3 / 1e9)  # both ranks' bytes over that time


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.reduce_max(1.25, "cpu") == 1.25
    assert bench.weak_value(2_000_000, 1.0, 1) == pytest.approx(2.0)


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
