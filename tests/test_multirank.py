"""The N > 1 host logic of bench.py on CPU: two gloo ranks (127.0.0.1).

Every rank runs an independent replica (no data-path collective); the job's
time is the slowest rank's and the throughput counts every rank's tokens.
The reference arm runs on rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        ms = [0.75, 1.25][rank]             # the second rank is slower
        job_ms = bench.max_over_ranks(ms, dist, torch.device("cpu"))
        q.put((rank, job_ms, bench.job_tokens_per_s(world, 32, job_ms)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_takes_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, job_ms, value in got:
        assert job_ms == 1.25
        assert value == pytest.approx(2 * 32 / 1.25e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.5, None, torch.device("cpu")) == 0.5
    assert bench.job_tokens_per_s(1, 32, 1.0) == pytest.approx(32000.0)


def test_reference_arm_is_rank_zero_only():
    """Ranks other than 0 exit 0 without work or output (torchrun launch of
    the reference arm)."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
