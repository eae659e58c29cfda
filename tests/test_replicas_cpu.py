"""The multi-GPU path is replicas only: sequences are independent, so each
rank runs its own draft steps and only the step time is reduced (the slowest
rank decides the job's time).  These tests run that host logic as two gloo
ranks on the CPU."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from block_diffusion_draft_gb300 import workloads as W  # noqa: E402


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, lr = bench.rank_env()
    ms = 1.0 + 0.5 * r  # rank 1 is slower
    slowest = bench.max_over_ranks(ms, dist, torch.device("cpu"))
    seed = bench.replica_seed(7, r, w)
    sched = W.serving_schedule(W.SPECS["serving_b32"], seed, steps=2)
    value = bench.job_value(w, 32, slowest)
    dist.barrier()
    out.put((r, w, lr, slowest, seed, list(sched.prefill), value))
    dist.destroy_process_group()


def test_two_gloo_replicas_reduce_the_slowest_time():
    world, port = 2, free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, w0, l0, s0, seed0, pre0, v0), (r1, w1, l1, s1, seed1, pre1, v1) = res
    assert (r0, r1) == (0, 1) and w0 == w1 == 2 and (l0, l1) == (0, 1)
    # both ranks see the slowest rank's time; the job value counts both
    # ranks' blocks over that time
    assert s0 == s1 == 1.5
    assert v0 == v1 == pytest.approx(2 * 32 / 1.5e-3)
    # each replica draws its own sequences
    assert seed0 != seed1 and pre0 != pre1


def test_single_process_defaults():
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    old = os.environ.copy()
    try:
        os.environ.clear()
        os.environ.update(env)
        assert bench.rank_env() == (1, 0, 0)
    finally:
        os.environ.clear()
        os.environ.update(old)
    assert bench.replica_seed(7, 0, 1) == 7
    assert bench.max_over_ranks(2.5, None, None) == 2.5


def test_reference_arm_runs_on_rank_zero_only():
    # a non-zero rank of the reference arm exits 0 without work or output
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "1"],
                       env=env, capture_output=True, text=True, timeout=120, cwd=ROOT)
    assert r.returncode == 0 and r.stdout.strip() == ""
