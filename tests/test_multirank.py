"""Replicas on several ranks (bench.py under torchrun): two gloo ranks on the
CPU check how the benchmark combines its ranks -- the slowest rank's time,
the whole-job rate over all ranks' units -- and that the reference arm runs
on rank 0 only.  No GPU is involved."""
import multiprocessing as mp
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    w, r, local = bench.init_ranks("gloo")
    t_local = 1.0 + 0.5 * r                      # rank r took 1 + r/2 seconds
    t_max = bench.max_over_ranks(t_local, "cpu")
    rate = bench.whole_job_rate(10.0, w, t_max)  # 10 units per rank
    dist.barrier()
    dist.destroy_process_group()
    out.put((r, w, local, t_max, rate))


@pytest.mark.parametrize("world", [2])
def test_replica_timing_takes_the_slowest_rank(world):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    slowest = 1.0 + 0.5 * (world - 1)
    for r, (rank, w, local, t_max, rate) in enumerate(got):
        assert (rank, w, local) == (r, world, r)
        assert t_max == slowest
        assert rate == pytest.approx(10.0 * world / slowest)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    env = {k: os.environ.pop(k) for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK") if k in os.environ}
    try:
        assert bench.init_ranks("gloo") == (1, 0, 0)
        assert not dist.is_initialized()
        assert bench.max_over_ranks(2.5, "cpu") == 2.5
        assert bench.whole_job_rate(6.0, 1, 2.0) == 3.0
    finally:
        os.environ.update(env)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
