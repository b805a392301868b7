"""The benchmark's N > 1 path on CPU: world_size-2 gloo ranks.

Each rank is an independent replica; the job time is the slowest rank's
timed region and the throughput counts every rank's steps.  The reference
(oracle) arm runs on rank 0 only.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local = 10.0 + 5.0 * rank                     # rank 1 is the slow replica
    job = bench.job_time_ms(local, dist)
    out[rank] = (job, bench.job_tflops(1e12, 4, world, job))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_job_time_is_the_max_and_throughput_counts_all_ranks():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        job, tf = res[rank]
        assert job == 15.0
        assert abs(tf - 1e12 * 4 * 2 / 15e-3 / 1e12) < 1e-9


def test_single_rank_job_time_is_local():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.job_time_ms(3.5) == 3.5


@pytest.mark.parametrize("rank", ["1"])
def test_reference_arm_non_zero_rank_exits_without_work(rank):
    env = dict(os.environ, RANK=rank, WORLD_SIZE="2", LOCAL_RANK=rank)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "1"], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def _env_without_ranks():
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "LOCAL_WORLD_SIZE", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(k, None)
    return env


def test_gpus_flag_launches_that_many_ranks():
    """`bench.py --gpus 2` outside torch.distributed.run starts two ranks; the
    reference arm's line (rank 0 only) then reports n_gpus = 2."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "1", "--workload", "b1_h1_n128_d64",
                        "--reference-step-s", "0.3"], env=_env_without_ranks(), capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    import json

    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2


@pytest.mark.parametrize("gpus_args", [["--gpus", "4"], []])
def test_gpus_flag_must_match_the_world_size(gpus_args):
    """Under torch.distributed.run (WORLD_SIZE set) a --gpus that differs from
    the world size is an error, not a silently relabelled run."""
    env = dict(_env_without_ranks(), RANK="0", WORLD_SIZE="2", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "1", "--workload", "b1_h1_n128_d64"] + gpus_args,
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0
    assert r.stdout.strip() == ""
    assert "WORLD_SIZE=2" in r.stderr
