"""The benchmark's multi-rank host logic on CPU: two gloo ranks on
127.0.0.1, no GPU. Each rank is an independent replica (the path shards
over requests and heads with no exchange); the whole job's time is the
slowest rank's and its value counts every rank's units. The reference arm
prints from rank 0 only."""

import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    times = [3.0, 7.5]                       # rank 1 is the slow one
    slowest = bench.max_over_ranks(times[rank], "cpu")
    value = bench.whole_job_rate(1e9, world, slowest, "GB/s")
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"slowest": slowest, "value": value}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time(tmp_path):
    port = 29500 + os.getpid() % 1000
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn")
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    assert got[0] == got[1]
    assert got[0]["slowest"] == 7.5
    # two replicas of 1e9 bytes each in 7.5 s
    assert abs(got[0]["value"] - 2e9 / 7.5 / 1e9) < 1e-12


def test_single_process_max_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.25, "cpu") == 4.25


def test_reference_arm_prints_from_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "fwd_f32_single_head", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
