"""Host logic of the multi-GPU bench path on CPU (gloo, world size 2).

The forward shards by sequence with no exchange step, so ``bench.py --gpus N``
runs N independent replicas; the only cross-rank steps are the max of the step
time over the ranks and rank 0 alone printing (and, for the reference arm,
alone running the oracle).  These run here with the gloo backend.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank's step time differs; every rank must see the slowest
        ms = bench.max_over_ranks(1.5 + rank, world)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"ms": ms}, f)
    finally:
        dist.destroy_process_group()


def test_step_time_is_the_max_over_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    got = [json.load(open(tmp_path / f"rank{r}.json"))["ms"] for r in range(world)]
    assert got == [2.5, 2.5]


def test_single_rank_is_unchanged():
    assert bench.max_over_ranks(0.1746, 1) == 0.1746


def test_whole_job_value_counts_every_replica():
    # 2 replicas of 128 block tokens in 0.2 ms each: 1.28 M tokens/s for the job
    assert bench.job_tokens_per_s(128, 2, 0.2e-3) == pytest.approx(1.28e6)
    assert bench.job_tokens_per_s(128, 1, 0.2e-3) == pytest.approx(0.64e6)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
