"""bench.py's multi-rank host logic on the CPU: two gloo ranks (127.0.0.1),
each with its own timings; every rank must see the slowest rank's times, and
the job value counts all ranks' work over that time. Also: under a
multi-rank launch, only rank 0 runs and prints the reference arm."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = [1.0 + rank, 0.25 * (rank + 1), 0.5, 2.0 - rank]    # total, fwd, bwd, e2e (ms)
    got = bench.max_over_ranks(mine, dist, "cpu")
    dist.barrier()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(got, f)
    dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for rank in (0, 1):
        got = json.load(open(tmp_path / f"rank{rank}.json"))
        assert got == [2.0, 0.5, 0.5, 2.0], (rank, got)


def test_single_process_keeps_its_times():
    assert bench.max_over_ranks([3.0, 1.0], None, "cpu") == [3.0, 1.0]


def test_job_value_counts_every_rank():
    one = bench.job_tflops(7e12, 1, 1000.0)          # 7 TFLOP per step, 1 s per step
    assert one == pytest.approx(7.0)
    assert bench.job_tflops(7e12, 4, 1000.0) == pytest.approx(4 * one)   # weak scaling


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3", "--workload", "tiny_fp32"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
