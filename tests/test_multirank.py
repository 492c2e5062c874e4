"""Host-side logic of the multi-process bench path on CPU: two ranks over the
gloo backend (no GPU).  The layer forward is data-parallel over tokens, so
N GPUs run N independent replicas with no collective on the data path; the
only cross-rank steps are the barrier around the timed region and taking the
slowest rank's time."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dist.barrier()
    out[rank] = bench.max_over_ranks(times[rank], "cpu")
    dist.barrier()
    dist.destroy_process_group()


def test_slowest_rank_time_over_gloo():
    world = 2
    times = [3.25, 7.5]
    out = mp.get_context("spawn").Manager().list([0.0] * world)
    mp.spawn(_rank_main, args=(world, _free_port(), times, out), nprocs=world, join=True)
    assert list(out) == [7.5, 7.5]


def test_single_process_passes_time_through():
    assert bench.max_over_ranks(4.0, "cpu") == 4.0


def test_job_throughput_counts_every_replica():
    # 2 replicas x 10 steps x 8 tokens in 5 ms (slowest rank) = 32,000 tokens/s
    assert bench.job_tokens_per_s(2, 10, 8, 5.0) == pytest.approx(32000.0)
    assert bench.job_tokens_per_s(1, 10, 8, 5.0) == pytest.approx(16000.0)


def test_reference_arm_prints_nothing_on_other_ranks():
    """Under torchrun only rank 0 runs and prints the reference arm."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
