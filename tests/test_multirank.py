"""The benchmark's multi-rank host logic on CPU: two gloo ranks (no GPU), the replicated run's slowest-rank step time
and whole-job throughput, and the reference arm's rank-0-only line."""
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


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.reduce_max(10.0 + 5.0 * rank, world, "cpu")  # rank 1 is the slow one
        value = bench.job_throughput(2.0e9, ms, world)
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{ms} {value}\n")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_step(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    got = [tuple(map(float, (tmp_path / f"rank{r}.txt").read_text().split())) for r in range(2)]
    assert got[0] == got[1] == (15.0, 2 * 2.0e9 / 15e-3 / 1e9)


def test_single_rank_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.5, 1, "cpu") == 3.5
    assert bench.job_throughput(1.0e9, 1.0, 1) == 1000.0


def test_reference_arm_prints_on_rank_zero_only():
    """Under torchrun every rank but 0 exits without work or output."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3"], capture_output=True, text=True, env=env, timeout=120)
    assert out.returncode == 0 and out.stdout.strip() == ""
