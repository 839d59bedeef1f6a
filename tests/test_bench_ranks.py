"""Multi-rank plumbing of bench.py on the CPU: two gloo ranks agree on the slowest rank's time and on the
whole-job rate, and the reference arm prints nothing on ranks other than 0."""
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 10.0 + 5.0 * rank          # rank 1 is slower
    slowest = bench.max_over_ranks(local_ms, dist)
    rate = bench.whole_job_rate(1000.0, 4, world, slowest)
    out[rank] = torch.tensor([slowest, rate], dtype=torch.float64)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    world = 2
    out = torch.zeros(world, 2, dtype=torch.float64).share_memory_()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        assert out[r, 0].item() == 15.0
        assert abs(out[r, 1].item() - 1000.0 * 4 * world / 15e-3) < 1e-6


def test_single_process_aggregation_is_identity():
    import bench

    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.whole_job_rate(10.0, 2, 1, 4.0) == 10.0 * 2 / 4e-3


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
