"""bench.py's multi-rank bookkeeping (replicas: barrier, max over ranks,
whole-job GB/s) on two gloo ranks on the CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(10.0 + 5.0 * rank)
    out[rank] = (ms, bench.whole_job_gbs(world, 1 << 30, 4, ms))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    ctx = mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    del ctx
    assert out[0][0] == out[1][0] == 15.0
    # two replicas moving 4 GiB each in 15 ms
    assert abs(out[0][1] - 2 * 4 * (1 << 30) / 15e-3 / 1e9) < 1e-6


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_gbs(1, 10 ** 9, 1, 1000.0) == 1.0


def test_reference_arm_runs_on_rank_zero_only():
    # under torchrun the oracle's arm runs on rank 0 alone; the other ranks
    # exit 0 without work or output
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
