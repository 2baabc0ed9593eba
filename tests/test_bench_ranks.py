"""The benchmark's multi-process host logic on CPU (gloo, two ranks): the
step time is the maximum over ranks, the job's throughput counts every
rank's replica, and the reference arm runs on rank 0 only.  No GPU."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, values, out):
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    try:
        ms_max = bench.max_over_ranks(values[rank], "cpu", world)
        out[rank] = (ms_max, bench.job_tflops(world, 2.0e12, ms_max))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp

    values = [12.5, 20.0]
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(2, _free_port(), values, out), nprocs=2, join=True)
        res = dict(out)
    for rank in range(2):
        ms_max, tflops = res[rank]
        assert ms_max == 20.0  # every rank sees the slowest rank's time
        assert tflops == pytest.approx(2 * 2.0e12 / 20.0e-3 / 1e12)  # 200 TFLOP/s for the two replicas


def test_single_process_is_identity():
    import bench

    assert bench.max_over_ranks(7.25, "cpu", 1) == 7.25
    assert bench.job_tflops(1, 1.0e12, 10.0) == pytest.approx(100.0)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
