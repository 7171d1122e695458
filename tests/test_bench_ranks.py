"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): the timings every rank
reports are the maximum over ranks, the whole-job value scales with the rank count, and only
rank 0 runs the reference arm."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        names = ["gemm_q8_0", "gemv_q8_0"]
        # rank 1 is slower on the GEMV, rank 0 on the GEMM
        mean = {"gemm_q8_0": 0.060 if rank == 0 else 0.050, "gemv_q8_0": 0.050 + 0.010 * rank}
        step = sum(mean.values()) + 0.001 * rank
        step_max, mean_max = bench.max_over_ranks(step, mean, names, torch.device("cpu"))
        out[rank] = (step_max, mean_max["gemm_q8_0"], mean_max["gemv_q8_0"])
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    step_max, gemm_max, gemv_max = res[0]
    assert gemm_max == pytest.approx(0.060)
    assert gemv_max == pytest.approx(0.060)
    assert step_max == pytest.approx(0.050 + 0.060 + 0.001)


def test_whole_job_value_is_weak_scaling():
    assert bench.whole_job_value(5000.0, 1) == 5000.0
    assert bench.whole_job_value(5000.0, 8) == 40000.0


def test_reference_arm_runs_on_rank_zero_only():
    class A:
        steps, warmup = 1, 0
    assert bench.run_reference(A, rank=1, world=2) is None
