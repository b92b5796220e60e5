"""The N > 1 path of bench.py (independent replicas, one per GPU): the
timed region's time is the maximum over ranks and the job's throughput is
every rank's units over that time.  Run as two gloo ranks on the CPU."""
import os
import socket
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


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sys.path.insert(0, ROOT)
        import bench
        ms = [12.5, 20.0][rank]                       # rank 1 is the slow one
        ms_max = bench.max_over_ranks(torch, ms, world, device="cpu")
        out[rank] = (ms_max, bench.job_rate(1000.0, world, ms_max))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_is_max_and_rate_counts_all_ranks():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms_max, rate = res[rank]
        assert ms_max == 20.0
        assert rate == pytest.approx(2 * 1000.0 / 0.020)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(torch, 7.25, 1) == 7.25
    assert bench.job_rate(500.0, 1, 250.0) == pytest.approx(2000.0)


def test_reference_arm_prints_on_rank_zero_only(capsys):
    """Under torchrun the reference arm (the CPU oracle) runs on rank 0 only;
    every other rank returns at once without output."""
    sys.path.insert(0, ROOT)
    import types
    import bench
    bench.run_reference(types.SimpleNamespace(steps=1, warmup=3), world=2, rank=1)
    assert capsys.readouterr().out == ""
