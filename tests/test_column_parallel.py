"""The column-parallel split (quantized_gemv_gemm_gb300.partition): slabs of
whole 16-row groups, and two gloo ranks that each compute their slab with
the oracle and all-gather it must reproduce the unsplit product bit for
bit (the rows of the product are independent)."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from quantized_gemv_gemm_gb300 import synth  # noqa: E402
from quantized_gemv_gemm_gb300.partition import column_slabs  # noqa: E402


@pytest.mark.parametrize("N,world", [(256, 2), (200, 2), (17408, 8), (5, 4), (0, 2), (4096, 3), (33, 1)])
def test_slabs_cover_rows_in_whole_groups(N, world):
    slabs = column_slabs(N, world)
    assert len(slabs) == world
    assert slabs[0][0] == 0 and slabs[-1][1] == N
    for (a0, a1), (b0, b1) in zip(slabs, slabs[1:]):
        assert a1 == b0
    sizes = [b - a for a, b in slabs]
    assert all(s >= 0 for s in sizes)
    assert all(a % 16 == 0 for a, _ in slabs if a < N)
    groups = [-(-s // 16) for s in sizes]
    assert max(groups) - min(groups) <= 1


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


CASES = [(synth.Q4_K, 200, 1024, 3), (synth.Q6_K, 300, 512, 2)]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sys.path.insert(0, ROOT)
        import oracle
        from quantized_gemv_gemm_gb300.partition import all_gather_rows
        res = []
        for fmt, N, K, M in CASES:
            disk = synth.disk_weights(fmt, N, K, synth.rng_for(130, fmt))
            q = oracle.quantize_q8k(synth.activations(M, K, synth.rng_for(131, fmt)))
            slabs = column_slabs(N, world)
            n0, n1 = slabs[rank]
            y_slab = torch.from_numpy(np.ascontiguousarray(oracle.gemm(fmt, disk[n0:n1], *q)))
            y = all_gather_rows(torch, y_slab, slabs, rank)
            res.append(y.numpy())
        out[rank] = res
    finally:
        dist.destroy_process_group()


def test_two_ranks_all_gather_equals_unsplit_product():
    import oracle
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for i, (fmt, N, K, M) in enumerate(CASES):
        disk = synth.disk_weights(fmt, N, K, synth.rng_for(130, fmt))
        q = oracle.quantize_q8k(synth.activations(M, K, synth.rng_for(131, fmt)))
        ref = oracle.gemm(fmt, disk, *q)
        for rank in range(world):
            assert res[rank][i].shape == (M, N)
            np.testing.assert_array_equal(res[rank][i], ref)
