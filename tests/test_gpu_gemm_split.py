"""The tensor-core GEMM's split-tile schedule (KQ_LAUNCH_GEMM_SPLIT forces it).

One block per SM takes an even share of the tiles x superblocks steps; a tile
cut between blocks is finished by the last of them, which adds the blocks'
fp32 partial tiles in block order.  At the small shapes here every block gets
a step or a few, so each tile is cut between many blocks: the integer sums
must still equal the oracle's bit for bit ([kq-arc], kq v3 panel-scratch
commit, the tile-vs-GEMV bit-exactness gate), the outputs must stay within
the oracle's tolerance, and a repeated call must give the same bits (the
partial tiles are added in a fixed order).
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_gemv_gemm_gb300 import synth

from gpu_util import assert_row_tol, kq, oracle_q8k, pack, q8k_to_dev
from test_gpu_gemm_partials import check_against_oracle_and_gemv, extreme_tokens, extreme_weights

pytestmark = pytest.mark.gpu
FMTS = [synth.Q4_K, synth.Q5_K, synth.Q6_K]
SHAPES = [(200, 1280, 300), (128, 2560, 16), (33, 512, 129), (384, 3072, 160)]


@pytest.fixture(scope="module")
def K():
    assert torch.cuda.is_available()
    return kq()


@pytest.fixture
def split(K):
    old = K.kq_set_launch_flags(K.kq_get_launch_flags() | K.KQ_LAUNCH_GEMM_SPLIT)
    yield
    K.kq_set_launch_flags(old)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("N,Kdim,M", SHAPES[:3])
def test_split_partials_bit_exact(K, split, fmt, N, Kdim, M):
    rng = synth.rng_for(150, fmt * 1000 + N)
    disk = synth.disk_weights(fmt, N, Kdim, rng)
    planes = oracle_q8k(synth.activations(M, Kdim, rng))
    got_i, got_m = K.kq_debug_gemm_partials(fmt, pack(K, fmt, disk), N, Kdim, q8k_to_dev(K, planes))
    torch.cuda.synchronize()
    check_against_oracle_and_gemv(K, fmt, disk, planes, got_i.cpu().numpy(), got_m.cpu().numpy())


@pytest.mark.parametrize("fmt", FMTS)
def test_split_partials_worst_case_fields(K, split, fmt):
    """Every field at its extreme (sums past 2^24, the most accumulator units
    per superblock) with the superblocks of each tile spread over blocks."""
    rng = synth.rng_for(151, fmt)
    N, Kdim, M = 512 if fmt == synth.Q6_K else 160, 768, 40
    disk = extreme_weights(fmt, N, Kdim, rng)
    planes = extreme_tokens(M, Kdim, rng)
    got_i, got_m = K.kq_debug_gemm_partials(fmt, pack(K, fmt, disk), N, Kdim, q8k_to_dev(K, planes))
    torch.cuda.synchronize()
    ref_i = check_against_oracle_and_gemv(K, fmt, disk, planes, got_i.cpu().numpy(), got_m.cpu().numpy())
    assert np.abs(ref_i).max() > 2 ** 24


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("N,Kdim,M", SHAPES)
def test_split_outputs_within_tolerance(K, split, fmt, N, Kdim, M):
    rng = synth.rng_for(152, fmt * 1000 + N)
    disk = synth.disk_weights(fmt, N, Kdim, rng)
    planes = oracle_q8k(synth.activations(M, Kdim, rng))
    y = K.kq_gemm(fmt, pack(K, fmt, disk), N, Kdim, q8k_to_dev(K, planes))
    torch.cuda.synchronize()
    assert_row_tol(y.cpu().numpy(), oracle.gemm(fmt, disk, *planes))


@pytest.mark.parametrize("fmt", FMTS)
def test_split_repeatable_and_close_to_tile_schedule(K, fmt):
    """Two calls give the same bits; the one-block-per-tile schedule (the
    smallest workspace) agrees within float rounding."""
    N, Kdim, M = 384, 3072, 160
    rng = synth.rng_for(153, fmt)
    disk = synth.disk_weights(fmt, N, Kdim, rng)
    packed = pack(K, fmt, disk)
    a = q8k_to_dev(K, oracle_q8k(synth.activations(M, Kdim, rng)))
    old = K.kq_set_launch_flags(K.kq_get_launch_flags() | K.KQ_LAUNCH_GEMM_SPLIT)
    try:
        y1 = K.kq_gemm(fmt, packed, N, Kdim, a)
        y2 = K.kq_gemm(fmt, packed, N, Kdim, a)
        ws_min = torch.empty(K.kq_gemm_min_workspace_bytes(fmt, M, N, Kdim), dtype=torch.uint8, device="cuda")
        y_tile = K.kq_gemm(fmt, packed, N, Kdim, a, workspace=ws_min)
    finally:
        K.kq_set_launch_flags(old)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    assert_row_tol(y1.cpu().numpy(), y_tile.cpu().numpy().astype(np.float64))
