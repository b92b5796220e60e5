"""Parity of the Q8_0 GEMM (kq_gemm_q8_0) with the oracle: the Q8_0 weights x
Q8_0-form activations product for M token rows ([kq-arc], MoE prefill fix:
the Q8_0 GEMMs read the Q8_0-form batch image), one float fold per 32-block
after an exact int32 dot."""
import numpy as np
import pytest
import torch

import oracle
from quantized_gemv_gemm_gb300 import synth

from gpu_util import assert_row_tol, check_guard, kq, poisoned, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    assert torch.cuda.is_available()
    return kq()


def run(K, disk, d_a, q_a):
    N, nb, _ = disk.shape
    Kdim, M = nb * 32, q_a.shape[0]
    packed = K.kq_repack(synth.Q8_0, to_dev(disk.reshape(-1)), N, Kdim)
    full, y = poisoned((M, N))
    K.kq_gemm_q8_0(packed, N, Kdim, to_dev(d_a), to_dev(q_a), y=y)
    torch.cuda.synchronize()
    check_guard(full, M * N)
    return y.cpu().numpy()


@pytest.mark.parametrize("M,N,Kdim", [(16, 300, 1024), (100, 200, 2560), (512, 130, 768), (1, 64, 256),
                                      (65, 17, 512), (7, 128, 5120)])
def test_q8_0_gemm_matches_oracle(K, M, N, Kdim):
    """Every output of ragged token tiles (M not a multiple of 64) and weight
    tiles (N not a multiple of 16 or 128) against the oracle."""
    rng = synth.rng_for(150, M * 7 + N + Kdim)
    disk = synth.disk_weights_q8_0(N, Kdim, rng)
    d_a, q_a = oracle.quantize_q8_0(synth.activations(M, Kdim, rng, outliers=True))
    y = run(K, disk, d_a, q_a)
    assert_row_tol(y, oracle.gemm_q8_0(disk, d_a, q_a))


def test_q8_0_gemm_exact_at_extremes(K):
    """Scales of 1 and quants at +-127 (and -128 in the activations, which the
    quantizer never writes but the call accepts): every output is an exact
    integer below 2^24, so it must equal the oracle exactly."""
    rng = synth.rng_for(151, 0)
    M, N, Kdim = 70, 40, 512
    disk = np.zeros((N, Kdim // 32, 34), np.uint8)
    disk[:, :, 0:2] = [0x00, 0x3C]                                   # d = 1
    qw = rng.choice(np.array([-127, 127, -1, 0, 1], np.int8), size=(N, Kdim // 32, 32))
    qw[0] = 127
    disk[:, :, 2:] = qw.view(np.uint8)
    q_a = rng.choice(np.array([-128, -127, 127, 5], np.int8), size=(M, Kdim))
    q_a[0] = 127
    d_a = np.ones((M, Kdim // 32), np.float32)
    y = run(K, disk, d_a, q_a)
    ref = oracle.gemm_q8_0(disk, d_a, q_a)
    assert np.abs(ref).max() < 2 ** 24
    np.testing.assert_array_equal(y.astype(np.float64), ref)
    # and the per-block integer dots behind it
    P = oracle.partials_q8_0(disk, q_a)
    np.testing.assert_array_equal(P.sum(axis=2).astype(np.float64), ref)


def test_q8_0_gemm_row_equals_gemv(K):
    """A token row of the GEMM equals the Q8_0 GEMV of that row within the
    tolerance (both fold per block; the summation orders differ)."""
    rng = synth.rng_for(152, 0)
    M, N, Kdim = 20, 256, 2560
    disk = synth.disk_weights_q8_0(N, Kdim, rng)
    d_a, q_a = oracle.quantize_q8_0(synth.activations(M, Kdim, rng))
    y = run(K, disk, d_a, q_a)
    packed = K.kq_repack(synth.Q8_0, to_dev(disk.reshape(-1)), N, Kdim)
    for m in (0, 7, 19):
        yv = K.kq_gemv_q8_0(packed, N, Kdim, to_dev(d_a[m]), to_dev(q_a[m]))
        torch.cuda.synchronize()
        assert_row_tol(y[m][None, :], yv.cpu().numpy()[None, :].astype(np.float64))
