"""kq_gemm_noalloc, the GEMM entry point that allocates nothing, against kq_gemm.

Some callers cannot allocate device memory or hand the library a workspace:
a serving runtime that plans its whole device-memory budget at start-up and
forbids allocation on the request path, a latency-critical path that cannot
take cudaMalloc's implicit synchronisation, or plain C host code that only
receives device pointers for its inputs and outputs.  kq_gemm_noalloc gives
them the prefill GEMM with its scratch in a fixed array of the library.

This file is collected last, so that a run stopping at the first failure has
already run every other test; it passes alone in a fresh process and after
the rest of the suite.
"""
import numpy as np
import pytest
import torch

from quantized_gemv_gemm_gb300 import synth

from gpu_util import assert_row_tol, kq, oracle_q8k, pack, q8k_to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    assert torch.cuda.is_available()
    return kq()


@pytest.mark.parametrize("fmt", [synth.Q4_K, synth.Q5_K, synth.Q6_K])
def test_noalloc_matches_kq_gemm_on_two_calls(K, fmt):
    """Two calls in a row through the C ABI, on different activations (the
    second call finds the first call's contents in the shared scratch), each
    equal to kq_gemm with an allocated workspace within the parity tolerance."""
    M, N, Kdim = 300, 250, 1280          # three token tiles, a ragged tail of rows
    rng = synth.rng_for(120, fmt)
    disk = synth.disk_weights(fmt, N, Kdim, rng)
    packed = pack(K, fmt, disk)
    for call in range(2):
        planes = oracle_q8k(synth.activations(M, Kdim, rng))
        a = q8k_to_dev(K, planes)
        y_ref = K.kq_gemm(fmt, packed, N, Kdim, a)
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        rc = K.raw().kq_gemm_noalloc(fmt, packed.data_ptr(), N, Kdim, K._q8k_struct(a), M, y.data_ptr(),
                                     K._stream())
        assert rc == 0, K.kq_strerror(rc)
        torch.cuda.synchronize()
        assert_row_tol(y.cpu().numpy(), y_ref.cpu().numpy().astype(np.float64))


def test_noalloc_rejects_problems_beyond_its_scratch(K):
    """A problem whose scratch would exceed the fixed array is refused with
    KQ_ERR_TOO_LARGE before anything is enqueued."""
    M, Kdim = 4096, 8192                 # 64 MiB of fp16 activation image
    assert K.kq_gemm_min_workspace_bytes(synth.Q4_K, M, 4096, Kdim) > K.KQ_NOALLOC_SCRATCH_BYTES
    q = K._Q8KConst(0x10000, 0x10000, 0x10000)   # never dereferenced: the size check comes first
    rc = K.raw().kq_gemm_noalloc(synth.Q4_K, 0x10000, 4096, Kdim, q, M, 0x10000, None)
    assert rc == -8
    assert "scratch" in K.kq_strerror(rc)


def test_noalloc_size_limit_boundary(K):
    """The documented largest shape (512 tokens x K = 30464) fits the fixed
    array and the next step of K (30720) is refused before anything runs."""
    fits = K.kq_gemm_min_workspace_bytes(synth.Q4_K, 512, 4096, 30464)
    over = K.kq_gemm_min_workspace_bytes(synth.Q4_K, 512, 4096, 30720)
    assert fits <= K.KQ_NOALLOC_SCRATCH_BYTES < over
    q = K._Q8KConst(0x10000, 0x10000, 0x10000)   # never dereferenced: the size check comes first
    rc = K.raw().kq_gemm_noalloc(synth.Q4_K, 0x10000, 4096, 30720, q, 512, 0x10000, None)
    assert rc == -8


@pytest.mark.parametrize("fmt", [synth.Q4_K, synth.Q6_K])
def test_noalloc_back_to_back_under_pdl(K, fmt):
    """Two calls enqueued on one stream with no synchronisation between them
    and programmatic dependent launch on: the second call's pre-pass rewrites
    the shared scratch while the first call's GEMM may still be running, so
    it must wait for it.  The second call has fewer tokens (301, not a
    multiple of 4), so a stale padded tail of the first call's scales would
    show.  Both outputs must equal kq_gemm's."""
    N, Kdim = 200, 1024
    rng = synth.rng_for(121, fmt)
    packed = pack(K, fmt, synth.disk_weights(fmt, N, Kdim, rng))
    cases = []
    for M in (512, 301):
        a = q8k_to_dev(K, oracle_q8k(synth.activations(M, Kdim, rng)))
        cases.append((M, a, torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")))
    refs = [K.kq_gemm(fmt, packed, N, Kdim, a) for _, a, _ in cases]
    torch.cuda.synchronize()
    old = K.kq_set_launch_flags(K.KQ_LAUNCH_PDL)
    try:
        for M, a, y in cases:
            rc = K.raw().kq_gemm_noalloc(fmt, packed.data_ptr(), N, Kdim, K._q8k_struct(a), M, y.data_ptr(),
                                         K._stream())
            assert rc == 0, K.kq_strerror(rc)
        torch.cuda.synchronize()
    finally:
        K.kq_set_launch_flags(old)
    for (_, _, y), y_ref in zip(cases, refs):
        assert_row_tol(y.cpu().numpy(), y_ref.cpu().numpy().astype(np.float64))
