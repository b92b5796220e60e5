"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bit-exact: Q8_K quantization (d8, q8, bsums), the repacked image's decode,
and the int32 partials of the fold.  Floating point: every output within
1e-3 x max|row output| of the oracle's fp64 value, per token row.
Full-size workloads are checked on sampled outputs computed one by one by
the oracle, in the launch configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_gemv_gemm_gb300 import synth

from gpu_util import (assert_row_tol, check_guard, kq, oracle_q8k, pack, poisoned, q8k_to_dev, to_dev)

pytestmark = pytest.mark.gpu
FMTS = [synth.Q4_K, synth.Q5_K, synth.Q6_K]


@pytest.fixture(scope="module")
def K():
    assert torch.cuda.is_available()
    return kq()


# ---------------------------------------------------------------- Q8_K
@pytest.mark.parametrize("M,Kdim,outliers", [(1, 1024, False), (3, 2560, False), (512, 5120, True),
                                             (4096, 2048, False), (7, 256, False)])
def test_quantize_bit_exact(K, M, Kdim, outliers):
    rng = synth.rng_for(100, M * 7 + Kdim)
    x = synth.activations(M, Kdim, rng, outliers=outliers)
    if M >= 3:
        x[0, :256] = 0.0                           # zero block
        x[1, 256 * (Kdim // 512):] *= np.float32(1e-30)
        x[2, 5] = np.float32(3e4)
        x[2, :256] = np.float32(2.5)               # ties: x*iscale lands on .5
        x[2, 0] = np.float32(127.0)
    ref = oracle_q8k(x)
    got = K.kq_quantize_q8k(to_dev(x))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got.d.cpu().numpy(), ref[0])
    np.testing.assert_array_equal(got.qs.cpu().numpy(), ref[1])
    np.testing.assert_array_equal(got.bsums.cpu().numpy(), ref[2])


# ---------------------------------------------------------------- repack
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("N,Kdim", [(1, 256), (200, 768), (37, 2560)])
def test_repack_round_trip(K, fmt, N, Kdim):
    disk = synth.disk_weights(fmt, N, Kdim, synth.rng_for(101, fmt * 1000 + N))
    packed = pack(K, fmt, disk)
    dec = K.kq_debug_decode(fmt, packed, N, Kdim)
    torch.cuda.synchronize()
    nsb = Kdim // 256
    nsub = 16 if fmt == synth.Q6_K else 8
    q = dec["q"].cpu().numpy().reshape(N, nsb, 256)
    sc = dec["sc"].cpu().numpy()
    mn = dec["m"].cpu().numpy()
    d = dec["d"].cpu().numpy()
    dmin = dec["dmin"].cpu().numpy()
    for n in range(N):
        for s in range(nsb):
            ref = oracle.decode(fmt, disk[n, s])
            np.testing.assert_array_equal(q[n, s], ref["q"])
            np.testing.assert_array_equal(sc[n, s, :nsub], ref["sc"])
            np.testing.assert_array_equal(mn[n, s], ref["m"])
            assert d[n, s] == np.float32(ref["d"]) and dmin[n, s] == np.float32(ref["dmin"])


# ---------------------------------------------------------------- partials
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("N,Kdim,M", [(1, 256, 1), (8, 768, 3), (200, 2560, 2)])
def test_partials_bit_exact(K, fmt, N, Kdim, M):
    rng = synth.rng_for(102, fmt * 100 + N)
    disk = synth.disk_weights(fmt, N, Kdim, rng)
    x = synth.activations(M, Kdim, rng)
    planes = oracle_q8k(x)
    ref_i, ref_m = oracle.partials(fmt, disk, planes[1], planes[2])
    got_i, got_m = K.kq_debug_partials(fmt, pack(K, fmt, disk), N, Kdim, q8k_to_dev(K, planes))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got_i.cpu().numpy(), ref_i)
    np.testing.assert_array_equal(got_m.cpu().numpy(), ref_m)


@pytest.mark.parametrize("fmt", FMTS)
def test_partials_worst_case_fields(K, fmt):
    """Every stored field at its extreme (q max, sub-scales max / -128, q8 = -127):
    the int32 partials still match exactly (the page's |iacc| < 2^28 bound)."""
    blk = np.full((2, 1, synth.BLOCK_BYTES[fmt]), 255, np.uint8)
    if fmt == synth.Q6_K:
        blk[0, 0, 192:208] = np.array([-128] * 16, np.int8).view(np.uint8)
        blk[1, 0, 192:208] = np.array([127] * 16, np.int8).view(np.uint8)
        blk[:, 0, 208:210] = [0x00, 0x3C]
    else:
        blk[:, 0, 0:4] = [0x00, 0x3C, 0x00, 0x3C]
    planes = (np.ones((2, 1), np.float32), np.array([[-127] * 256, [127] * 256], np.int8),
              np.array([[-127 * 16] * 16, [127 * 16] * 16], np.int16))
    ref_i, ref_m = oracle.partials(fmt, blk, planes[1], planes[2])
    got_i, got_m = K.kq_debug_partials(fmt, pack(K, fmt, blk), 2, 256, q8k_to_dev(K, planes))
    np.testing.assert_array_equal(got_i.cpu().numpy(), ref_i)
    np.testing.assert_array_equal(got_m.cpu().numpy(), ref_m)


# ---------------------------------------------------------------- GEMV
def run_gemv(K, fmt, disk, x):
    N, nsb, _ = disk.shape
    Kdim = nsb * 256
    planes = oracle_q8k(x)
    full, y = poisoned((N,))
    K.kq_gemv(fmt, pack(K, fmt, disk), N, Kdim, q8k_to_dev(K, planes), y=y)
    torch.cuda.synchronize()
    check_guard(full, N)
    return y.cpu().numpy(), planes


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("N,Kdim", [(1, 256), (8, 1024), (200, 768), (1000, 2560), (77, 4096)])
def test_gemv_small_shapes(K, fmt, N, Kdim):
    rng = synth.rng_for(103, fmt * 10000 + N)
    disk = synth.disk_weights(fmt, N, Kdim, rng)
    x = synth.activations(1, Kdim, rng)
    y, planes = run_gemv(K, fmt, disk, x)
    ref = oracle.gemm(fmt, disk, *planes)[0]
    assert_row_tol(y, ref)


def test_gemv_tiny_config(K):
    """The tiny Q4_K GEMV workload: N=256, K=1024, seed 0."""
    cfg = synth.configs()[0]
    m = cfg.matrices[0]
    disk = synth.disk_weights(m.fmt, m.N, m.K, synth.rng_for(0, 0))
    x = synth.activations(1, m.K, synth.rng_for(0, 1))
    y, planes = run_gemv(K, m.fmt, disk, x)
    assert_row_tol(y, oracle.gemm(m.fmt, disk, *planes)[0])


@pytest.mark.parametrize("cfg_index", [1, 3])
def test_gemv_full_size_layers(K, cfg_index):
    """Decode layers at full size (Qwen3-4B-shaped layer; 27B-shaped FFN at M=1),
    every output compared."""
    cfg = synth.configs()[cfg_index]
    for i, m in enumerate(cfg.matrices):
        disk = synth.disk_weights(m.fmt, m.N, m.K, synth.rng_for(cfg_index, 2 * i))
        x = synth.activations(1, m.K, synth.rng_for(cfg_index, 2 * i + 1), outliers=cfg.outliers)
        y, planes = run_gemv(K, m.fmt, disk, x)
        assert_row_tol(y, oracle.gemm(m.fmt, disk, *planes)[0])


@pytest.mark.parametrize("fmt,N,Kdim", [(synth.Q6_K, 2560, 9728), (synth.Q4_K, 2563, 4096),
                                        (synth.Q5_K, 3000, 768), (synth.Q4_K, 4096 + 16 * 3, 256),
                                        (synth.Q6_K, 17, 1024)])
@pytest.mark.parametrize("always_cut", [False, True])
def test_gemv_workspace_modes(K, fmt, N, Kdim, always_cut):
    """With a workspace an SM gets an even share of the superblocks (always,
    under KQ_LAUNCH_GEMV_SPLIT; else where whole row groups leave a warp well
    above it) and the row groups cut between two blocks are finished through
    it; without one the blocks take whole row groups.  All agree with the
    oracle, each gives the same bits on every call, and the workspace is left
    zero-filled."""
    rng = synth.rng_for(112, fmt * 100000 + N + Kdim)
    disk = synth.disk_weights(fmt, N, Kdim, rng)
    x = synth.activations(1, Kdim, rng, outliers=True)
    planes = oracle_q8k(x)
    ref = oracle.gemm(fmt, disk, *planes)[0]
    packed = pack(K, fmt, disk)
    a = q8k_to_dev(K, planes)
    ws = torch.zeros(K.KQ_GEMV_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
    old = K.kq_set_launch_flags(K.KQ_LAUNCH_GEMV_SPLIT if always_cut else 0)
    try:
        for mode in (ws, False):
            outs = []
            for _ in range(3):
                full, y = poisoned((N,))
                K.kq_gemv(fmt, packed, N, Kdim, a, y=y, workspace=mode)
                torch.cuda.synchronize()
                check_guard(full, N)
                outs.append(y.cpu().numpy())
            assert_row_tol(outs[0], ref)
            np.testing.assert_array_equal(outs[1], outs[0])
            np.testing.assert_array_equal(outs[2], outs[0])
    finally:
        K.kq_set_launch_flags(old)
    assert int(torch.count_nonzero(ws)) == 0   # every exchange word emptied again


def test_gemv_row_stride(K):
    """8 rows, each perturbed differently: each output equals its own row's
    dot (the page's multi-row stride gate)."""
    fmt, N, Kdim = synth.Q4_K, 8, 2560
    rng = synth.rng_for(104, 0)
    base = synth.disk_weights(fmt, 1, Kdim, rng)
    disk = np.repeat(base, N, axis=0)
    for n in range(N):
        disk[n, :, 20 + n] ^= np.uint8(0x5A)
    x = synth.activations(1, Kdim, rng)
    y, planes = run_gemv(K, fmt, disk, x)
    for n in range(N):
        assert_row_tol(y[n:n + 1], oracle.gemm(fmt, disk[n:n + 1], *planes)[0], row_max=np.abs(y).max())


# ---------------------------------------------------------------- GEMM
def run_gemm(K, fmt, disk, planes, M):
    N, nsb, _ = disk.shape
    full, y = poisoned((M, N))
    K.kq_gemm(fmt, pack(K, fmt, disk), N, nsb * 256, q8k_to_dev(K, planes), y=y)
    torch.cuda.synchronize()
    check_guard(full, M * N)
    return y.cpu().numpy()


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M,N,Kdim", [(2, 200, 768), (3, 64, 256), (17, 130, 1024), (100, 200, 768),
                                      (129, 136, 512), (300, 250, 1280)])
def test_gemm_small_shapes(K, fmt, M, N, Kdim):
    rng = synth.rng_for(105, fmt * 100000 + M * 100 + N)
    disk = synth.disk_weights(fmt, N, Kdim, rng)
    planes = oracle_q8k(synth.activations(M, Kdim, rng))
    y = run_gemm(K, fmt, disk, planes, M)
    assert_row_tol(y, oracle.gemm(fmt, disk, *planes))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M,N,Kdim", [(5, 333, 2560), (8, 2560, 9728), (9, 1000, 768), (15, 77, 1024),
                                      (6, 40, 17408)])
def test_gemm_small_batch(K, fmt, M, N, Kdim):
    """Small batches (M < 16) run on the decode GEMV's weight stream in passes
    of up to 8 tokens (4 when K is long): every output against the oracle, and
    each token row equal to the GEMV of that token alone."""
    rng = synth.rng_for(114, fmt * 100000 + M * 1000 + N)
    disk = synth.disk_weights(fmt, N, Kdim, rng)
    planes = oracle_q8k(synth.activations(M, Kdim, rng, outliers=True))
    y = run_gemm(K, fmt, disk, planes, M)
    assert_row_tol(y, oracle.gemm(fmt, disk, *planes))
    packed = pack(K, fmt, disk)
    for m in (0, M - 1):
        one = tuple(p[m:m + 1] for p in planes)
        g = K.kq_gemv(fmt, packed, N, Kdim, q8k_to_dev(K, one)).cpu().numpy()
        assert_row_tol(y[m], g.astype(np.float64), rel=1e-5)


def sample_check(y, fmt, disk, planes, rng, n_rows=48, n_toks=6):
    """Oracle on all tokens x sampled rows, and sampled tokens x all rows."""
    M, N = y.shape
    rows = np.sort(rng.choice(N, size=min(n_rows, N), replace=False))
    rows[0], rows[-1] = 0, N - 1
    ref = oracle.gemm(fmt, disk, *planes, n_idx=rows)
    toks = np.unique(np.concatenate([[0, M - 1], rng.choice(M, size=min(n_toks, M), replace=False)]))
    ref_t = oracle.gemm(fmt, disk, *planes, tok_idx=toks)
    assert_row_tol(y[toks], ref_t)
    # sampled rows of every token: scale by the largest |output| among them
    # (never larger than the full row's, so no looser than the bound)
    assert_row_tol(y[:, rows], ref)


@pytest.mark.parametrize("half", [0, 1])
def test_gemm_prefill_qwen3_4b(K, half):
    """Qwen3-4B-shaped prefill pp512: all-Q5_K layer, then all-Q6_K layer."""
    cfg = synth.configs()[2]
    M = cfg.M
    for i, m in enumerate(cfg.matrices[7 * half:7 * half + 7]):
        j = 7 * half + i
        disk = synth.disk_weights(m.fmt, m.N, m.K, synth.rng_for(2, 2 * j))
        planes = oracle_q8k(synth.activations(M, m.K, synth.rng_for(2, 2 * j + 1)))
        y = run_gemm(K, m.fmt, disk, planes, M)
        sample_check(y, m.fmt, disk, planes, synth.rng_for(902, j))


def test_gemm_prefill_27b_ffn(K):
    cfg = synth.configs()[3]
    M = cfg.M
    for i, m in enumerate(cfg.matrices):
        disk = synth.disk_weights(m.fmt, m.N, m.K, synth.rng_for(3, 2 * i))
        planes = oracle_q8k(synth.activations(M, m.K, synth.rng_for(3, 2 * i + 1), outliers=True))
        y = run_gemm(K, m.fmt, disk, planes, M)
        sample_check(y, m.fmt, disk, planes, synth.rng_for(903, i))


def test_gemm_row_equals_gemv(K):
    """Row m of the GEMM equals the GEMV of token m (within the tolerance; the
    int32 partials themselves are checked bit-exact above)."""
    fmt, N, Kdim, M = synth.Q6_K, 300, 2560, 40
    rng = synth.rng_for(106, 0)
    disk = synth.disk_weights(fmt, N, Kdim, rng)
    planes = oracle_q8k(synth.activations(M, Kdim, rng))
    y = run_gemm(K, fmt, disk, planes, M)
    packed = pack(K, fmt, disk)
    for m in (0, 17, M - 1):
        one = tuple(p[m:m + 1] for p in planes)
        g = K.kq_gemv(fmt, packed, N, Kdim, q8k_to_dev(K, one)).cpu().numpy()
        assert_row_tol(y[m], g)


# ---------------------------------------------------------------- grouped
def run_grouped(K, fmt, disks, planes, offsets):
    E = len(disks)
    N, nsb, _ = disks[0].shape
    Kdim = nsb * 256
    per = K.kq_repack_bytes(fmt, N, Kdim)
    packed = torch.empty(per * E, dtype=torch.uint8, device="cuda")
    for e in range(E):
        K.kq_repack(fmt, to_dev(disks[e].reshape(-1)), N, Kdim, packed=packed[e * per:(e + 1) * per])
    M = int(offsets[-1])
    full, y = poisoned((M, N))
    K.kq_gemm_grouped(fmt, packed, E, to_dev(offsets.astype(np.int32)), N, Kdim, q8k_to_dev(K, planes), y=y)
    torch.cuda.synchronize()
    check_guard(full, M * N)
    return y.cpu().numpy()


@pytest.mark.parametrize("fmt", FMTS)
def test_grouped_uneven_and_empty_experts(K, fmt):
    rng = synth.rng_for(107, fmt)
    E, N, Kdim = 6, 72, 512
    counts = np.array([5, 0, 17, 1, 0, 40])
    offsets = np.concatenate([[0], np.cumsum(counts)])
    disks = [synth.disk_weights(fmt, N, Kdim, rng) for _ in range(E)]
    planes = oracle_q8k(synth.activations(int(offsets[-1]), Kdim, rng))
    y = run_grouped(K, fmt, disks, planes, offsets)
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        if a == b:
            continue
        sl = tuple(p[a:b] for p in planes)
        assert_row_tol(y[a:b], oracle.gemm(fmt, disks[e], *sl))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("counts", [[0, 300, 0, 129, 1, 0, 270], [0, 0, 600], [128, 0, 256, 17]])
def test_grouped_later_token_tiles(K, fmt, counts):
    """Experts with more rows than one 128-token tile (the later tiles are
    found from the offsets), empty experts among them (also first, whose
    weights the kernel unpacks before it knows the expert is empty), a weight
    tile count with a ragged tail (N = 300), and all rows on one expert:
    every output against the oracle with its expert."""
    rng = synth.rng_for(118, fmt * 100 + len(counts))
    E, N, Kdim = len(counts), 300, 512
    offsets = np.concatenate([[0], np.cumsum(counts)])
    disks = [synth.disk_weights(fmt, N, Kdim, rng) for _ in range(E)]
    planes = oracle_q8k(synth.activations(int(offsets[-1]), Kdim, rng))
    y = run_grouped(K, fmt, disks, planes, offsets)
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        if a == b:
            continue
        sl = tuple(p[a:b] for p in planes)
        assert_row_tol(y[a:b], oracle.gemm(fmt, disks[e], *sl))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("counts", [[0, 1, 0, 0, 1, 1, 0, 1, 0, 1, 1, 0, 0, 1, 0, 1],
                                    [0, 3, 0, 1, 2, 0, 0, 5, 0, 0, 1, 0, 0, 0, 1, 0]])
def test_grouped_decode_rows(K, fmt, counts):
    """A few rows grouped by expert (MoE decode: one token routed to 8 of 16
    experts; and 13 rows with several on one expert) run as one GEMV over
    every row's expert: each row against the oracle with its own expert."""
    rng = synth.rng_for(115, fmt * 10 + sum(counts))
    E, N, Kdim = len(counts), 200, 1024
    offsets = np.concatenate([[0], np.cumsum(counts)])
    disks = [synth.disk_weights(fmt, N, Kdim, rng) for _ in range(E)]
    planes = oracle_q8k(synth.activations(int(offsets[-1]), Kdim, rng))
    y = run_grouped(K, fmt, disks, planes, offsets)
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        if a == b:
            continue
        sl = tuple(p[a:b] for p in planes)
        assert_row_tol(y[a:b], oracle.gemm(fmt, disks[e], *sl))


def test_grouped_moe_30b_a3b(K):
    """The MoE workload: 128 experts, top-8 of 512 tokens (4096 rows grouped by
    expert); gate/up Q4_K [768 x 2048], down Q6_K [2048 x 768]."""
    cfg = synth.configs()[4]
    T, E = cfg.M, cfg.experts
    row_token, row_expert, offsets = synth.moe_routing(T, E, cfg.topk, synth.rng_for(4, 0))
    x_tok = synth.activations(T, 2048, synth.rng_for(4, 1))
    check_rng = synth.rng_for(904, 0)
    for i, m in enumerate(cfg.matrices):
        disks = [synth.disk_weights(m.fmt, m.N, m.K, synth.rng_for(4, 10 + 1000 * i + e)) for e in range(E)]
        if m.name == "down":
            x = synth.activations(len(row_token), m.K, synth.rng_for(4, 2))
        else:
            x = x_tok[row_token]
        planes = oracle_q8k(x)
        y = run_grouped(K, m.fmt, disks, planes, offsets)
        # every expert's first and last row, plus a few random rows, all N
        rows = set()
        for e in range(E):
            if offsets[e] < offsets[e + 1]:
                rows.update({int(offsets[e]), int(offsets[e + 1]) - 1})
        rows.update(check_rng.choice(len(row_token), 32, replace=False).tolist())
        for r in sorted(rows):
            e = int(row_expert[r])
            one = tuple(p[r:r + 1] for p in planes)
            assert_row_tol(y[r:r + 1], oracle.gemm(m.fmt, disks[e], *one))


# ---------------------------------------------------------------- PDL chains
def test_pdl_chain_matches_plain_launches(K):
    """With programmatic dependent launch on, a chain of producer kernel ->
    quantize -> GEMV -> consumer gives the same bits as plain launches: each
    kernel waits for the previous ones before touching their data."""
    fmt, N, Kdim = synth.Q4_K, 4096, 2560
    rng = synth.rng_for(108, 0)
    disk = synth.disk_weights(fmt, N, Kdim, rng)
    packed = pack(K, fmt, disk)
    x0 = to_dev(synth.activations(1, Kdim, rng))
    torch.cuda.synchronize()

    def chain():
        outs = []
        a = K.q8k_empty(1, Kdim)
        for i in range(6):
            x = x0 * (1.0 + 0.25 * i)          # produced by the kernel right before
            K.kq_quantize_q8k(x, out=a)
            y = K.kq_gemv(fmt, packed, N, Kdim, a)
            outs.append(y * 2.0)               # consumed right after
        torch.cuda.synchronize()
        return torch.stack(outs).cpu().numpy()

    old = K.kq_set_launch_flags(0)
    try:
        plain = chain()
        K.kq_set_launch_flags(K.KQ_LAUNCH_PDL)
        assert K.kq_get_launch_flags() == K.KQ_LAUNCH_PDL
        pdl = chain()
    finally:
        K.kq_set_launch_flags(old)
    np.testing.assert_array_equal(pdl, plain)
    planes = oracle_q8k((x0 * 2.25).cpu().numpy())
    assert_row_tol(pdl[5] / 2.0, oracle.gemm(fmt, disk, *planes)[0])


def test_pdl_gemm_chain_matches_plain_launches(K):
    """The same for the tensor-core GEMM (dense and grouped): with programmatic
    dependent launch the GEMM's unpack starts before the activation image is
    written, and every output still equals the plain launches' bits."""
    fmt, N, Kdim, M = synth.Q5_K, 384, 1024, 96
    rng = synth.rng_for(116, 0)
    disk = synth.disk_weights(fmt, N, Kdim, rng)
    packed = pack(K, fmt, disk)
    E = 3
    disks = [synth.disk_weights(fmt, N, Kdim, rng) for _ in range(E)]
    per = K.kq_repack_bytes(fmt, N, Kdim)
    packed_e = torch.empty(per * E, dtype=torch.uint8, device="cuda")
    for e in range(E):
        K.kq_repack(fmt, to_dev(disks[e].reshape(-1)), N, Kdim, packed=packed_e[e * per:(e + 1) * per])
    offsets = to_dev(np.array([0, 40, 40, M], np.int32))
    x0 = to_dev(synth.activations(M, Kdim, rng))
    torch.cuda.synchronize()

    def chain():
        outs = []
        a = K.q8k_empty(M, Kdim)
        for i in range(4):
            x = x0 * (1.0 + 0.25 * i)          # produced by the kernel right before
            K.kq_quantize_q8k(x, out=a)
            y = K.kq_gemm(fmt, packed, N, Kdim, a)
            yg = K.kq_gemm_grouped(fmt, packed_e, E, offsets, N, Kdim, a)
            outs.append(torch.cat([y * 2.0, yg * 2.0]))   # consumed right after
        torch.cuda.synchronize()
        return torch.stack(outs).cpu().numpy()

    old = K.kq_set_launch_flags(0)
    try:
        plain = chain()
        K.kq_set_launch_flags(K.KQ_LAUNCH_PDL)
        pdl = chain()
    finally:
        K.kq_set_launch_flags(old)
    np.testing.assert_array_equal(pdl, plain)
    planes = oracle_q8k((x0 * 1.75).cpu().numpy())
    assert_row_tol(pdl[3][:M] / 2.0, oracle.gemm(fmt, disk, *planes))


# ---------------------------------------------------------------- fused GEMV
@pytest.mark.parametrize("fmt", FMTS)
def test_gemv_fused_multi_matrix_bit_identical(K, fmt):
    """kq_gemv_fused over several matrices sharing x agrees with kq_quantize_q8k
    + kq_gemv per matrix (the quantization is bit-identical; the fp32 sums
    may be split differently across warps) and with the oracle."""
    rng = synth.rng_for(109, fmt)
    Kdim = 2560
    Ns = [4096, 1000, 8, 333]
    disks = [synth.disk_weights(fmt, N, Kdim, rng) for N in Ns]
    packs = [pack(K, fmt, d) for d in disks]
    x = synth.activations(1, Kdim, rng, outliers=True)
    xd = to_dev(x[0])
    ys = K.kq_gemv_fused(fmt, packs, Ns, Kdim, xd)
    a = K.kq_quantize_q8k(xd)
    planes = oracle_q8k(x)
    for N, pk, y, disk in zip(Ns, packs, ys, disks):
        y_sep = K.kq_gemv(fmt, pk, N, Kdim, a)
        torch.cuda.synchronize()
        assert_row_tol(y.cpu().numpy(), y_sep.cpu().numpy().astype(np.float64), rel=1e-5)
        assert_row_tol(y.cpu().numpy(), oracle.gemm(fmt, disk, *planes)[0])


@pytest.mark.parametrize("fmt", FMTS)
def test_gemv_fused_cuts_across_matrices(K, fmt):
    """Ragged matrices and few superblocks per row group: the blocks' item
    ranges cut row groups at matrix edges and inside them."""
    rng = synth.rng_for(113, fmt)
    Kdim = 768
    Ns = [1000, 8, 333, 4100]
    disks = [synth.disk_weights(fmt, N, Kdim, rng) for N in Ns]
    packs = [pack(K, fmt, d) for d in disks]
    x = synth.activations(1, Kdim, rng)
    planes = oracle_q8k(x)
    old = K.kq_set_launch_flags(K.KQ_LAUNCH_GEMV_SPLIT)
    try:
        fulls = [poisoned((N,)) for N in Ns]
        K.kq_gemv_fused(fmt, packs, Ns, Kdim, to_dev(x[0]), [f[1] for f in fulls])
        torch.cuda.synchronize()
    finally:
        K.kq_set_launch_flags(old)
    for N, disk, (full, y) in zip(Ns, disks, fulls):
        check_guard(full, N)
        assert_row_tol(y.cpu().numpy(), oracle.gemm(fmt, disk, *planes)[0])


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M,Kdim", [(2, 2560), (3, 1024), (5, 4096), (8, 768), (11, 256), (6, 9728)])
def test_gemv_fused_batch(K, fmt, M, Kdim):
    """Fused quantize + GEMV of a small batch over several matrices sharing the
    rows: every output of every row against the oracle on that row's Q8_K
    planes (the in-kernel quantization is bit-identical to kq_quantize_q8k),
    and row 0 equal to kq_gemv_fused of that row alone."""
    rng = synth.rng_for(117, fmt * 1000 + M * 10 + Kdim // 256)
    Ns = [300, 16, 77]
    disks = [synth.disk_weights(fmt, N, Kdim, rng) for N in Ns]
    packs = [pack(K, fmt, d) for d in disks]
    x = synth.activations(M, Kdim, rng, outliers=True)
    fulls = [poisoned((M, N)) for N in Ns]
    K.kq_gemv_fused_batch(fmt, packs, Ns, Kdim, to_dev(x), [f[1] for f in fulls])
    torch.cuda.synchronize()
    planes = oracle_q8k(x)
    for N, disk, (full, y) in zip(Ns, disks, fulls):
        check_guard(full, M * N)
        assert_row_tol(y.cpu().numpy(), oracle.gemm(fmt, disk, *planes))
    one = K.kq_gemv_fused(fmt, packs, Ns, Kdim, to_dev(x[0]))
    for (full, y), y1 in zip(fulls, one):
        assert_row_tol(y[0].cpu().numpy(), y1.cpu().numpy().astype(np.float64), rel=1e-5)


def test_gemv_fused_layer_groups_and_edges(K):
    """The decode layer's launch groups (q/k/v; gate/up), a single-superblock
    K, N = 1, a skipped empty matrix, and the host-side argument checks."""
    fmt = synth.Q4_K
    rng = synth.rng_for(110, 0)
    for Kdim, Ns in ((2560, [4096, 1024, 1024]), (2560, [9728, 9728]), (256, [1, 7, 0, 9])):
        disks = [synth.disk_weights(fmt, max(N, 1), Kdim, rng) for N in Ns]
        packs = [pack(K, fmt, d) for d in disks]
        x = synth.activations(1, Kdim, rng)
        fulls = [poisoned((max(N, 1),)) for N in Ns]
        K.kq_gemv_fused(fmt, packs, Ns, Kdim, to_dev(x[0]), [f[1] for f in fulls])
        torch.cuda.synchronize()
        planes = oracle_q8k(x)
        for N, disk, (full, y) in zip(Ns, disks, fulls):
            if N == 0:
                assert np.isnan(full.cpu().numpy()).all()
                continue
            check_guard(full, N)
            assert_row_tol(y.cpu().numpy(), oracle.gemm(fmt, disk[:N], *planes)[0])
    with pytest.raises(K.KQError):
        K.kq_gemv_fused(fmt, packs * 2, [1] * 8, 256, to_dev(x[0]))       # more than 4 matrices
    with pytest.raises(K.KQError):
        K.kq_gemv_fused(fmt, packs[:1], [1], 40960 + 256, to_dev(np.zeros(41216, np.float32)))


# ---------------------------------------------------------------- Q6_K sub-scale range
@pytest.mark.parametrize("sc_range", [(-128, 128), (-64, 65), (60, 70), (-62, 63)])
def test_gemm_q6k_full_subscale_range(K, sc_range):
    """Real Q6_K files use signed sub-scales over the whole int8 range, beyond
    what one exact fp16 plane holds (|sc| <= 62); the tensor-core path splits
    those superblocks into two exact planes.  Checked against the oracle."""
    fmt, M, N, Kdim = synth.Q6_K, 64, 256, 1024
    rng = synth.rng_for(111, sc_range[0] + 1000)
    disk = synth.disk_weights(fmt, N, Kdim, rng)
    lo, hi = sc_range
    disk[..., 192:208] = rng.integers(lo, hi, size=(N, Kdim // 256, 16)).astype(np.int8).view(np.uint8)
    planes = oracle_q8k(synth.activations(M, Kdim, rng))
    y = run_gemm(K, fmt, disk, planes, M)
    assert_row_tol(y, oracle.gemm(fmt, disk, *planes))
    # the GEMV on the same weights agrees too
    one = tuple(p[:1] for p in planes)
    g = K.kq_gemv(fmt, pack(K, fmt, disk), N, Kdim, q8k_to_dev(K, one)).cpu().numpy()
    assert_row_tol(g, oracle.gemm(fmt, disk, *one)[0])


def test_gemm_device_status_clean(K):
    """After the tensor-core launches above, no bounded wait has timed out."""
    assert K.kq_device_status() == 0


def test_measure_mma_s8_checksum(K):
    """The int8 mma.sync rate kernel does the MMAs it claims: all-ones
    operands give 32 per MMA per accumulator, 1024 * iters per thread."""
    out = K.kq_measure_mma_s8(3, 7)
    torch.cuda.synchronize()
    assert out.shape == (3 * 256,)
    assert bool((out == 1024 * 7).all())


# ---------------------------------------------------------------- Q8_0 rail
@pytest.mark.parametrize("M,Kdim,outliers", [(1, 256, False), (3, 5120, True), (2, 96, False), (5, 17408, False)])
def test_q8_0_quantize_bit_exact(K, M, Kdim, outliers):
    """Q8_0-form activations: scales and quants bit-identical to the oracle,
    including a zero block, 1e-30 values, exact ties and a large outlier."""
    rng = synth.rng_for(120, M * 7 + Kdim)
    x = synth.activations(M, Kdim, rng, outliers=outliers)
    if M >= 3:
        x[0, :32] = 0.0
        x[1, 32:64] *= np.float32(1e-30)
        x[2, :32] = np.float32(2.5)
        x[2, 0] = np.float32(127.0)
        x[2, 40] = np.float32(3e4)
    ref_d, ref_q = oracle.quantize_q8_0(x)
    d, q = K.kq_quantize_q8_0(to_dev(x))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(d.cpu().numpy(), ref_d)
    np.testing.assert_array_equal(q.cpu().numpy(), ref_q)


def _q8_0_image(disk: np.ndarray) -> np.ndarray:
    """The Q8_0 image layout written out independently (test side): qs plane of
    4096-byte chunks (row r's 16 quants of columns 16k.. at 256k + 16r), then
    the fp16 scale plane of 256-byte chunks (row r's 8 scales at 16r)."""
    N, nb, _ = disk.shape
    nsb, groups = nb // 8, -(-N // 16)
    rows = np.zeros((groups * 16, nb, 34), np.uint8)
    rows[:N] = disk
    q = rows[:, :, 2:].reshape(groups, 16, nsb, 16, 16)          # g, r, sb, piece k, byte
    qs = q.transpose(0, 2, 3, 1, 4).reshape(-1)                    # chunk (g, sb), 256k + 16r + byte
    d = rows[:, :, :2].reshape(groups, 16, nsb, 16).transpose(0, 2, 1, 3).reshape(-1)
    pad = lambda a: np.concatenate([a, np.zeros(-len(a) % 256, np.uint8)])
    return np.concatenate([pad(qs), pad(d)])


@pytest.mark.parametrize("N,Kdim", [(1, 256), (37, 512), (200, 2560)])
def test_q8_0_repack_layout(K, N, Kdim):
    """The repacked Q8_0 image equals the documented layout byte for byte
    (every disk byte kept once, padding rows zero)."""
    disk = synth.disk_weights_q8_0(N, Kdim, synth.rng_for(121, N))
    packed = K.kq_repack(synth.Q8_0, to_dev(disk.reshape(-1)), N, Kdim)
    torch.cuda.synchronize()
    want = _q8_0_image(disk)
    got = packed.cpu().numpy()
    assert got.size == K.kq_repack_bytes(synth.Q8_0, N, Kdim) == want.size
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("N,Kdim", [(256, 1024), (300, 2560), (17, 256), (1, 5120), (4096, 2560),
                                    (5120, 17408), (17408, 5120), (40, 40960)])
def test_q8_0_gemv(K, N, Kdim):
    """Q8_0 GEMV against the oracle on every output (ragged row groups, one
    superblock, the longest K), and bit-identical on a second run."""
    rng = synth.rng_for(122, N + Kdim)
    disk = synth.disk_weights_q8_0(N, Kdim, rng)
    x = synth.activations(1, Kdim, rng, outliers=True)
    d_a, q_a = oracle.quantize_q8_0(x)
    packed = K.kq_repack(synth.Q8_0, to_dev(disk.reshape(-1)), N, Kdim)
    full, y = poisoned((N,))
    dd, qd = to_dev(d_a[0]), to_dev(q_a[0])
    K.kq_gemv_q8_0(packed, N, Kdim, dd, qd, y=y)
    y2 = K.kq_gemv_q8_0(packed, N, Kdim, dd, qd)
    torch.cuda.synchronize()
    check_guard(full, N)
    assert_row_tol(y.cpu().numpy()[None, :], oracle.gemv_q8_0(disk, d_a, q_a))
    assert torch.equal(y, y2)


@pytest.mark.parametrize("N,Kdim", [(300, 2560), (17, 256), (5120, 17408), (17408, 5120), (40, 40960)])
def test_q8_0_fused_equals_quantize_then_gemv(K, N, Kdim):
    """The fused Q8_0 GEMV quantizes the row inside every block: its output is
    bit-identical to kq_quantize_q8_0 followed by kq_gemv_q8_0 (zero block,
    tiny and outlier values included), and within tolerance of the oracle."""
    rng = synth.rng_for(124, N + Kdim)
    disk = synth.disk_weights_q8_0(N, Kdim, rng)
    x = synth.activations(1, Kdim, rng, outliers=True)
    x[0, :32] = 0.0
    x[0, 64:96] *= np.float32(1e-30)
    packed = K.kq_repack(synth.Q8_0, to_dev(disk.reshape(-1)), N, Kdim)
    xd = to_dev(x[0])
    d, q = K.kq_quantize_q8_0(xd)
    want = K.kq_gemv_q8_0(packed, N, Kdim, d, q)
    full, y = poisoned((N,))
    K.kq_gemv_q8_0_fused(packed, N, Kdim, xd, y=y)
    torch.cuda.synchronize()
    check_guard(full, N)
    assert torch.equal(y, want)
    d_a, q_a = oracle.quantize_q8_0(x)
    assert_row_tol(y.cpu().numpy()[None, :], oracle.gemv_q8_0(disk, d_a, q_a))


def test_q8_0_pdl_chain_matches_plain_launches(K):
    """The Q8_0 rail under programmatic dependent launch: the GEMV loads its
    first weights before the dependency wait, while the activations are still
    being written by the kernel launched just before it (the quantize, or for
    the fused form the elementwise op); every output equals the plain
    launches' bits, and the last against the oracle."""
    N, Kdim = 300, 2560
    rng = synth.rng_for(123, 0)
    disk = synth.disk_weights_q8_0(N, Kdim, rng)
    disk2 = synth.disk_weights_q8_0(N, 5120, rng)
    packed = K.kq_repack(synth.Q8_0, to_dev(disk.reshape(-1)), N, Kdim)
    packed2 = K.kq_repack(synth.Q8_0, to_dev(disk2.reshape(-1)), N, 5120)
    x0 = to_dev(synth.activations(1, Kdim, rng)[0])
    h0 = to_dev(synth.activations(1, 5120, rng)[0])
    torch.cuda.synchronize()

    def chain():
        outs = []
        for i in range(4):
            x = x0 * (1.0 + 0.25 * i)            # produced by the kernel right before
            d, q = K.kq_quantize_q8_0(x)
            y = K.kq_gemv_q8_0(packed, N, Kdim, d, q)
            d2, q2 = K.kq_quantize_q8_0(h0 + y.sum() * 0.0 + 0.1 * i)
            y2 = K.kq_gemv_q8_0(packed2, N, 5120, d2, q2)
            y3 = K.kq_gemv_q8_0_fused(packed2, N, 5120, y2[:1].repeat(5120) * 0.0 + h0 * (0.5 + i))
            outs.append(torch.cat([y * 2.0, y2 * 2.0, y3]))   # consumed right after
        torch.cuda.synchronize()
        return torch.stack(outs).cpu().numpy()

    old = K.kq_set_launch_flags(0)
    try:
        plain = chain()
        K.kq_set_launch_flags(K.KQ_LAUNCH_PDL)
        pdl = chain()
    finally:
        K.kq_set_launch_flags(old)
    np.testing.assert_array_equal(pdl, plain)
    d_a, q_a = oracle.quantize_q8_0((x0 * 1.75).cpu().numpy())
    assert_row_tol(pdl[3][None, :N] / 2.0, oracle.gemv_q8_0(disk, d_a, q_a))


def test_grouped_more_experts_than_the_tensor_core_path(K):
    """E above the grouped tensor-core kernel's expert limit: the call runs
    on the CUDA-core token-group kernel; every row against the oracle with its
    own expert (empty experts among them)."""
    fmt, E, N, Kdim = synth.Q4_K, 1100, 64, 256
    rng = synth.rng_for(124, 0)
    counts = np.zeros(E, np.int64)
    counts[rng.choice(E, 30, replace=False)] = rng.integers(1, 4, size=30)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    disks = [synth.disk_weights(fmt, N, Kdim, rng) for _ in range(E)]
    planes = oracle_q8k(synth.activations(int(offsets[-1]), Kdim, rng))
    y = run_grouped(K, fmt, disks, planes, offsets)
    for e in np.nonzero(counts)[0]:
        a, b = offsets[e], offsets[e + 1]
        sl = tuple(p[a:b] for p in planes)
        assert_row_tol(y[a:b], oracle.gemm(fmt, disks[e], *sl))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("counts,sets", [([0, 1, 0, 0, 1, 1, 0, 1, 0, 1, 1, 0, 0, 1, 0, 1], 2),
                                         ([0, 3, 0, 1, 2, 0, 0, 5, 0, 0, 1, 0, 0, 0, 1, 0], 1),
                                         ([2, 0, 1, 0, 0, 1], 4)])
def test_grouped_decode_fused(K, fmt, counts, sets):
    """MoE decode with the quantize in the kernel and several weight sets per
    launch (gate and up): every row of every set against the oracle with its
    own expert, and bit-identical to quantize + kq_gemm_grouped per set."""
    rng = synth.rng_for(125, fmt * 100 + sets * 10 + len(counts))
    E, Kdim = len(counts), 1024
    Ns = [200, 136, 77, 16][:sets]
    offsets = np.concatenate([[0], np.cumsum(counts)])
    M = int(offsets[-1])
    disks = [[synth.disk_weights(fmt, N, Kdim, rng) for _ in range(E)] for N in Ns]
    packs = []
    for st, N in enumerate(Ns):
        per = K.kq_repack_bytes(fmt, N, Kdim)
        buf = torch.empty(per * E, dtype=torch.uint8, device="cuda")
        for e in range(E):
            K.kq_repack(fmt, to_dev(disks[st][e].reshape(-1)), N, Kdim, packed=buf[e * per:(e + 1) * per])
        packs.append(buf)
    x = synth.activations(M, Kdim, rng, outliers=True)
    off_d = to_dev(offsets.astype(np.int32))
    fulls = [poisoned((M, N)) for N in Ns]
    K.kq_gemv_grouped_fused(fmt, packs, Ns, Kdim, E, off_d, to_dev(x), [f[1] for f in fulls])
    a = K.kq_quantize_q8k(to_dev(x))
    refs = [K.kq_gemm_grouped(fmt, packs[st], E, off_d, N, Kdim, a) for st, N in enumerate(Ns)]
    torch.cuda.synchronize()
    planes = oracle_q8k(x)
    for st, N in enumerate(Ns):
        full, y = fulls[st]
        check_guard(full, M * N)
        assert torch.equal(y, refs[st])
        got = y.cpu().numpy()
        for e in range(E):
            lo, hi = offsets[e], offsets[e + 1]
            if lo < hi:
                sl = tuple(p[lo:hi] for p in planes)
                assert_row_tol(got[lo:hi], oracle.gemm(fmt, disks[st][e], *sl))


def test_grouped_decode_fused_uncovered_row_and_limits(K):
    """A row that no expert range holds is left untouched; the limits on sets
    x rows are checked on the host."""
    fmt, E, N, Kdim = synth.Q4_K, 4, 64, 512
    rng = synth.rng_for(126, 0)
    disk = [synth.disk_weights(fmt, N, Kdim, rng) for _ in range(E)]
    per = K.kq_repack_bytes(fmt, N, Kdim)
    buf = torch.empty(per * E, dtype=torch.uint8, device="cuda")
    for e in range(E):
        K.kq_repack(fmt, to_dev(disk[e].reshape(-1)), N, Kdim, packed=buf[e * per:(e + 1) * per])
    x = synth.activations(3, Kdim, rng)
    off_d = to_dev(np.array([0, 1, 1, 2, 2], np.int32))     # row 2 outside every range
    full, y = poisoned((3, N))
    K.kq_gemv_grouped_fused(fmt, [buf], [N], Kdim, E, off_d, to_dev(x), [y])
    torch.cuda.synchronize()
    got = y.cpu().numpy()
    assert np.isnan(got[2]).all()
    planes = oracle_q8k(x)
    assert_row_tol(got[0:1], oracle.gemm(fmt, disk[0], *(p[0:1] for p in planes)))
    assert_row_tol(got[1:2], oracle.gemm(fmt, disk[2], *(p[1:2] for p in planes)))
    with pytest.raises(K.KQError):   # 3 sets x 6 rows > 16 matrices
        K.kq_gemv_grouped_fused(fmt, [buf] * 3, [N] * 3, Kdim, E, off_d, to_dev(synth.activations(6, Kdim, rng)))


def test_moe_decode_bench_shapes(K):
    """The MoE decode the benchmark times, at its shapes: one token routed to 8
    of 128 experts, gate and up (Q4_K 768x2048) in one kq_gemv_grouped_fused
    launch, down (Q6_K 2048x768) in another; every output of every routed
    row against the oracle with its expert (only the routed experts' images
    are written: the kernel reads no other)."""
    cfg = synth.configs()[4]
    E, topk = cfg.experts, cfg.topk
    gate, up, down = cfg.matrices
    rng = synth.rng_for(127, 0)
    chosen = np.sort(rng.choice(E, topk, replace=False))
    cnt = np.zeros(E, np.int64)
    cnt[chosen] = 1
    off_d = to_dev(np.concatenate([[0], np.cumsum(cnt)]).astype(np.int32))

    def images(m, seed):
        per = K.kq_repack_bytes(m.fmt, m.N, m.K)
        buf = torch.empty(per * E, dtype=torch.uint8, device="cuda")
        disks = {}
        for e in chosen:
            disks[e] = synth.disk_weights(m.fmt, m.N, m.K, synth.rng_for(127, seed + int(e)))
            K.kq_repack(m.fmt, to_dev(disks[e].reshape(-1)), m.N, m.K, packed=buf[int(e) * per:(int(e) + 1) * per])
        return buf, disks

    (pg, dg), (pu, du), (pd, dd) = images(gate, 1000), images(up, 2000), images(down, 3000)
    x = np.repeat(synth.activations(1, gate.K, rng), topk, axis=0)
    h = synth.activations(topk, down.K, rng)
    yg, yu = K.kq_gemv_grouped_fused(gate.fmt, [pg, pu], [gate.N, up.N], gate.K, E, off_d, to_dev(x))
    (yd,) = K.kq_gemv_grouped_fused(down.fmt, [pd], [down.N], down.K, E, off_d, to_dev(h))
    torch.cuda.synchronize()
    px, ph = oracle_q8k(x), oracle_q8k(h)
    for row, e in enumerate(chosen):
        one = tuple(p[row:row + 1] for p in px)
        assert_row_tol(yg[row:row + 1].cpu().numpy(), oracle.gemm(gate.fmt, dg[e], *one))
        assert_row_tol(yu[row:row + 1].cpu().numpy(), oracle.gemm(up.fmt, du[e], *one))
        oneh = tuple(p[row:row + 1] for p in ph)
        assert_row_tol(yd[row:row + 1].cpu().numpy(), oracle.gemm(down.fmt, dd[e], *oneh))


def test_bounded_wait_times_out_and_reports(K):
    """Failure detection without a GPU fault: a wait that nothing satisfies
    gives up after its limit (2 ms here), kq_device_status reports
    KQ_ERR_TIMEOUT once and clears it, and the context stays usable."""
    assert K.kq_device_status() == 0
    K.kq_debug_wait_timeout(2_000_000)
    torch.cuda.synchronize()
    assert K.kq_device_status() == -5          # KQ_ERR_TIMEOUT
    assert K.kq_device_status() == 0           # read and cleared
    fmt, N, Kdim = synth.Q4_K, 64, 512
    disk = synth.disk_weights(fmt, N, Kdim, synth.rng_for(128, 0))
    x = synth.activations(1, Kdim, synth.rng_for(128, 1))
    y = K.kq_gemv(fmt, pack(K, fmt, disk), N, Kdim, q8k_to_dev(K, oracle_q8k(x)))
    torch.cuda.synchronize()
    assert_row_tol(y.cpu().numpy()[None, :], oracle.gemm(fmt, disk, *oracle_q8k(x)))
    assert K.kq_device_status() == 0


@pytest.mark.parametrize("M", [2, 4, 8])
def test_gemv_fused_batch_layer_shapes(K, M):
    """The small-batch line's launches at its shapes: the Qwen3-4B-shaped
    layer's four groups (q/k/v, o, gate/up, down) through kq_gemv_fused_batch
    with M rows; every output of every matrix against the oracle."""
    layer = synth.configs()[1].matrices
    by = {m.name: m for m in layer}
    groups = [["wq", "wk", "wv"], ["wo"], ["gate", "up"], ["down"]]
    rng = synth.rng_for(129, M)
    for names in groups:
        ms = [by[n] for n in names]
        disks = [synth.disk_weights(m.fmt, m.N, m.K, rng) for m in ms]
        packs = [pack(K, m.fmt, d) for m, d in zip(ms, disks)]
        x = synth.activations(M, ms[0].K, rng)
        ys = K.kq_gemv_fused_batch(ms[0].fmt, packs, [m.N for m in ms], ms[0].K, to_dev(x))
        torch.cuda.synchronize()
        planes = oracle_q8k(x)
        for m, d, y in zip(ms, disks, ys):
            assert_row_tol(y.cpu().numpy(), oracle.gemm(m.fmt, d, *planes))


# ---------------------------------------------------------------- host transport
def test_copy_in_from_pinned_host(K):
    """kq_copy_in moves pinned host bytes into device memory exactly, for
    sizes that leave partial blocks and partial vectors of the copy grid."""
    g = torch.Generator().manual_seed(7)
    for n in (4, 516, 4096 + 12, 18944):
        src = torch.randint(-2**31, 2**31 - 1, (n,), dtype=torch.int32, generator=g).pin_memory()
        full, dst = poisoned((n,))
        K.kq_copy_in(src, dst.view(torch.int32))
        torch.cuda.synchronize()
        assert torch.equal(dst.view(torch.int32).cpu(), src)
        check_guard(full, n)  # nothing written past the end


def test_copy_in_chain_under_pdl(K):
    """Under programmatic dependent launch kq_copy_in reads the host rows
    early but overwrites the device row only after the GEMV before it (which
    reads that row) has finished: every output equals the plain launches',
    and each against the oracle on its own row."""
    fmt, N, Kdim = synth.Q4_K, 300, 2560
    rng = synth.rng_for(131, 0)
    disk = synth.disk_weights(fmt, N, Kdim, rng)
    packed = pack(K, fmt, disk)
    rows = synth.activations(4, Kdim, rng, outliers=True)
    hosts = [torch.from_numpy(rows[i].copy()).pin_memory() for i in range(4)]
    x_dev = torch.empty(Kdim, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()

    def chain():
        outs = []
        for i in range(4):
            K.kq_copy_in(hosts[i], x_dev)
            outs.append(K.kq_gemv_fused(fmt, [packed], [N], Kdim, x_dev)[0])
        torch.cuda.synchronize()
        return torch.stack(outs).cpu().numpy()

    old = K.kq_set_launch_flags(0)
    try:
        plain = chain()
        K.kq_set_launch_flags(K.KQ_LAUNCH_PDL)
        pdl = chain()
    finally:
        K.kq_set_launch_flags(old)
    np.testing.assert_array_equal(pdl, plain)
    planes = oracle_q8k(rows)
    assert_row_tol(pdl, oracle.gemm(fmt, disk, *planes))


def test_gemv_fused_writes_pinned_host_outputs(K):
    """The fused GEMV stores into pinned host outputs directly: the same bits
    as device outputs, nothing written past the rows."""
    fmt, Kdim, Ns = synth.Q6_K, 9728, [2560]
    rng = synth.rng_for(132, 0)
    disk = synth.disk_weights(fmt, Ns[0], Kdim, rng)
    packed = pack(K, fmt, disk)
    x = to_dev(synth.activations(1, Kdim, rng)[0])
    y_dev = K.kq_gemv_fused(fmt, [packed], Ns, Kdim, x)[0]
    y_host = torch.full((Ns[0] + 16,), float("nan"), dtype=torch.float32).pin_memory()
    K.kq_gemv_fused(fmt, [packed], Ns, Kdim, x, [y_host[:Ns[0]]])
    torch.cuda.synchronize()
    assert torch.equal(y_host[:Ns[0]], y_dev.cpu())
    assert bool(torch.isnan(y_host[Ns[0]:]).all())

