"""The tensor-core GEMM's integer sums, bit for bit.

kq_debug_gemm_partials runs the kq_gemm / kq_gemm_grouped kernel with its
epilogue switched from the float fold to integers: the exact per-superblock
int32 sums isum and msum the tensor pipe's accumulator units add up to.  They
must equal the oracle's partials and the decode GEMV's (kq_debug_partials):
[kq-arc], kq v3 panel-scratch commit, the tile-vs-GEMV bit-exactness gate,
and k5/k6 kq-v2 commit, the int32 folds exact with |iacc|, |32*bacc| < 2^28.
The worst-case fields push every superblock sum far past 2^24, where an fp32
accumulator over a whole superblock would round.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_gemv_gemm_gb300 import synth

from gpu_util import kq, oracle_q8k, pack, q8k_to_dev, to_dev

pytestmark = pytest.mark.gpu
FMTS = [synth.Q4_K, synth.Q5_K, synth.Q6_K]


@pytest.fixture(scope="module")
def K():
    assert torch.cuda.is_available()
    return kq()


def extreme_tokens(M, Kdim, rng):
    """Q8_K planes of M token rows: all +127, all -127, alternating +-127,
    then random quants in [-127, 127]; bsums are the sums of 16."""
    q = rng.integers(-127, 128, size=(M, Kdim)).astype(np.int8)
    q[0] = 127
    q[1] = -127
    q[2] = np.where(np.arange(Kdim) % 2 == 0, 127, -127)
    bs = q.astype(np.int32).reshape(M, Kdim // 16, 16).sum(axis=2).astype(np.int16)
    d8 = np.ones((M, Kdim // 256), np.float32)
    return d8, q, bs


def extreme_weights(fmt, N, Kdim, rng):
    """Superblocks with every field at its extreme: Q4_K/Q5_K quants at their
    maximum and 6-bit sub-scales and sub-mins at 63; Q6_K rows in three
    blocks of 128 (one weight tile each) with the largest |sub-scale| at
    most 32 / 33..62 / up to -128 and 127 (one accumulator unit per half,
    two, four with split planes), and a fourth block whose first half has
    small sub-scales and its second half -128 (1 + 4 units in a superblock).
    Q6_K quants alternate between rows at 0 (v = -32) and 63 (v = 31); row
    256 has every sub-scale at -128 (w' = 4096 everywhere)."""
    nsb = Kdim // 256
    blk = np.full((N, nsb, synth.BLOCK_BYTES[fmt]), 255, np.uint8)
    if fmt == synth.Q6_K:
        q = np.where((np.arange(N) % 2 == 0)[:, None, None], 0, 255).astype(np.uint8)
        blk[:, :, 0:192] = q                                     # ql, qh: q = 0 or 63
        sc = np.zeros((N, nsb, 16), np.int8)
        for n in range(N):
            tile = (n // 128) % 4
            if tile == 0:
                sc[n] = rng.choice([-32, 32, -31, 17], size=(nsb, 16))
            elif tile == 1:
                sc[n] = rng.choice([-62, 62, 33, -40], size=(nsb, 16))
            elif tile == 2:
                sc[n] = rng.choice([-128, 127, -100, 63], size=(nsb, 16))
            else:
                sc[n, :, :8] = rng.choice([-32, 32], size=(nsb, 8))
                sc[n, :, 8:] = -128
        if N > 257:
            sc[256] = -128                                       # q = 0: w' = 4096 throughout
            sc[257] = 127                                        # q = 63: w' = 3937
        blk[:, :, 192:208] = sc.view(np.uint8)
        blk[:, :, 208:210] = [0x00, 0x3C]                        # d = 1
    else:
        blk[:, :, 0:4] = [0x00, 0x3C, 0x00, 0x3C]                # d = dmin = 1
    return blk


def check_against_oracle_and_gemv(K, fmt, disk, planes, got_i, got_m):
    ref_i, ref_m = oracle.partials(fmt, disk, planes[1], planes[2])
    np.testing.assert_array_equal(got_i, ref_i)
    np.testing.assert_array_equal(got_m, ref_m)
    N, nsb, _ = disk.shape
    gv_i, gv_m = K.kq_debug_partials(fmt, pack(K, fmt, disk), N, nsb * 256, q8k_to_dev(K, planes))
    np.testing.assert_array_equal(got_i, gv_i.cpu().numpy())
    np.testing.assert_array_equal(got_m, gv_m.cpu().numpy())
    return ref_i


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("N,Kdim,M", [(200, 1280, 300), (128, 2560, 16), (33, 512, 129)])
def test_gemm_partials_bit_exact(K, fmt, N, Kdim, M):
    """Random superblocks and N(0,1) activations: several token tiles with a
    ragged tail, a ragged weight tile, and enough superblocks to run both
    parities of every ring."""
    rng = synth.rng_for(140, fmt * 1000 + N)
    disk = synth.disk_weights(fmt, N, Kdim, rng)
    planes = oracle_q8k(synth.activations(M, Kdim, rng))
    got_i, got_m = K.kq_debug_gemm_partials(fmt, pack(K, fmt, disk), N, Kdim, q8k_to_dev(K, planes))
    torch.cuda.synchronize()
    check_against_oracle_and_gemv(K, fmt, disk, planes, got_i.cpu().numpy(), got_m.cpu().numpy())


@pytest.mark.parametrize("fmt", FMTS)
def test_gemm_partials_worst_case_fields(K, fmt):
    """Every field at its extreme against tokens of +-127: the superblock sums
    reach 256*945*127 (Q4_K), 256*1953*127 (Q5_K) and 256*4096*127 (Q6_K),
    past 2^24, and still come out exact."""
    rng = synth.rng_for(141, fmt)
    N, Kdim, M = 512 if fmt == synth.Q6_K else 160, 768, 40
    disk = extreme_weights(fmt, N, Kdim, rng)
    planes = extreme_tokens(M, Kdim, rng)
    got_i, got_m = K.kq_debug_gemm_partials(fmt, pack(K, fmt, disk), N, Kdim, q8k_to_dev(K, planes))
    torch.cuda.synchronize()
    ref_i = check_against_oracle_and_gemv(K, fmt, disk, planes, got_i.cpu().numpy(), got_m.cpu().numpy())
    assert np.abs(ref_i).max() > 2 ** 24                   # the case a single fp32 accumulator rounds
    top = {synth.Q4_K: 256 * 945 * 127, synth.Q5_K: 256 * 1953 * 127, synth.Q6_K: 256 * 4096 * 127}[fmt]
    assert np.abs(ref_i).max() == top


@pytest.mark.parametrize("fmt", FMTS)
def test_gemm_outputs_at_worst_case_fields(K, fmt):
    """The production epilogue on the same extreme inputs: every output within
    the tolerance of the oracle (the float fold sees the exact units)."""
    from gpu_util import assert_row_tol
    rng = synth.rng_for(142, fmt)
    N, Kdim, M = 512 if fmt == synth.Q6_K else 160, 768, 40
    disk = extreme_weights(fmt, N, Kdim, rng)
    planes = extreme_tokens(M, Kdim, rng)
    y = K.kq_gemm(fmt, pack(K, fmt, disk), N, Kdim, q8k_to_dev(K, planes))
    torch.cuda.synchronize()
    assert_row_tol(y.cpu().numpy(), oracle.gemm(fmt, disk, *planes))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("counts", [[5, 0, 17, 1, 0, 140], [0, 300, 0, 129]])
def test_grouped_gemm_partials_bit_exact(K, fmt, counts):
    """The grouped (MoE) kernel: uneven and empty experts, experts of more
    than one token tile; every row's partials against the oracle's with its
    expert's weights."""
    rng = synth.rng_for(143, fmt * 100 + len(counts))
    E, N, Kdim = len(counts), 200, 512
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    disks = [synth.disk_weights(fmt, N, Kdim, rng) for _ in range(E)]
    M = int(offsets[-1])
    planes = oracle_q8k(synth.activations(M, Kdim, rng))
    per = K.kq_repack_bytes(fmt, N, Kdim)
    packed = torch.empty(per * E, dtype=torch.uint8, device="cuda")
    for e in range(E):
        K.kq_repack(fmt, to_dev(disks[e].reshape(-1)), N, Kdim, packed=packed[e * per:(e + 1) * per])
    got_i, got_m = K.kq_debug_gemm_partials(fmt, packed, N, Kdim, q8k_to_dev(K, planes), E=E,
                                            row_offsets=to_dev(offsets))
    torch.cuda.synchronize()
    got_i, got_m = got_i.cpu().numpy(), got_m.cpu().numpy()
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        if a == b:
            continue
        ref_i, ref_m = oracle.partials(fmt, disks[e], planes[1][a:b], planes[2][a:b])
        np.testing.assert_array_equal(got_i[a:b], ref_i)
        np.testing.assert_array_equal(got_m[a:b], ref_m)


def _bounds_plane(fmt, N, Kdim, image: np.ndarray) -> np.ndarray:
    """The bounds plane of a packed image, uint32 [row groups, K/256, 2],
    located by the image layout documented in kq.h (data planes of 128 /
    16 | 32 / 16 | 64 / 16 / 2 bytes per row and superblock, each padded to
    256 bytes, then the bounds plane)."""
    units = {synth.Q4_K: [128, 16], synth.Q5_K: [128, 32, 16], synth.Q6_K: [128, 64, 16, 2]}[fmt]
    groups, nsb = -(-N // 16), Kdim // 256
    off = 0
    for u in units:
        off += -(-(groups * 16 * nsb * u) // 256) * 256
    return image[off:off + groups * nsb * 8].view(np.uint32).reshape(groups, nsb, 2)


@pytest.mark.parametrize("fmt", FMTS)
def test_repack_bounds_plane(K, fmt):
    """The W1 bounds the repack derives: per row group and superblock half,
    the largest sum over the group's rows of |sub-scale| * |q| (Q6_K q - 32),
    from the oracle's decode of the disk bytes.  N = 40 leaves a padded group
    whose zero rows must not raise the bound."""
    rng = synth.rng_for(144, fmt)
    N, Kdim = 40, 768
    disk = synth.disk_weights(fmt, N, Kdim, rng)
    disk[3, 1] = extreme_weights(fmt, 1, 256, rng)[0, 0]      # one extreme superblock
    image = pack(K, fmt, disk).cpu().numpy()
    got = _bounds_plane(fmt, N, Kdim, image)
    want = np.zeros_like(got)
    per_sub = 16 if fmt == synth.Q6_K else 32
    for n in range(N):
        for s in range(Kdim // 256):
            dec = oracle.decode(fmt, disk[n, s])
            q = dec["q"].astype(np.int64) - (32 if fmt == synth.Q6_K else 0)
            w = np.abs(np.repeat(dec["sc"].astype(np.int64), per_sub)) * np.abs(q)
            for h in range(2):
                want[n // 16, s, h] = max(want[n // 16, s, h], w[128 * h:128 * (h + 1)].sum())
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("fmt", [synth.Q4_K, synth.Q6_K])
@pytest.mark.parametrize("M", [8, 5])
def test_batch_mma_partials_bit_exact(K, fmt, M):
    """The 8-token passes' integer warp-MMA fold: int32 partials per (token,
    row, superblock) equal the oracle's and the GEMV's, on random fields and
    on every field at its extreme (a ragged row group, fewer tokens than 8)."""
    rng = synth.rng_for(145, fmt * 10 + M)
    N, Kdim = 200, 768
    disk = synth.disk_weights(fmt, N, Kdim, rng)
    disk[16:48] = extreme_weights(fmt, 32, Kdim, rng)
    for planes in (oracle_q8k(synth.activations(M, Kdim, rng)), extreme_tokens(max(M, 3), Kdim, rng)):
        planes = tuple(p_[:M] for p_ in planes)
        got_i, got_m = K.kq_debug_batch_partials(fmt, pack(K, fmt, disk), N, Kdim, q8k_to_dev(K, planes))
        torch.cuda.synchronize()
        check_against_oracle_and_gemv(K, fmt, disk, planes, got_i.cpu().numpy(), got_m.cpu().numpy())
