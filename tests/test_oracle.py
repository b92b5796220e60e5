"""Pins for the CPU oracle: closed forms, brute force and invariants.

Everything here runs on the CPU (``-m "not gpu"``).  The oracle is checked
against values that do not come from the oracle:

* hand-built superblocks with closed-form results (tests/golden), which pin
  the block decoders (element order, 6-bit scale packing, Q5_K high bit,
  Q6_K 2-bit highs and signed sub-scales) and the integer fold (sub-scale
  term, min term and its sign, Q6_K's -32 offset via bsums);
* Q8_K cases whose rounding is fixed by IEEE fp32 arithmetic;
* a float64 dequantize-then-dot brute force, written per element, which
  the fold (written per sub-block, with bsums) must equal;
* invariants of Q8_K quantization on random data.
"""
import numpy as np
import pytest

import oracle
from quantized_gemv_gemm_gb300 import synth

from golden_util import FMT, act_planes, block_bytes, fill_array, load

GOLD = load()


@pytest.mark.parametrize("case", GOLD["cases"], ids=[c["name"] for c in GOLD["cases"]])
def test_closed_form_superblock(case):
    fmt = FMT[case["fmt"]]
    blk = block_bytes(case["fmt"], case["block"])
    d8, q8, bs = act_planes(case["act"])
    isum, msum = oracle.partials(fmt, blk[None, None, :], q8, bs)
    assert int(isum[0, 0, 0]) == case["isum"]
    assert int(msum[0, 0, 0]) == case["msum"]
    y = oracle.gemm(fmt, blk[None, None, :], d8, q8, bs)
    assert y[0, 0] == case["y"]
    # the dequantize-then-dot brute force must give the same closed form
    assert oracle.bruteforce_dot(fmt, blk[None, :], d8[0], q8[0]) == pytest.approx(case["y"], abs=1e-9)


@pytest.mark.parametrize("case", GOLD["q8k_cases"], ids=[c["name"] for c in GOLD["q8k_cases"]])
def test_q8k_closed_form(case):
    x = fill_array(case["x"], 256, np.float32)[None, :]
    d8, q8, bs = oracle.quantize_q8k(x)
    if "d8_expr" in case:
        expect_d8 = np.float32(50) / np.float32(127)
    else:
        expect_d8 = np.float32(case["d8"])
    assert d8[0, 0] == expect_d8
    np.testing.assert_array_equal(q8[0], fill_array(case["q8"], 256, np.int8))
    np.testing.assert_array_equal(bs[0], fill_array(case["bsums"], 16, np.int16))


def test_q8k_invariants_random():
    rng = np.random.default_rng(123)
    x = rng.standard_normal((7, 1024)).astype(np.float32)
    x[3, 256:512] = 0.0                      # an all-zero block
    x[5] *= np.float32(1e-30)                 # tiny magnitudes
    x[6, :8] = np.float32(1e4)                # outliers
    d8, q8, bs = oracle.quantize_q8k(x)
    M, K = x.shape
    xb = x.reshape(M, K // 256, 256).astype(np.float64)
    qb = q8.reshape(M, K // 256, 256).astype(np.int64)
    assert q8.min() >= -127 and q8.max() <= 127
    # bsums are the per-16 sums of q
    np.testing.assert_array_equal(bs.astype(np.int64), qb.reshape(M, -1, 16).sum(-1).reshape(M, -1))
    for m in range(M):
        for s in range(K // 256):
            amax = np.abs(xb[m, s]).max()
            if amax == 0:
                assert d8[m, s] == 0 and not qb[m, s].any()
                continue
            # the largest element lands on +-127, with its sign
            j = int(np.abs(xb[m, s]).argmax())
            assert qb[m, s, j] == 127 * np.sign(xb[m, s, j])
            # round-to-nearest: |x - d8*q| <= d8/2 (plus fp32 slack)
            err = np.abs(xb[m, s] - np.float64(d8[m, s]) * qb[m, s])
            assert err.max() <= 0.5 * d8[m, s] * (1 + 1e-5) + 1e-30
            assert d8[m, s] == np.float32(np.float32(amax) / np.float32(127.0))


@pytest.mark.parametrize("fmt", [synth.Q4_K, synth.Q5_K, synth.Q6_K])
@pytest.mark.parametrize("K", [256, 512, 1024])
def test_fold_matches_fp64_bruteforce(fmt, K):
    rng = np.random.default_rng([7, fmt, K])
    N, M = 8, 3
    disk = synth.disk_weights(fmt, N, K, rng)
    x = synth.activations(M, K, rng)
    d8, q8, bs = oracle.quantize_q8k(x)
    Y = oracle.gemm(fmt, disk, d8, q8, bs)
    for m in range(M):
        for n in range(N):
            ref = oracle.bruteforce_dot(fmt, disk[n], d8[m], q8[m])
            w = oracle.dequant(fmt, disk[n:n + 1])[0]
            a = np.repeat(d8[m].astype(np.float64), 256) * q8[m]
            scale = np.abs(w * a).sum()
            assert abs(Y[m, n] - ref) <= 1e-12 * scale
    # partials fold back into the same outputs
    isum, msum = oracle.partials(fmt, disk, q8, bs)
    dd = np.array([[oracle.decode(fmt, disk[n, s])["d"] for s in range(K // 256)] for n in range(N)])
    dm = np.array([[oracle.decode(fmt, disk[n, s])["dmin"] for s in range(K // 256)] for n in range(N)])
    Yp = (dd[None] * d8[:, None, :] * isum - dm[None] * d8[:, None, :] * msum).sum(-1)
    np.testing.assert_allclose(Yp, Y, rtol=1e-12, atol=1e-12 * np.abs(Y).max())


@pytest.mark.parametrize("fmt", [synth.Q4_K, synth.Q5_K, synth.Q6_K])
def test_special_case_plain_int_dot(fmt):
    """All sub-scales 1, mins 0, d = 1, d8 = 1: the fold reduces to the plain
    integer dot of the stored quants (minus 32 for Q6_K) with q8."""
    rng = np.random.default_rng([11, fmt])
    disk = synth.disk_weights(fmt, 1, 256, rng)
    blk = disk[0, 0]
    if fmt in (synth.Q4_K, synth.Q5_K):
        blk[0:2] = [0x00, 0x3C]
        blk[2:4] = 0
        blk[4:16] = [1, 1, 1, 1, 0, 0, 0, 0, 1, 1, 1, 1]
    else:
        blk[192:208] = 1
        blk[208:210] = [0x00, 0x3C]
    q = oracle.decode(fmt, blk)["q"].astype(np.int64)
    if fmt == synth.Q6_K:
        q = q - 32
    a = rng.integers(-127, 128, 256).astype(np.int8)
    bs = a.astype(np.int64).reshape(16, 16).sum(1).astype(np.int16)
    y = oracle.gemm(fmt, disk, np.ones((1, 1), np.float32), a[None], bs[None])
    assert y[0, 0] == float(int((q * a).sum()))


@pytest.mark.parametrize("fmt", [synth.Q4_K, synth.Q5_K, synth.Q6_K])
def test_exactness_bound_worst_case(fmt):
    """The page bounds |iacc| and |32 bacc| below 2^28; at the extremes of every
    field the int32 partials are still exact (compare with int64 sums)."""
    blk = np.full(synth.BLOCK_BYTES[fmt], 255, np.uint8)
    if fmt == synth.Q6_K:
        blk[192:208] = np.array([-128] * 16, np.int8).view(np.uint8)
        blk[208:210] = [0x00, 0x3C]
    else:
        blk[0:4] = [0x00, 0x3C, 0x00, 0x3C]
    a = np.full(256, -127, np.int8)
    bs = np.full(16, -127 * 16, np.int16)
    isum, msum = oracle.partials(fmt, blk[None, None], a[None], bs[None])
    dec = oracle.decode(fmt, blk)
    q = dec["q"].astype(np.int64)
    if fmt == synth.Q6_K:
        sc = np.repeat(dec["sc"].astype(np.int64), 16)
        assert int(isum[0, 0, 0]) == int((sc * (q - 32) * a).sum())
        assert abs(int((sc * q * a).sum())) < 2 ** 28
    else:
        sc = np.repeat(dec["sc"].astype(np.int64), 32)
        mn = np.repeat(dec["m"].astype(np.int64), 32)
        assert int(isum[0, 0, 0]) == int((sc * q * a).sum())
        assert int(msum[0, 0, 0]) == int((mn * a).sum())


def test_gemm_index_selection_and_rows():
    """Selecting tokens / rows returns the same values as the full product, and
    each row of a multi-row problem equals that row computed alone (the
    multi-row stride gate of the page's 'test_kq_gemv_rows')."""
    rng = np.random.default_rng(5)
    fmt, N, K, M = synth.Q4_K, 9, 768, 4
    disk = synth.disk_weights(fmt, N, K, rng)
    d8, q8, bs = oracle.quantize_q8k(synth.activations(M, K, rng))
    Y = oracle.gemm(fmt, disk, d8, q8, bs)
    ti, ni = np.array([3, 0]), np.array([8, 2, 5])
    np.testing.assert_array_equal(oracle.gemm(fmt, disk, d8, q8, bs, ti, ni), Y[np.ix_(ti, ni)])
    for n in range(N):
        single = oracle.gemm(fmt, disk[n:n + 1], d8, q8, bs)
        np.testing.assert_array_equal(single[:, 0], Y[:, n])


def test_oracle_rejects_bad_arguments():
    disk = np.zeros((1, 1, 144), np.uint8)
    with pytest.raises(ValueError):
        oracle.gemm(synth.Q4_K, disk, np.zeros((1, 1), np.float32), np.zeros((1, 256), np.int8),
                    np.zeros((1, 16), np.int16), tok_idx=np.array([2]))
    assert oracle.lib().ko_block_bytes(9) == 0
    assert oracle.lib().ko_decode(9, None, None, None, None, None, None) == -1


# ---------------------------------------------------------------- Q8_0 rail
def _q8_0_row(d_bits, quants):
    """One Q8_0 row [nb, 34] from fp16 bit patterns [nb] and int quants [nb, 32]."""
    quants = np.asarray(quants, np.int64).reshape(len(d_bits), 32)
    row = np.zeros((len(d_bits), 34), np.uint8)
    for b, h in enumerate(d_bits):
        row[b, 0], row[b, 1] = h & 0xFF, h >> 8
        row[b, 2:] = quants[b].astype(np.int8).view(np.uint8)
    return row


def test_q8_0_quantize_closed_forms():
    """Q8_0 activations: zero block, ties to even at iscale = 1 (amax 127),
    the extreme value mapped to +-127, one scale per 32 values."""
    x = np.zeros((1, 64), np.float32)
    x[0, 32:36] = [127.0, 2.5, 3.5, -2.5]
    x[0, 36] = -0.5
    d, q = oracle.quantize_q8_0(x)
    assert d[0, 0] == 0.0 and not q[0, :32].any()
    assert d[0, 1] == np.float32(1.0)
    assert q[0, 32:37].tolist() == [127, 2, 4, -2, 0]
    x2 = np.full((1, 32), -3.0, np.float32)
    d2, q2 = oracle.quantize_q8_0(x2)
    assert q2[0].tolist() == [-127] * 32 and d2[0, 0] == np.float32(3.0) / np.float32(127.0)


def test_q8_0_quantize_invariants_random():
    rng = synth.rng_for(900, 1)
    x = synth.activations(3, 512, rng, outliers=True)
    d, q = oracle.quantize_q8_0(x)
    xb = x.reshape(3, -1, 32).astype(np.float64)
    db = d.astype(np.float64)[..., None]
    assert np.all(np.abs(q.reshape(3, -1, 32)).max(axis=2) == 127)
    assert np.all(np.abs(xb - db * q.reshape(3, -1, 32)) <= db / 2 * (1 + 1e-6))


def test_q8_0_gemv_closed_forms():
    K = 256
    x = np.ones((1, K), np.float32)
    d_a, q_a = oracle.quantize_q8_0(x)               # q = 127, d = fl32(1/127)
    one = 0x3C00                                      # fp16 1.0
    rows = np.stack([
        _q8_0_row([one] * 8, np.ones(K)),                              # all ones
        _q8_0_row([one] * 8, np.tile([1, -1], K // 2)),                # cancels exactly
        _q8_0_row([0] * 3 + [0x4000] + [0] * 4, np.arange(K) % 7 - 3),  # only block 3, d = 2
    ])
    y = oracle.gemv_q8_0(rows, d_a, q_a)[0]
    inv = float(np.float32(1.0) / np.float32(127.0))
    assert y[0] == pytest.approx(K * 127 * inv, rel=1e-15)
    assert y[1] == 0.0
    blk3 = (np.arange(K) % 7 - 3)[96:128]
    assert y[2] == pytest.approx(2.0 * inv * 127 * blk3.sum(), rel=1e-15)


@pytest.mark.parametrize("K", [32, 256, 1024])
def test_q8_0_fold_matches_fp64_bruteforce(K):
    rng = synth.rng_for(900, K)
    disk = synth.disk_weights_q8_0(5, K, rng)
    d_a, q_a = oracle.quantize_q8_0(synth.activations(2, K, rng, outliers=True))
    Y = oracle.gemv_q8_0(disk, d_a, q_a)
    for m in range(2):
        for n in range(5):
            bf = oracle.bruteforce_q8_0(disk[n], d_a[m], q_a[m])
            assert Y[m, n] == pytest.approx(bf, rel=1e-12, abs=1e-12)
    # a permuted weight block must change the result (pins the element order)
    d2 = disk.copy()
    d2[0, 0, 2:] = disk[0, 0, 2:][::-1]
    assert oracle.gemv_q8_0(d2, d_a, q_a)[0, 0] != Y[0, 0]


def test_q8_0_partials_closed_forms():
    """Per-block int32 dots of the Q8_0 product: all ones against +127 tokens
    gives 32 * 127 per block; alternating signs cancel to 0; the extremes
    (+127 weights, -127 tokens) give -32 * 127 * 127; a weight nonzero in
    one block only contributes to that block; each token row is its own."""
    K = 256
    one = 0x3C00
    rows = np.stack([
        _q8_0_row([one] * 8, np.ones(K)),
        _q8_0_row([one] * 8, np.tile([1, -1], K // 2)),
        _q8_0_row([one] * 8, np.full(K, 127)),
        _q8_0_row([one] * 8, np.where(np.arange(K) // 32 == 5, np.arange(K) % 32 - 16, 0)),
    ])
    q_a = np.stack([np.full(K, 127), np.full(K, -127), np.tile([3, 3], K // 2)]).astype(np.int8)
    p = oracle.partials_q8_0(rows, q_a)
    assert p.shape == (3, 4, 8)
    assert (p[0, 0] == 32 * 127).all() and (p[1, 0] == -32 * 127).all()
    assert (p[:, 1] == 0).all()
    assert (p[1, 2] == -32 * 127 * 127).all()
    want5 = int((np.arange(32) - 16).sum()) * 3
    assert p[2, 3, 5] == want5 and (np.delete(p[2, 3], 5) == 0).all()


@pytest.mark.parametrize("M,K", [(3, 256), (4, 1024)])
def test_q8_0_gemm_rows_from_partials_and_bruteforce(M, K):
    """The M-row product: each output equals the fp64 brute force of its own
    row, and folding the per-block partials by d_w * d_a reproduces it."""
    rng = synth.rng_for(901, M * K)
    disk = synth.disk_weights_q8_0(6, K, rng)
    d_a, q_a = oracle.quantize_q8_0(synth.activations(M, K, rng, outliers=True))
    Y = oracle.gemm_q8_0(disk, d_a, q_a)
    P = oracle.partials_q8_0(disk, q_a)
    d_w = disk[:, :, :2].copy().view(np.float16)[..., 0].astype(np.float64)
    for m in range(M):
        for n in range(6):
            assert Y[m, n] == pytest.approx(oracle.bruteforce_q8_0(disk[n], d_a[m], q_a[m]), rel=1e-12, abs=1e-12)
            fold = float((d_w[n] * d_a[m].astype(np.float64) * P[m, n]).sum())
            assert Y[m, n] == pytest.approx(fold, rel=1e-12, abs=1e-12)
