"""Scalar CPU oracle for the K-quant x Q8_K products (TEST INFRASTRUCTURE).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's
``cpu_baseline`` / reference leg may import this package.  The product path
(``quantized_gemv_gemm_gb300``) never imports it and has no CPU fallback.

The arithmetic lives in ``kq_oracle.c`` (plain C, built with gcc,
``-ffp-contract=off``, no fast-math).  This module compiles it on first use
and marshals numpy arrays through ctypes; it holds none of the method.

Method source, cited as [kq-arc]: the page "dasLLAMA: K-quant kernel arc -
kq v2 integer folds, kq v3 panel-scratch tiles, chain regrain, parity gates"
(daScript #3450), section "The pieces" and the kq-v2 commit messages.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

Q4_K, Q5_K, Q6_K = 1, 2, 3
BLOCK_BYTES = {Q4_K: 144, Q5_K: 176, Q6_K: 210}
QK = 256

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kq_oracle.c")
_HDR = os.path.join(_HERE, "kq_oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libkq_oracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, OpenMP if available)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    newest_src = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= newest_src:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", "-frounding-math", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            P = ctypes.c_void_p
            i64 = ctypes.c_int64
            i32 = ctypes.c_int
            L.ko_block_bytes.argtypes = [i32]
            L.ko_decode.argtypes = [i32, P, P, P, P, P, P]
            L.ko_dequant.argtypes = [i32, P, P]
            L.ko_quantize_q8k.argtypes = [P, i64, i64, P, P, P]
            L.ko_quantize_q8k.restype = None
            L.ko_partials_block.argtypes = [i32, P, P, P, P, P]
            L.ko_partials_block.restype = None
            L.ko_partials.argtypes = [i32, P, i64, i64, P, P, i64, P, P]
            L.ko_dot.argtypes = [i32, P, i64, P, P, P]
            L.ko_dot.restype = ctypes.c_double
            L.ko_gemm.argtypes = [i32, P, i64, i64, P, P, P, i64, P, i64, P, i64, P]
            L.ko_bruteforce_dot.argtypes = [i32, P, i64, P, P]
            L.ko_bruteforce_dot.restype = ctypes.c_double
            L.ko_quantize_q8_0.argtypes = [P, i64, i64, P, P]
            L.ko_quantize_q8_0.restype = None
            L.ko_gemv_q8_0.argtypes = [P, i64, i64, P, P, i64, P]
            L.ko_partials_q8_0.argtypes = [P, i64, i64, P, i64, P]
            L.ko_bruteforce_q8_0.argtypes = [P, i64, P, P]
            L.ko_bruteforce_q8_0.restype = ctypes.c_double
            L.ko_num_threads.argtypes = []
            L.ko_set_num_threads.argtypes = [i32]
            L.ko_set_num_threads.restype = None
            _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return lib().ko_num_threads()


def set_num_threads(n: int) -> None:
    lib().ko_set_num_threads(int(n))


def decode(fmt: int, blk: np.ndarray) -> dict:
    """Decode one disk superblock (uint8[bytes]) into its fields."""
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    assert blk.size == BLOCK_BYTES[fmt]
    d = np.zeros(1, np.float64)
    dmin = np.zeros(1, np.float64)
    sc = np.zeros(16, np.int32)
    mn = np.zeros(8, np.int32)
    q = np.zeros(QK, np.int32)
    nsub = lib().ko_decode(fmt, _p(blk), _p(d), _p(dmin), _p(sc), _p(mn), _p(q))
    if nsub < 0:
        raise ValueError("unknown format")
    return {"d": float(d[0]), "dmin": float(dmin[0]), "sc": sc[:nsub].copy(),
            "m": mn.copy(), "q": q}


def dequant(fmt: int, disk: np.ndarray) -> np.ndarray:
    """Dequantize disk weights [N, K/256, bytes] to float64 [N, K]."""
    disk = np.ascontiguousarray(disk, dtype=np.uint8)
    N, nsb, bb = disk.shape
    assert bb == BLOCK_BYTES[fmt]
    out = np.zeros((N, nsb * QK), np.float64)
    L = lib()
    for n in range(N):
        for s in range(nsb):
            w = np.zeros(QK, np.float64)
            L.ko_dequant(fmt, _p(np.ascontiguousarray(disk[n, s])), _p(w))
            out[n, s * QK:(s + 1) * QK] = w
    return out


def quantize_q8k(x: np.ndarray):
    """Q8_K of float32 [M, K] -> (d8 f32 [M, K/256], q8 i8 [M, K], bsums i16 [M, K/16])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim == 1:
        x = x[None, :]
    M, K = x.shape
    assert K % QK == 0
    d8 = np.zeros((M, K // QK), np.float32)
    q8 = np.zeros((M, K), np.int8)
    bs = np.zeros((M, K // 16), np.int16)
    lib().ko_quantize_q8k(_p(x), M, K, _p(d8), _p(q8), _p(bs))
    return d8, q8, bs


def partials(fmt: int, disk: np.ndarray, q8: np.ndarray, bs: np.ndarray):
    """int32 (isum, msum), each [M, N, K/256]."""
    disk = np.ascontiguousarray(disk, dtype=np.uint8)
    q8 = np.ascontiguousarray(q8, dtype=np.int8)
    bs = np.ascontiguousarray(bs, dtype=np.int16)
    N, nsb, _ = disk.shape
    M, K = q8.shape
    assert K == nsb * QK
    isum = np.zeros((M, N, nsb), np.int32)
    msum = np.zeros((M, N, nsb), np.int32)
    rc = lib().ko_partials(fmt, _p(disk), N, K, _p(q8), _p(bs), M, _p(isum), _p(msum))
    if rc:
        raise ValueError("ko_partials rejected its arguments")
    return isum, msum


def gemm(fmt: int, disk: np.ndarray, d8: np.ndarray, q8: np.ndarray, bs: np.ndarray,
         tok_idx=None, n_idx=None) -> np.ndarray:
    """Y[tokens, rows] in float64 for the selected tokens / weight rows."""
    disk = np.ascontiguousarray(disk, dtype=np.uint8)
    d8 = np.ascontiguousarray(d8, dtype=np.float32)
    q8 = np.ascontiguousarray(q8, dtype=np.int8)
    bs = np.ascontiguousarray(bs, dtype=np.int16)
    N, nsb, _ = disk.shape
    M, K = q8.shape
    assert K == nsb * QK
    ti = None if tok_idx is None else np.ascontiguousarray(tok_idx, dtype=np.int64)
    ni = None if n_idx is None else np.ascontiguousarray(n_idx, dtype=np.int64)
    ntok = M if ti is None else ti.size
    nn = N if ni is None else ni.size
    Y = np.zeros((ntok, nn), np.float64)
    rc = lib().ko_gemm(fmt, _p(disk), N, K, _p(d8), _p(q8), _p(bs), M,
                       None if ti is None else _p(ti), ntok,
                       None if ni is None else _p(ni), nn, _p(Y))
    if rc:
        raise ValueError("ko_gemm rejected its arguments")
    return Y


def bruteforce_dot(fmt: int, row: np.ndarray, d8: np.ndarray, q8: np.ndarray) -> float:
    """Dequantize-then-dot in double for one weight row [K/256, bytes] and one token."""
    row = np.ascontiguousarray(row, dtype=np.uint8)
    d8 = np.ascontiguousarray(d8, dtype=np.float32)
    q8 = np.ascontiguousarray(q8, dtype=np.int8)
    return lib().ko_bruteforce_dot(fmt, _p(row), row.shape[0], _p(d8), _p(q8))


# ---- Q8_0 (the q8 rail: Q8_0 weights x Q8_0-form activations, blocks of 32)
Q8_0 = 4
Q8_0_BLOCK = 34
QK8_0 = 32


def quantize_q8_0(x: np.ndarray):
    """Q8_0 activations of float32 [M, K] -> (d f32 [M, K/32], q i8 [M, K])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim == 1:
        x = x[None, :]
    M, K = x.shape
    assert K % QK8_0 == 0
    d = np.zeros((M, K // QK8_0), np.float32)
    q = np.zeros((M, K), np.int8)
    lib().ko_quantize_q8_0(_p(x), M, K, _p(d), _p(q))
    return d, q


def partials_q8_0(disk: np.ndarray, q_a: np.ndarray) -> np.ndarray:
    """int32 per-block dots [M, N, K/32] of disk Q8_0 weights [N, K/32, 34] and M activation rows."""
    disk = np.ascontiguousarray(disk, dtype=np.uint8)
    q_a = np.ascontiguousarray(np.atleast_2d(q_a), dtype=np.int8)
    N, nb, bb = disk.shape
    assert bb == Q8_0_BLOCK
    M, K = q_a.shape
    assert K == nb * QK8_0
    isum = np.zeros((M, N, nb), np.int32)
    if lib().ko_partials_q8_0(_p(disk), N, K, _p(q_a), M, _p(isum)):
        raise ValueError("ko_partials_q8_0 rejected its arguments")
    return isum


def gemm_q8_0(disk: np.ndarray, d_a: np.ndarray, q_a: np.ndarray) -> np.ndarray:
    """Y[M, N] in float64: the Q8_0 product for M activation rows (the same
    definition as gemv_q8_0, which takes any number of rows)."""
    return gemv_q8_0(disk, d_a, q_a)


def gemv_q8_0(disk: np.ndarray, d_a: np.ndarray, q_a: np.ndarray) -> np.ndarray:
    """Y[M, N] in float64 for disk Q8_0 weights [N, K/32, 34] and M activation rows."""
    disk = np.ascontiguousarray(disk, dtype=np.uint8)
    d_a = np.ascontiguousarray(d_a, dtype=np.float32)
    q_a = np.ascontiguousarray(q_a, dtype=np.int8)
    N, nb, bb = disk.shape
    assert bb == Q8_0_BLOCK
    if q_a.ndim == 1:
        q_a, d_a = q_a[None, :], d_a[None, :]
    M, K = q_a.shape
    assert K == nb * QK8_0
    Y = np.zeros((M, N), np.float64)
    if lib().ko_gemv_q8_0(_p(disk), N, K, _p(d_a), _p(q_a), M, _p(Y)):
        raise ValueError("ko_gemv_q8_0 rejected its arguments")
    return Y


def bruteforce_q8_0(row: np.ndarray, d_a: np.ndarray, q_a: np.ndarray) -> float:
    """Dequantize-then-dot in double for one Q8_0 row [K/32, 34] and one activation row."""
    row = np.ascontiguousarray(row, dtype=np.uint8)
    d_a = np.ascontiguousarray(d_a, dtype=np.float32)
    q_a = np.ascontiguousarray(q_a, dtype=np.int8)
    return lib().ko_bruteforce_q8_0(_p(row), row.shape[0], _p(d_a), _p(q_a))
