"""Helpers of the GPU parity tests: upload inputs, compare with the oracle."""
import numpy as np
import torch

import oracle
from quantized_gemv_gemm_gb300 import synth


def kq():
    from quantized_gemv_gemm_gb300 import build
    build.build()
    from quantized_gemv_gemm_gb300 import kq as mod
    return mod


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def pack(K, fmt, disk: np.ndarray):
    """Repack disk superblocks on the device; returns (packed, N, K)."""
    N = disk.shape[0]
    return K.kq_repack(fmt, to_dev(disk.reshape(-1)), N, disk.shape[1] * 256)


def oracle_q8k(x: np.ndarray):
    return oracle.quantize_q8k(x)


def q8k_to_dev(K, planes):
    d8, q8, bs = planes
    return K.Q8K(to_dev(d8), to_dev(q8), to_dev(bs))


def assert_row_tol(y_gpu: np.ndarray, y_ref: np.ndarray, rel: float = 1e-3, row_max=None):
    """|err| <= rel * max|row output| per token row (the fixture-magnitude
    tolerance: Q6_K's signed sub-scales cancel within a row, so element-wise
    relative error is meaningless)."""
    y_gpu = np.atleast_2d(y_gpu).astype(np.float64)
    y_ref = np.atleast_2d(y_ref)
    assert y_gpu.shape == y_ref.shape
    assert np.isfinite(y_gpu).all(), "non-finite output"
    scale = np.abs(y_ref).max(axis=1, keepdims=True) if row_max is None else np.atleast_2d(row_max).T
    err = np.abs(y_gpu - y_ref)
    bad = err > rel * scale
    if bad.any():
        i, j = np.argwhere(bad)[0]
        raise AssertionError(f"{bad.sum()} outputs off; first at {i},{j}: gpu {y_gpu[i, j]} ref {y_ref[i, j]} "
                             f"tol {rel * scale[i, 0]}; max err/scale {float((err / scale).max()):.3e}")
    with np.errstate(divide="ignore", invalid="ignore"):
        return float(np.nanmax(np.where(scale > 0, err / np.where(scale > 0, scale, 1.0), 0.0)))


def poisoned(shape, guard=64):
    """Output buffer with NaN poison and a NaN guard band after it."""
    n = int(np.prod(shape))
    full = torch.full((n + guard,), float("nan"), dtype=torch.float32, device="cuda")
    return full, full[:n].view(*shape)


def check_guard(full: torch.Tensor, n: int):
    tail = full[n:].cpu().numpy()
    assert np.isnan(tail).all(), "guard band after the output was written"
