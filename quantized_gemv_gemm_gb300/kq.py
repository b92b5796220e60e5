"""Thin ctypes binding of libkq.so (include/kq.h), with the same names.

Argument marshalling only: torch tensors provide device memory and the
current CUDA stream; every step of the computation runs in libkq's CUDA
kernels.  Importing this module raises if libkq.so has not been built
(``python -m quantized_gemv_gemm_gb300.build``): there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import NamedTuple, Optional

import torch

Q4_K, Q5_K, Q6_K, Q8_0 = 1, 2, 3, 4
QK = 256

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkq.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(f"libkq.so is missing at {_LIB_PATH}: build it with "
                      "`python -m quantized_gemv_gemm_gb300.build` (no CPU fallback exists)")
_lib = ctypes.CDLL(_LIB_PATH)

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_INT = ctypes.c_int


class _Q8KConst(ctypes.Structure):
    _fields_ = [("d", _P), ("qs", _P), ("bsums", _P)]


_lib.kq_strerror.argtypes = [_INT]
_lib.kq_strerror.restype = ctypes.c_char_p
_lib.kq_block_bytes.argtypes = [_INT]
_lib.kq_block_bytes.restype = _SZ
_lib.kq_quantize_q8k.argtypes = [_P, _I64, _I64, _Q8KConst, _P]
_lib.kq_repack_bytes.argtypes = [_INT, _I64, _I64]
_lib.kq_repack_bytes.restype = _SZ
_lib.kq_repack.argtypes = [_INT, _P, _I64, _I64, _P, _P]
_lib.kq_gemv_workspace_bytes.argtypes = []
_lib.kq_gemv_workspace_bytes.restype = _SZ
_lib.kq_gemv.argtypes = [_INT, _P, _I64, _I64, _Q8KConst, _P, _P, _SZ, _P]
_lib.kq_gemv_fused.argtypes = [_INT, _INT, _P, _P, _I64, _P, _P, _P, _SZ, _P]
_lib.kq_gemv_fused_batch.argtypes = [_INT, _INT, _P, _P, _I64, _P, _I64, _P, _P, _SZ, _P]
_lib.kq_gemv_grouped_fused.argtypes = [_INT, _INT, _P, _P, _I64, _I64, _P, _P, _I64, _P, _P]
_lib.kq_gemm_workspace_bytes.argtypes = [_INT, _I64, _I64, _I64]
_lib.kq_gemm_workspace_bytes.restype = _SZ
_lib.kq_gemm_min_workspace_bytes.argtypes = [_INT, _I64, _I64, _I64]
_lib.kq_gemm_min_workspace_bytes.restype = _SZ
_lib.kq_gemm.argtypes = [_INT, _P, _I64, _I64, _Q8KConst, _I64, _P, _P, _SZ, _P]
_lib.kq_gemm_grouped.argtypes = [_INT, _P, _I64, _P, _I64, _I64, _Q8KConst, _I64, _P, _P, _SZ, _P]
_lib.kq_gemm_noalloc.argtypes = [_INT, _P, _I64, _I64, _Q8KConst, _I64, _P, _P]
_lib.kq_debug_partials.argtypes = [_INT, _P, _I64, _I64, _Q8KConst, _I64, _P, _P, _P]
_lib.kq_debug_batch_partials.argtypes = [_INT, _P, _I64, _I64, _Q8KConst, _I64, _P, _P, _P]
_lib.kq_debug_gemm_partials.argtypes = [_INT, _P, _I64, _P, _I64, _I64, _Q8KConst, _I64, _P, _P, _P, _SZ, _P]
_lib.kq_debug_decode.argtypes = [_INT, _P, _I64, _I64, _P, _P, _P, _P, _P, _P]
_lib.kq_device_status.argtypes = [_P]
_lib.kq_measure_mma_s8.argtypes = [_I64, _I64, _P, _P]
_lib.kq_copy_in.argtypes = [_P, _P, _SZ, _P]
_lib.kq_debug_wait_timeout.argtypes = [ctypes.c_uint64, _P]
_lib.kq_quantize_q8_0.argtypes = [_P, _I64, _I64, _P, _P, _P]
_lib.kq_gemv_q8_0.argtypes = [_P, _I64, _I64, _P, _P, _P, _P]
_lib.kq_gemm_q8_0.argtypes = [_P, _I64, _I64, _P, _P, _I64, _P, _P]
_lib.kq_gemv_q8_0_fused.argtypes = [_P, _I64, _I64, _P, _P, _P]
_lib.kq_set_launch_flags.argtypes = [ctypes.c_uint]
_lib.kq_set_launch_flags.restype = ctypes.c_uint
_lib.kq_get_launch_flags.argtypes = []
_lib.kq_get_launch_flags.restype = ctypes.c_uint
for _f in ("kq_quantize_q8k", "kq_repack", "kq_gemv", "kq_gemv_fused", "kq_gemv_fused_batch", "kq_gemm", "kq_gemm_grouped", "kq_gemm_noalloc",
           "kq_debug_partials", "kq_debug_gemm_partials", "kq_debug_batch_partials", "kq_debug_decode", "kq_device_status", "kq_measure_mma_s8",
           "kq_quantize_q8_0", "kq_gemv_q8_0", "kq_gemv_grouped_fused", "kq_debug_wait_timeout",
           "kq_gemv_q8_0_fused", "kq_copy_in", "kq_gemm_q8_0"):
    getattr(_lib, _f).restype = _INT

LIB_PATH = _LIB_PATH


class KQError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {kq_strerror(code)} ({code})")


class Q8K(NamedTuple):
    """Q8_K activation planes on the device."""
    d: torch.Tensor        # float32 [M, K/256]
    qs: torch.Tensor       # int8    [M, K]
    bsums: torch.Tensor    # int16   [M, K/16]


def kq_strerror(code: int) -> str:
    return _lib.kq_strerror(int(code)).decode()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream: Optional[torch.cuda.Stream] = None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc: int, where: str):
    if rc != 0:
        raise KQError(rc, where)


def _q8k_struct(a: Q8K) -> _Q8KConst:
    return _Q8KConst(a.d.data_ptr(), a.qs.data_ptr(), a.bsums.data_ptr())


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("libkq takes contiguous CUDA tensors")


def _need_out(*ts):
    """Outputs: contiguous CUDA tensors, or pinned host tensors (the kernel
    stores into the mapped host memory)."""
    for t in ts:
        if t is not None and (not t.is_contiguous() or not (t.is_cuda or (t.device.type == "cpu" and t.is_pinned()))):
            raise ValueError("libkq outputs are contiguous CUDA or pinned host tensors")


def kq_block_bytes(fmt: int) -> int:
    return int(_lib.kq_block_bytes(int(fmt)))


def q8k_empty(M: int, K: int, device="cuda") -> Q8K:
    return Q8K(torch.empty((M, K // QK), dtype=torch.float32, device=device),
               torch.empty((M, K), dtype=torch.int8, device=device),
               torch.empty((M, K // 16), dtype=torch.int16, device=device))


def kq_quantize_q8k(x: torch.Tensor, out: Optional[Q8K] = None, stream=None) -> Q8K:
    """Q8_K planes of float32 x [M, K] (or [K])."""
    if x.dim() == 1:
        x = x.view(1, -1)
    _need_cuda(x)
    if x.dtype != torch.float32:
        raise ValueError("x must be float32")
    M, K = x.shape
    if out is None:
        out = q8k_empty(M, K, x.device)
    _need_cuda(*out)
    _check(_lib.kq_quantize_q8k(_ptr(x), M, K, _q8k_struct(out), _stream(stream)), "kq_quantize_q8k")
    return out


def kq_repack_bytes(fmt: int, N: int, K: int) -> int:
    return int(_lib.kq_repack_bytes(int(fmt), int(N), int(K)))


def kq_repack(fmt: int, disk: torch.Tensor, N: int, K: int, packed: Optional[torch.Tensor] = None,
              stream=None) -> torch.Tensor:
    """Repack disk superblocks (uint8 device tensor, N*K/256*block_bytes bytes)."""
    _need_cuda(disk)
    nbytes = kq_repack_bytes(fmt, N, K)
    if packed is None:
        packed = torch.empty(nbytes, dtype=torch.uint8, device=disk.device)
    _need_cuda(packed)
    if packed.numel() < nbytes:
        raise ValueError("packed buffer too small")
    _check(_lib.kq_repack(int(fmt), _ptr(disk), N, K, _ptr(packed), _stream(stream)), "kq_repack")
    return packed


KQ_GEMV_WORKSPACE_BYTES = int(_lib.kq_gemv_workspace_bytes())
_gemv_ws: dict = {}


def gemv_workspace(device=None) -> torch.Tensor:
    """A zero-filled decode-GEMV workspace (KQ_GEMV_WORKSPACE_BYTES) for the
    device, allocated on first use and then shared by every kq_gemv /
    kq_gemv_fused call that passes none.  Calls that may run at the same time
    on different streams must each pass a workspace of their own."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    key = dev.index if dev.index is not None else torch.cuda.current_device()
    ws = _gemv_ws.get(key)
    if ws is None:
        ws = torch.zeros(KQ_GEMV_WORKSPACE_BYTES, dtype=torch.uint8, device=torch.device("cuda", key))
        _gemv_ws[key] = ws
    return ws


def _gemv_ws_args(workspace, device):
    """workspace=None: the device's shared one; False: none (whole row groups per block)."""
    if workspace is False:
        return None, 0
    if workspace is None:
        workspace = gemv_workspace(device)
    _need_cuda(workspace)
    return _ptr(workspace), workspace.numel() * workspace.element_size()


def kq_gemv(fmt: int, packed: torch.Tensor, N: int, K: int, a: Q8K, y: Optional[torch.Tensor] = None,
            workspace=None, stream=None) -> torch.Tensor:
    _need_cuda(packed, *a)
    if y is None:
        y = torch.empty(N, dtype=torch.float32, device=packed.device)
    _need_cuda(y)
    wp, wn = _gemv_ws_args(workspace, packed.device)
    _check(_lib.kq_gemv(int(fmt), _ptr(packed), N, K, _q8k_struct(a), _ptr(y), wp, wn, _stream(stream)), "kq_gemv")
    return y


def kq_gemv_fused(fmt: int, packed_list, N_list, K: int, x: torch.Tensor, y_list=None, workspace=None, stream=None):
    """Quantize the fp32 row x and multiply it by up to 4 matrices in one launch."""
    n = len(packed_list)
    _need_cuda(x, *packed_list)
    if x.dtype != torch.float32:
        raise ValueError("x must be float32")
    if y_list is None:
        y_list = [torch.empty(int(N), dtype=torch.float32, device=x.device) for N in N_list]
    _need_out(*y_list)
    pk = (ctypes.c_void_p * max(n, 1))(*[t.data_ptr() for t in packed_list])
    nn = (ctypes.c_int64 * max(n, 1))(*[int(v) for v in N_list])
    yy = (ctypes.c_void_p * max(n, 1))(*[t.data_ptr() for t in y_list])
    wp, wn = _gemv_ws_args(workspace, x.device)
    _check(_lib.kq_gemv_fused(int(fmt), n, pk, nn, int(K), _ptr(x), yy, wp, wn, _stream(stream)), "kq_gemv_fused")
    return y_list


def kq_gemv_fused_batch(fmt: int, packed_list, N_list, K: int, x: torch.Tensor, y_list=None, workspace=None,
                        stream=None):
    """Quantize the M fp32 rows of x [M, K] and multiply them by up to 4 matrices
    in one launch per pass of up to 8 rows; y_list[m] is [M, N_list[m]]."""
    n = len(packed_list)
    _need_cuda(x, *packed_list)
    if x.dtype != torch.float32 or x.dim() != 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous float32 [M, K] tensor")
    M = x.shape[0]
    if y_list is None:
        y_list = [torch.empty((M, int(N)), dtype=torch.float32, device=x.device) for N in N_list]
    _need_cuda(*y_list)
    pk = (ctypes.c_void_p * max(n, 1))(*[t.data_ptr() for t in packed_list])
    nn = (ctypes.c_int64 * max(n, 1))(*[int(v) for v in N_list])
    yy = (ctypes.c_void_p * max(n, 1))(*[t.data_ptr() for t in y_list])
    wp, wn = _gemv_ws_args(workspace, x.device)
    _check(_lib.kq_gemv_fused_batch(int(fmt), n, pk, nn, int(K), _ptr(x), int(M), yy, wp, wn, _stream(stream)),
           "kq_gemv_fused_batch")
    return y_list


def kq_gemv_grouped_fused(fmt: int, packed_list, N_list, K: int, E: int, row_offsets: torch.Tensor,
                          x: torch.Tensor, y_list=None, stream=None):
    """MoE decode: the M fp32 rows of x [M, K] (grouped by expert, row_offsets
    int32 [E+1]) quantized in the kernel and multiplied by their experts of
    every weight set in packed_list (E images each) in one launch."""
    n = len(packed_list)
    _need_cuda(x, row_offsets, *packed_list)
    if x.dtype != torch.float32 or x.dim() != 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous float32 [M, K] tensor")
    if row_offsets.dtype != torch.int32:
        raise ValueError("row_offsets must be int32")
    M = x.shape[0]
    if y_list is None:
        y_list = [torch.zeros((M, int(N)), dtype=torch.float32, device=x.device) for N in N_list]
    _need_cuda(*y_list)
    pk = (ctypes.c_void_p * max(n, 1))(*[t.data_ptr() for t in packed_list])
    nn = (ctypes.c_int64 * max(n, 1))(*[int(v) for v in N_list])
    yy = (ctypes.c_void_p * max(n, 1))(*[t.data_ptr() for t in y_list])
    _check(_lib.kq_gemv_grouped_fused(int(fmt), n, pk, nn, int(K), int(E), _ptr(row_offsets), _ptr(x), int(M), yy,
                                      _stream(stream)), "kq_gemv_grouped_fused")
    return y_list


def kq_gemm_workspace_bytes(fmt: int, M: int, N: int, K: int) -> int:
    return int(_lib.kq_gemm_workspace_bytes(int(fmt), int(M), int(N), int(K)))


def kq_gemm_min_workspace_bytes(fmt: int, M: int, N: int, K: int) -> int:
    return int(_lib.kq_gemm_min_workspace_bytes(int(fmt), int(M), int(N), int(K)))


def _workspace(fmt, M, N, K, workspace, device):
    need = kq_gemm_workspace_bytes(fmt, M, N, K)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    return workspace, (0 if workspace is None else workspace.numel())


def kq_gemm(fmt: int, packed: torch.Tensor, N: int, K: int, a: Q8K, y: Optional[torch.Tensor] = None,
            workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    _need_cuda(packed, *a)
    M = a.qs.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=packed.device)
    _need_cuda(y, workspace)
    workspace, ws_bytes = _workspace(fmt, M, N, K, workspace, packed.device)
    _check(_lib.kq_gemm(int(fmt), _ptr(packed), N, K, _q8k_struct(a), M, _ptr(y), _ptr(workspace), ws_bytes,
                        _stream(stream)), "kq_gemm")
    return y


def kq_gemm_grouped(fmt: int, packed: torch.Tensor, E: int, row_offsets: torch.Tensor, N: int, K: int,
                    a: Q8K, y: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                    stream=None) -> torch.Tensor:
    _need_cuda(packed, row_offsets, *a)
    if row_offsets.dtype != torch.int32:
        raise ValueError("row_offsets must be int32")
    M = a.qs.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=packed.device)
    _need_cuda(y, workspace)
    workspace, ws_bytes = _workspace(fmt, M, N, K, workspace, packed.device)
    _check(_lib.kq_gemm_grouped(int(fmt), _ptr(packed), E, _ptr(row_offsets), N, K, _q8k_struct(a), M, _ptr(y),
                                _ptr(workspace), ws_bytes, _stream(stream)), "kq_gemm_grouped")
    return y


KQ_NOALLOC_SCRATCH_BYTES = 32 << 20


def kq_gemm_noalloc(fmt: int, packed: torch.Tensor, N: int, K: int, a: Q8K, y: Optional[torch.Tensor] = None,
                    stream=None) -> torch.Tensor:
    """kq_gemm with the library's fixed scratch array instead of a workspace
    (for callers that cannot allocate device memory); y must be given by
    such callers, it is only allocated here when omitted."""
    _need_cuda(packed, *a)
    M = a.qs.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=packed.device)
    _need_cuda(y)
    _check(_lib.kq_gemm_noalloc(int(fmt), _ptr(packed), N, K, _q8k_struct(a), M, _ptr(y), _stream(stream)),
           "kq_gemm_noalloc")
    return y


def kq_debug_partials(fmt: int, packed: torch.Tensor, N: int, K: int, a: Q8K, stream=None):
    _need_cuda(packed, *a)
    M = a.qs.shape[0]
    isum = torch.zeros((M, N, K // QK), dtype=torch.int32, device=packed.device)
    msum = torch.zeros_like(isum)
    _check(_lib.kq_debug_partials(int(fmt), _ptr(packed), N, K, _q8k_struct(a), M, _ptr(isum), _ptr(msum),
                                  _stream(stream)), "kq_debug_partials")
    return isum, msum


def kq_debug_batch_partials(fmt: int, packed: torch.Tensor, N: int, K: int, a: Q8K, stream=None):
    """int32 (isum, msum) [M, N, K/256] from the 8-token passes' integer-MMA
    fold (Q4_K, Q6_K; M <= 8)."""
    _need_cuda(packed, *a)
    M = a.qs.shape[0]
    isum = torch.zeros((M, N, K // QK), dtype=torch.int32, device=packed.device)
    msum = torch.zeros_like(isum)
    _check(_lib.kq_debug_batch_partials(int(fmt), _ptr(packed), N, K, _q8k_struct(a), M, _ptr(isum), _ptr(msum),
                                        _stream(stream)), "kq_debug_batch_partials")
    return isum, msum


def kq_debug_gemm_partials(fmt: int, packed: torch.Tensor, N: int, K: int, a: Q8K, E: int = 1,
                           row_offsets: Optional[torch.Tensor] = None, stream=None):
    """int32 (isum, msum) [M, N, K/256] as the tensor-core GEMM (dense, or
    grouped with E experts and row_offsets) computes them; M >= 16."""
    _need_cuda(packed, *a)
    if row_offsets is not None:
        _need_cuda(row_offsets)
        if row_offsets.dtype != torch.int32:
            raise ValueError("row_offsets must be int32")
    M = a.qs.shape[0]
    isum = torch.zeros((M, N, K // QK), dtype=torch.int32, device=packed.device)
    msum = torch.zeros_like(isum)
    workspace, ws_bytes = _workspace(fmt, M, N, K, None, packed.device)
    _check(_lib.kq_debug_gemm_partials(int(fmt), _ptr(packed), E, _ptr(row_offsets), N, K, _q8k_struct(a), M,
                                       _ptr(isum), _ptr(msum), _ptr(workspace), ws_bytes, _stream(stream)),
           "kq_debug_gemm_partials")
    return isum, msum


def kq_debug_decode(fmt: int, packed: torch.Tensor, N: int, K: int, stream=None) -> dict:
    _need_cuda(packed)
    nsb = K // QK
    dev = packed.device
    q = torch.zeros((N, K), dtype=torch.int32, device=dev)
    sc = torch.zeros((N, nsb, 16), dtype=torch.int32, device=dev)
    mn = torch.zeros((N, nsb, 8), dtype=torch.int32, device=dev)
    d = torch.zeros((N, nsb), dtype=torch.float32, device=dev)
    dmin = torch.zeros((N, nsb), dtype=torch.float32, device=dev)
    _check(_lib.kq_debug_decode(int(fmt), _ptr(packed), N, K, _ptr(q), _ptr(sc), _ptr(mn), _ptr(d), _ptr(dmin),
                                _stream(stream)), "kq_debug_decode")
    return {"q": q, "sc": sc, "m": mn, "d": d, "dmin": dmin}


def kq_quantize_q8_0(x: torch.Tensor, d: Optional[torch.Tensor] = None, qs: Optional[torch.Tensor] = None,
                     stream=None):
    """Q8_0-form activations of float32 x [M, K] (or [K]): (d f32 [M, K/32], qs i8 [M, K])."""
    if x.dim() == 1:
        x = x.view(1, -1)
    _need_cuda(x)
    if x.dtype != torch.float32 or not x.is_contiguous():
        raise ValueError("x must be a contiguous float32 tensor")
    M, K = x.shape
    if d is None:
        d = torch.empty((M, K // 32), dtype=torch.float32, device=x.device)
    if qs is None:
        qs = torch.empty((M, K), dtype=torch.int8, device=x.device)
    _check(_lib.kq_quantize_q8_0(_ptr(x), M, K, _ptr(d), _ptr(qs), _stream(stream)), "kq_quantize_q8_0")
    return d, qs


def kq_gemv_q8_0(packed: torch.Tensor, N: int, K: int, d: torch.Tensor, qs: torch.Tensor,
                 y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """y [N] = Q8_0 weights (packed image) x one Q8_0-form activation row (d, qs)."""
    _need_cuda(packed, d, qs)
    if y is None:
        y = torch.empty(N, dtype=torch.float32, device=packed.device)
    _check(_lib.kq_gemv_q8_0(_ptr(packed), int(N), int(K), _ptr(d), _ptr(qs), _ptr(y), _stream(stream)),
           "kq_gemv_q8_0")
    return y


def kq_gemm_q8_0(packed: torch.Tensor, N: int, K: int, d: torch.Tensor, qs: torch.Tensor,
                 y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Q8_0 GEMM: y [M, N] from a KQ_Q8_0 image and Q8_0-form activations d [M, K/32], qs [M, K]."""
    _need_cuda(packed, d, qs)
    M = qs.shape[0] if qs.dim() == 2 else 1
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=packed.device)
    _need_cuda(y)
    _check(_lib.kq_gemm_q8_0(_ptr(packed), N, K, _ptr(d), _ptr(qs), M, _ptr(y), _stream(stream)), "kq_gemm_q8_0")
    return y


def kq_gemv_q8_0_fused(packed: torch.Tensor, N: int, K: int, x: torch.Tensor, y: Optional[torch.Tensor] = None,
                       stream=None) -> torch.Tensor:
    """y [N] = Q8_0 weights x the fp32 row x [K], quantized inside the kernel."""
    _need_cuda(packed, x)
    if x.dtype != torch.float32 or not x.is_contiguous():
        raise ValueError("x must be a contiguous float32 tensor")
    if y is None:
        y = torch.empty(N, dtype=torch.float32, device=packed.device)
    _check(_lib.kq_gemv_q8_0_fused(_ptr(packed), int(N), int(K), _ptr(x), _ptr(y), _stream(stream)),
           "kq_gemv_q8_0_fused")
    return y


def kq_measure_mma_s8(blocks: int, iters: int, out: torch.Tensor = None, device=None, stream=None) -> torch.Tensor:
    """Launch the int8 mma.sync rate kernel (blocks x 8 warps, iters x 8 MMAs
    of 16x8x32 per warp); returns the per-thread checksums (1024 * iters)."""
    if out is None:
        out = torch.empty(max(int(blocks), 1) * 256, dtype=torch.int32,
                          device=device if device is not None else "cuda")
    _need_cuda(out)
    _check(_lib.kq_measure_mma_s8(int(blocks), int(iters), _ptr(out), _stream(stream)), "kq_measure_mma_s8")
    return out


def kq_debug_wait_timeout(limit_ns: int, stream=None) -> None:
    """Launch the never-satisfied bounded wait (test hook of the timeout path)."""
    _check(_lib.kq_debug_wait_timeout(int(limit_ns), _stream(stream)), "kq_debug_wait_timeout")


def kq_device_status(stream=None) -> int:
    return int(_lib.kq_device_status(_stream(stream)))


KQ_LAUNCH_PDL = 1
KQ_LAUNCH_GEMV_SPLIT = 2
KQ_LAUNCH_GEMM_SPLIT = 4


def kq_set_launch_flags(flags: int) -> int:
    """Set the process-wide launch flags (KQ_LAUNCH_PDL, KQ_LAUNCH_GEMV_SPLIT, KQ_LAUNCH_GEMM_SPLIT); returns
    the old ones."""
    return int(_lib.kq_set_launch_flags(int(flags)))


def kq_get_launch_flags() -> int:
    return int(_lib.kq_get_launch_flags())


def raw():
    """The ctypes handle of libkq.so, for callers that pass raw pointers."""
    return _lib


def kq_copy_in(src: torch.Tensor, dst: torch.Tensor, stream=None) -> torch.Tensor:
    """Copy the pinned host tensor src into the device tensor dst (same number
    of bytes, a multiple of 16) with a kernel of the stream's launch chain."""
    if src.device.type != "cpu" or not src.is_pinned() or not src.is_contiguous():
        raise ValueError("src must be a contiguous pinned host tensor")
    _need_cuda(dst)
    n = src.numel() * src.element_size()
    if not dst.is_contiguous() or dst.numel() * dst.element_size() != n:
        raise ValueError("dst must be a contiguous device tensor of the same size")
    _check(_lib.kq_copy_in(_ptr(src), _ptr(dst), n, _stream(stream)), "kq_copy_in")
    return dst
