"""libkq.so loads, exports every entry point of include/kq.h, and rejects bad
arguments on the host (no GPU needed: argument checks run before any CUDA
call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kq.h")


@pytest.fixture(scope="module")
def kq():
    from quantized_gemv_gemm_gb300 import build
    build.build()
    from quantized_gemv_gemm_gb300 import kq as mod
    return mod


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kq_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(kq):
    lib = ctypes.CDLL(kq.LIB_PATH)
    names = declared_functions()
    assert len(names) >= 12
    for name in names:
        assert hasattr(lib, name), f"{name} declared in kq.h but not exported"


def test_sizes_and_names(kq):
    assert [kq.kq_block_bytes(f) for f in (1, 2, 3)] == [144, 176, 210]
    assert kq.kq_block_bytes(7) == 0
    for f, per_sb in ((1, 144), (2, 176), (3, 210)):
        for N, K in ((4096, 2560), (1, 256), (5, 17408)):
            nb = kq.kq_repack_bytes(f, N, K)
            assert nb % 256 == 0
            disk = N * (K // 256) * per_sb
            padded = -(-N // 16) * 16 * (K // 256) * per_sb   # rows padded to groups of 16
            bounds = -(-N // 16) * (K // 256) * 8             # the bounds plane: 8 B per (row group, superblock)
            assert disk + bounds <= nb <= padded + bounds + 5 * 255
    assert kq.kq_repack_bytes(1, 10, 100) == 0
    assert kq.kq_repack_bytes(1, -1, 256) == 0
    assert kq.kq_repack_bytes(5, 10, 256) == 0
    # Q8_0 images: qs plane (4096 B per 16 rows x 256 columns) + fp16 scale plane (256 B)
    assert kq.kq_block_bytes(4) == 34
    assert kq.kq_repack_bytes(4, 10, 256) == 4096 + 256
    for N, K in ((17408, 5120), (1, 256), (33, 768)):
        ch = -(-N // 16) * (K // 256)
        assert kq.kq_repack_bytes(4, N, K) == -(-ch * 4096 // 256) * 256 + -(-ch * 256 // 256) * 256
    assert kq.kq_repack_bytes(4, 10, 32) == 0
    assert "invalid" in kq.kq_strerror(-1)
    assert kq.kq_strerror(12345) == "unknown kq status"


def test_host_argument_checks(kq):
    lib = kq.raw()
    Q = kq._Q8KConst
    nullq = Q(0, 0, 0)
    fake = ctypes.c_void_p(0x10000)       # never dereferenced: checks fail first
    odd = ctypes.c_void_p(0x10004)
    goodq = Q(0x10000, 0x10000, 0x10000)
    ARG, ALIGN, FMT, WS = -1, -2, -3, -6
    # format (Q8_0 is not a K-quant: the K-quant entry points reject it)
    assert lib.kq_gemv(9, fake, 8, 256, goodq, fake, None, 0, None) == FMT
    assert lib.kq_gemv(4, fake, 8, 256, goodq, fake, None, 0, None) == FMT
    assert lib.kq_gemm(4, fake, 8, 256, goodq, 32, fake, None, 0, None) == FMT
    # Q8_0 rail
    assert lib.kq_quantize_q8_0(fake, 2, 48, fake, fake, None) == ARG
    assert lib.kq_quantize_q8_0(fake, -1, 64, fake, fake, None) == ARG
    assert lib.kq_quantize_q8_0(None, 0, 64, None, None, None) == 0
    assert lib.kq_quantize_q8_0(odd, 2, 64, fake, fake, None) == ALIGN
    assert lib.kq_gemv_q8_0(fake, 8, 200, fake, fake, fake, None) == ARG
    assert lib.kq_gemv_q8_0(fake, 8, 256 * 161, fake, fake, fake, None) == ARG
    assert lib.kq_gemv_q8_0(None, 0, 256, None, None, None, None) == 0
    assert lib.kq_gemv_q8_0(None, 8, 256, fake, fake, fake, None) == ARG
    assert lib.kq_gemv_q8_0(odd, 8, 256, fake, fake, fake, None) == ALIGN
    assert lib.kq_gemv_q8_0(fake, 8, 256, fake, odd, fake, None) == ALIGN
    assert lib.kq_copy_in(fake, fake, 24, None) == ARG
    assert lib.kq_copy_in(None, None, 0, None) == 0
    assert lib.kq_copy_in(None, fake, 32, None) == ARG
    assert lib.kq_copy_in(odd, fake, 32, None) == ALIGN
    assert lib.kq_copy_in(fake, odd, 32, None) == ALIGN
    assert lib.kq_gemv_q8_0_fused(fake, 8, 200, fake, fake, None) == ARG
    assert lib.kq_gemv_q8_0_fused(fake, 8, 256 * 161, fake, fake, None) == ARG
    assert lib.kq_gemv_q8_0_fused(None, 0, 256, None, None, None) == 0
    assert lib.kq_gemv_q8_0_fused(fake, 8, 256, None, fake, None) == ARG
    assert lib.kq_gemv_q8_0_fused(fake, 8, 256, odd, fake, None) == ALIGN
    assert lib.kq_repack(0, fake, 8, 256, fake, None) == FMT
    # shapes
    assert lib.kq_gemv(1, fake, 8, 100, goodq, fake, None, 0, None) == ARG
    assert lib.kq_gemv(1, fake, -1, 256, goodq, fake, None, 0, None) == ARG
    assert lib.kq_quantize_q8k(fake, -1, 256, goodq, None) == ARG
    assert lib.kq_quantize_q8k(fake, 2, 300, goodq, None) == ARG
    # null pointers
    assert lib.kq_gemv(1, None, 8, 256, goodq, fake, None, 0, None) == ARG
    assert lib.kq_gemv(1, fake, 8, 256, nullq, fake, None, 0, None) == ARG
    assert lib.kq_gemm(1, fake, 8, 256, goodq, 4, None, None, 0, None) == ARG
    assert lib.kq_gemm_grouped(1, fake, 4, None, 8, 256, goodq, 4, fake, None, 0, None) == ARG
    assert lib.kq_quantize_q8k(None, 2, 256, goodq, None) == ARG
    # alignment
    assert lib.kq_gemv(1, odd, 8, 256, goodq, fake, None, 0, None) == ALIGN
    assert lib.kq_gemv(1, fake, 8, 256, Q(0x10000, 0x10004, 0x10000), fake, None, 0, None) == ALIGN
    assert lib.kq_quantize_q8k(odd, 2, 256, goodq, None) == ALIGN
    assert lib.kq_repack(1, odd, 8, 256, fake, None) == ALIGN
    # GEMV workspace: too small / misaligned
    wsn = kq.KQ_GEMV_WORKSPACE_BYTES
    assert wsn == lib.kq_gemv_workspace_bytes() == 64 * 1024
    assert lib.kq_gemv(1, fake, 8, 256, goodq, fake, fake, wsn - 1, None) == WS
    assert lib.kq_gemv(1, fake, 8, 256, goodq, fake, odd, wsn, None) == ALIGN
    pk1 = (ctypes.c_void_p * 1)(0x10000)
    n1 = (ctypes.c_int64 * 1)(8)
    y1 = (ctypes.c_void_p * 1)(0x10000)
    assert lib.kq_gemv_fused(1, 1, pk1, n1, 256, fake, y1, fake, 16, None) == WS
    # fused batch: negative M, and M = 0 is a no-op that needs no x
    assert lib.kq_gemv_fused_batch(1, 1, pk1, n1, 256, fake, -1, y1, None, 0, None) == ARG
    assert lib.kq_gemv_fused_batch(1, 1, pk1, n1, 256, None, 0, y1, None, 0, None) == 0
    assert lib.kq_gemv_fused_batch(1, 1, pk1, n1, 256, odd, 2, y1, None, 0, None) == ALIGN
    assert lib.kq_gemv_fused_batch(1, 5, pk1, n1, 256, fake, 2, y1, None, 0, None) == ARG
    # fused grouped decode: sets x rows over 16, too many sets, K not a multiple of 256, zero rows
    off = ctypes.c_void_p(0x10000)
    pk4 = (ctypes.c_void_p * 5)(*([0x10000] * 5))
    n4 = (ctypes.c_int64 * 5)(*([8] * 5))
    y4 = (ctypes.c_void_p * 5)(*([0x10000] * 5))
    assert lib.kq_gemv_grouped_fused(1, 2, pk4, n4, 256, 4, off, fake, 9, y4, None) == ARG
    assert lib.kq_gemv_grouped_fused(1, 5, pk4, n4, 256, 4, off, fake, 1, y4, None) == ARG
    assert lib.kq_gemv_grouped_fused(1, 1, pk4, n4, 300, 4, off, fake, 1, y4, None) == ARG
    assert lib.kq_gemv_grouped_fused(4, 1, pk4, n4, 256, 4, off, fake, 1, y4, None) == FMT
    assert lib.kq_gemv_grouped_fused(1, 1, pk4, n4, 256, 4, None, None, 0, y4, None) == 0
    assert lib.kq_gemv_grouped_fused(1, 1, pk4, n4, 256, 4, off, odd, 2, y4, None) == ALIGN
    # the timeout test hook refuses a zero or over-one-second limit (no launch)
    assert lib.kq_debug_wait_timeout(0, None) == ARG
    assert lib.kq_debug_wait_timeout(2_000_000_000, None) == ARG
    # int8 MMA rate hook: argument checks only (no launch)
    assert lib.kq_measure_mma_s8(-1, 10, fake, None) == ARG
    assert lib.kq_measure_mma_s8(4, -1, fake, None) == ARG
    assert lib.kq_measure_mma_s8(4, 10, None, None) == ARG
    assert lib.kq_measure_mma_s8(0, 10, None, None) == 0
    # empty problems are no-ops that touch nothing
    assert lib.kq_gemv(1, None, 0, 256, nullq, None, None, 0, None) == 0
    assert lib.kq_gemm(2, None, 16, 512, nullq, 0, None, None, 0, None) == 0
    assert lib.kq_quantize_q8k(None, 0, 256, nullq, None) == 0
    # workspace: required size must be provided when non-zero
    need = kq.kq_gemm_workspace_bytes(1, 512, 4096, 2560)
    if need:
        assert lib.kq_gemm(1, fake, 4096, 2560, goodq, 512, fake, None, 0, None) == WS


def test_launch_flags_mask(kq):
    """Unknown flag bits are dropped; the three defined ones are kept."""
    old = kq.kq_set_launch_flags(0xFFFF)
    try:
        assert kq.kq_get_launch_flags() == kq.KQ_LAUNCH_PDL | kq.KQ_LAUNCH_GEMV_SPLIT | kq.KQ_LAUNCH_GEMM_SPLIT
        assert kq.kq_set_launch_flags(0) == kq.KQ_LAUNCH_PDL | kq.KQ_LAUNCH_GEMV_SPLIT | kq.KQ_LAUNCH_GEMM_SPLIT
        assert kq.kq_get_launch_flags() == 0
    finally:
        kq.kq_set_launch_flags(old)


def test_header_is_plain_c(tmp_path):
    """include/kq.h is a C header (the boundary other languages bind to): a C11
    translation unit that includes it and takes the address of every entry
    point compiles with gcc -Wall -Werror."""
    import re
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    cuda_inc = "/usr/local/cuda/include"
    if not gcc or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime_api.h")):
        pytest.skip("gcc or the CUDA headers not available")
    hdr = os.path.join(ROOT, "include", "kq.h")
    names = sorted(set(re.findall(r"^(?:int|size_t|unsigned|const char \*)\s*\**\s*(kq_\w+)\(",
                                  open(hdr).read(), re.M)))
    assert len(names) >= 15
    src = tmp_path / "use_kq.c"
    src.write_text('#include "kq.h"\n' + "".join(f"void *p_{n} = (void *)&{n};\n" for n in names))
    r = subprocess.run([gcc, "-std=c11", "-Wall", "-Werror", "-fsyntax-only", "-I", os.path.join(ROOT, "include"),
                        "-I", cuda_inc, str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
