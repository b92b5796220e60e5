"""K-quant (Q4_K / Q5_K / Q6_K) x Q8_K GEMV and GEMM for GB300 (sm_103a).

The compute path is the C-ABI library ``libkq.so`` (hand-written CUDA in
``csrc/``); :mod:`quantized_gemv_gemm_gb300.kq` is its thin ctypes binding
and raises at import when the library is missing.  :mod:`.synth` holds the
seeded synthetic inputs and imports nothing else from this package.
"""
