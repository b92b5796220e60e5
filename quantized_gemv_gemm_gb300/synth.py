"""Seeded synthetic inputs for the K-quant x Q8_K path.

This module is shared by the oracle tests, the CUDA parity tests and the
benchmark.  It draws random bytes and floats only: it holds none of the
method's arithmetic (no decode, no quantization, no fold).

Every tensor draws from ``numpy.random.default_rng([0, config, tensor])``.
Weights are GGUF-order disk superblocks, shape ``[N, K/256, block_bytes]``:

* every byte uniform on 0..255 (this makes every packed 4/5/6-bit quant and
  every 6-bit scale/min uniform, since the packings use all their bits);
* the fp16 super-scales ``d`` (and ``dmin`` for Q4_K/Q5_K) uniform on
  [1e-3, 1e-2), stored little-endian;
* Q6_K's 16 signed sub-scales uniform on -32..31.

Activations are float32 N(0, 1); the 27B-shaped layer multiplies each
element by 20 with probability 0.01 ("1% outliers x20").
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

Q4_K, Q5_K, Q6_K = 1, 2, 3
FORMAT_NAMES = {Q4_K: "Q4_K", Q5_K: "Q5_K", Q6_K: "Q6_K"}
BLOCK_BYTES = {Q4_K: 144, Q5_K: 176, Q6_K: 210}
QK = 256


def rng_for(config: int, tensor: int) -> np.random.Generator:
    return np.random.default_rng([0, int(config), int(tensor)])


def _put_f16(raw: np.ndarray, offset: int, values: np.ndarray) -> None:
    b = np.ascontiguousarray(values.astype("<f2")).view(np.uint8)
    raw[..., offset:offset + 2] = b.reshape(values.shape + (2,))


def disk_weights(fmt: int, N: int, K: int, rng: np.random.Generator) -> np.ndarray:
    """Random GGUF-order superblocks, uint8 [N, K/256, block_bytes]."""
    assert K % QK == 0
    nsb = K // QK
    bb = BLOCK_BYTES[fmt]
    raw = rng.integers(0, 256, size=(N, nsb, bb), dtype=np.uint8)
    if fmt in (Q4_K, Q5_K):
        _put_f16(raw, 0, rng.uniform(1e-3, 1e-2, size=(N, nsb)))
        _put_f16(raw, 2, rng.uniform(1e-3, 1e-2, size=(N, nsb)))
    elif fmt == Q6_K:
        sc = rng.integers(-32, 32, size=(N, nsb, 16)).astype(np.int8)
        raw[..., 192:208] = sc.view(np.uint8)
        _put_f16(raw, 208, rng.uniform(1e-3, 1e-2, size=(N, nsb)))
    else:
        raise ValueError(f"unknown format {fmt}")
    return raw


Q8_0 = 4
Q8_0_BLOCK = 34   # fp16 d + 32 int8 quants (GGUF order)
QK8_0 = 32


def disk_weights_q8_0(N: int, K: int, rng: np.random.Generator) -> np.ndarray:
    """Random GGUF-order Q8_0 blocks, uint8 [N, K/32, 34]: fp16 d ~ U(1e-3, 1e-2),
    quants ~ U{-127..127}."""
    assert K % QK8_0 == 0
    nb = K // QK8_0
    raw = np.empty((N, nb, Q8_0_BLOCK), np.uint8)
    raw[..., 2:] = rng.integers(-127, 128, size=(N, nb, QK8_0)).astype(np.int8).view(np.uint8)
    _put_f16(raw, 0, rng.uniform(1e-3, 1e-2, size=(N, nb)))
    return raw


def activations(M: int, K: int, rng: np.random.Generator, outliers: bool = False) -> np.ndarray:
    x = rng.standard_normal((M, K), dtype=np.float32)
    if outliers:
        mask = rng.random((M, K)) < 0.01
        x[mask] *= np.float32(20.0)
    return x


def moe_routing(tokens: int, experts: int, topk: int, rng: np.random.Generator):
    """Top-k routing drawn uniformly: each token picks ``topk`` distinct experts.

    Returns (row_token int32 [tokens*topk], row_expert int32, offsets int32
    [experts+1]) with rows stable-sorted by (expert, token)."""
    choice = np.argsort(rng.random((tokens, experts)), axis=1)[:, :topk]
    tok = np.repeat(np.arange(tokens, dtype=np.int64), topk)
    exp = choice.reshape(-1).astype(np.int64)
    order = np.lexsort((tok, exp))
    row_token = tok[order].astype(np.int32)
    row_expert = exp[order].astype(np.int32)
    counts = np.bincount(row_expert, minlength=experts)
    offsets = np.zeros(experts + 1, np.int32)
    offsets[1:] = np.cumsum(counts)
    return row_token, row_expert, offsets


@dataclass
class Matrix:
    name: str
    fmt: int
    N: int
    K: int

    @property
    def weight_bytes(self) -> int:
        return self.N * (self.K // QK) * BLOCK_BYTES[self.fmt]


@dataclass
class Config:
    index: int
    name: str
    M: int
    matrices: list = field(default_factory=list)
    outliers: bool = False
    experts: int = 0
    topk: int = 0


def qwen3_4b_layer(fmt_main: int, fmt_down: int):
    return [
        Matrix("wq", fmt_main, 4096, 2560),
        Matrix("wk", fmt_main, 1024, 2560),
        Matrix("wv", fmt_main, 1024, 2560),
        Matrix("wo", fmt_main, 2560, 4096),
        Matrix("gate", fmt_main, 9728, 2560),
        Matrix("up", fmt_main, 9728, 2560),
        Matrix("down", fmt_down, 2560, 9728),
    ]


def configs():
    """The five workloads: shapes, formats and token counts."""
    return [
        Config(0, "tiny Q4_K GEMV 256x1024", 1, [Matrix("w", Q4_K, 256, 1024)]),
        Config(1, "Qwen3-4B-shaped decode layer, M=1", 1, qwen3_4b_layer(Q4_K, Q6_K)),
        Config(2, "Qwen3-4B-shaped prefill pp512 (all Q5_K, then all Q6_K)", 512,
               qwen3_4b_layer(Q5_K, Q5_K) + qwen3_4b_layer(Q6_K, Q6_K)),
        Config(3, "27B-shaped dense FFN, Q4_K, M=1 and M=512", 512,
               [Matrix("gate", Q4_K, 17408, 5120), Matrix("up", Q4_K, 17408, 5120),
                Matrix("down", Q4_K, 5120, 17408)], outliers=True),
        Config(4, "30B-A3B-shaped MoE grouped GEMM, 128 experts top-8, 512 tokens", 512,
               [Matrix("gate", Q4_K, 768, 2048), Matrix("up", Q4_K, 768, 2048),
                Matrix("down", Q6_K, 2048, 768)], experts=128, topk=8),
    ]
