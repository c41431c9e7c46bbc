"""Seeded synthetic inputs shared by the tests, the bench and the oracle runs.

This module only draws random numbers and lays the drawn fields out at the byte
offsets of the GGUF block formats (minfer "CUDA Backend Design", §2.3 weight
registry; the per-type byte counts 34/32, 144/256 and 210/256). It holds none of
the method's arithmetic: no dequantisation, no scale packing, no quantisation.

Field distributions follow the five hot-path workloads (Qwen2.5-0.5B/7B shaped):

* Q8_0 (32 elements, 34 bytes): f16 ``d = |N(0,1)| * d_scale`` then 32 int8 ``qs``
  uniform on [-127, 127].
* Q4_K (256 elements, 144 bytes): f16 ``d = |N| * 0.02``, f16 ``dmin = |N| * 0.01``,
  12 scale bytes and 128 ``qs`` bytes uniform on [0, 255].  Uniform bytes make every
  packed 6-bit sub-block scale and min uniform on [0, 63] and independent, and every
  4-bit quant uniform on [0, 15], because each bit of those 140 bytes belongs to
  exactly one field.
* Q6_K (256 elements, 210 bytes): ``ql`` (128) and ``qh`` (64) bytes uniform on
  [0, 255] (so each 6-bit quant is uniform on [0, 63]), 16 int8 sub-scales uniform on
  [-128, 127], f16 ``d = |N| * 0.005``.
* Q4_0 (32 elements, 18 bytes): f16 ``d = |N| * 0.02`` then 16 quant bytes uniform on
  [0, 255] (each 4-bit quant uniform on [0, 15]).
* Q4_1 (32 elements, 20 bytes): f16 ``d = |N| * 0.02``, f16 ``m = -|N| * 0.1`` then 16
  quant bytes uniform on [0, 255].
* Q5_0 (32 elements, 22 bytes): f16 ``d = |N| * 0.01``, 4 fifth-bit bytes and 16 quant
  bytes uniform on [0, 255] (each 5-bit quant uniform on [0, 31]).
* Q5_1 (32 elements, 24 bytes): f16 ``d = |N| * 0.01``, f16 ``m = -|N| * 0.1``, then 4 + 16
  bytes as Q5_0.
* Q5_K (256 elements, 176 bytes): as Q4_K (f16 ``d = |N| * 0.02``, ``dmin = |N| * 0.01``,
  12 scale bytes) then 32 high-bit bytes and 128 quant bytes, all uniform on [0, 255]
  (each 5-bit quant uniform on [0, 31]).
* F16 (one element, 2 bytes): ``N(0,1) * 0.02`` rounded to f16.
* BF16 (one element, 2 bytes): the upper 16 bits of the f32 ``N(0,1) * 0.02`` (the value
  truncated toward zero to bfloat16).
* activations: f32 ``N(0,1) * x_scale``.

Random draws use ``numpy.random.Generator(PCG64(seed))``; within a weight the
fields are drawn in the order they are listed above, each for all blocks at once.
"""
from __future__ import annotations

import numpy as np

Q4_0, Q4_1, Q5_0, Q5_1, Q8_0, Q4_K, Q5_K, Q6_K = 2, 3, 6, 7, 8, 12, 13, 14  # GGUF type ids
F16, BF16 = 1, 30

# type id -> (elements per block, bytes per block)
BLOCK = {Q4_0: (32, 18), Q4_1: (32, 20), Q5_0: (32, 22), Q5_1: (32, 24), Q8_0: (32, 34),
         Q4_K: (256, 144), Q5_K: (256, 176), Q6_K: (256, 210), F16: (1, 2), BF16: (1, 2)}
TYPE_NAME = {Q4_0: "Q4_0", Q4_1: "Q4_1", Q5_0: "Q5_0", Q5_1: "Q5_1", Q8_0: "Q8_0",
             Q4_K: "Q4_K", Q5_K: "Q5_K", Q6_K: "Q6_K", F16: "F16", BF16: "BF16"}


def nbytes(qtype: int, N: int, K: int) -> int:
    be, bb = BLOCK[qtype]
    if K % be:
        raise ValueError(f"K={K} is not a multiple of {be}")
    return N * (K // be) * bb


def _absnormal_f16(rng, n, scale):
    return (np.abs(rng.standard_normal(n)) * scale).astype(np.float16)


def q8_0_weights(N: int, K: int, seed: int, d_scale: float = 0.01) -> np.ndarray:
    nb = N * (K // 32)
    rng = np.random.Generator(np.random.PCG64(seed))
    out = np.empty((nb, 34), dtype=np.uint8)
    out[:, 0:2] = _absnormal_f16(rng, nb, d_scale).view(np.uint8).reshape(nb, 2)
    out[:, 2:34] = rng.integers(-127, 128, size=(nb, 32), dtype=np.int8).view(np.uint8)
    return out.reshape(-1)


def q4_k_weights(N: int, K: int, seed: int, d_scale: float = 0.02,
                 dmin_scale: float = 0.01) -> np.ndarray:
    nb = N * (K // 256)
    rng = np.random.Generator(np.random.PCG64(seed))
    out = np.empty((nb, 144), dtype=np.uint8)
    out[:, 0:2] = _absnormal_f16(rng, nb, d_scale).view(np.uint8).reshape(nb, 2)
    out[:, 2:4] = _absnormal_f16(rng, nb, dmin_scale).view(np.uint8).reshape(nb, 2)
    out[:, 4:16] = rng.integers(0, 256, size=(nb, 12), dtype=np.uint8)
    out[:, 16:144] = rng.integers(0, 256, size=(nb, 128), dtype=np.uint8)
    return out.reshape(-1)


def q6_k_weights(N: int, K: int, seed: int, d_scale: float = 0.005) -> np.ndarray:
    nb = N * (K // 256)
    rng = np.random.Generator(np.random.PCG64(seed))
    out = np.empty((nb, 210), dtype=np.uint8)
    out[:, 0:128] = rng.integers(0, 256, size=(nb, 128), dtype=np.uint8)
    out[:, 128:192] = rng.integers(0, 256, size=(nb, 64), dtype=np.uint8)
    out[:, 192:208] = rng.integers(-128, 128, size=(nb, 16), dtype=np.int8).view(np.uint8)
    out[:, 208:210] = _absnormal_f16(rng, nb, d_scale).view(np.uint8).reshape(nb, 2)
    return out.reshape(-1)


def q4_0_weights(N: int, K: int, seed: int, d_scale: float = 0.02) -> np.ndarray:
    nb = N * (K // 32)
    rng = np.random.Generator(np.random.PCG64(seed))
    out = np.empty((nb, 18), dtype=np.uint8)
    out[:, 0:2] = _absnormal_f16(rng, nb, d_scale).view(np.uint8).reshape(nb, 2)
    out[:, 2:18] = rng.integers(0, 256, size=(nb, 16), dtype=np.uint8)
    return out.reshape(-1)


def q32_min_weights(N: int, K: int, seed: int, nbytes: int, with_min: bool, qh: bool,
                    d_scale: float) -> np.ndarray:
    """Q4_1 / Q5_0 / Q5_1: f16 d, [f16 m], [4 fifth-bit bytes], 16 quant bytes."""
    nb = N * (K // 32)
    rng = np.random.Generator(np.random.PCG64(seed))
    out = np.empty((nb, nbytes), dtype=np.uint8)
    out[:, 0:2] = _absnormal_f16(rng, nb, d_scale).view(np.uint8).reshape(nb, 2)
    o = 2
    if with_min:
        out[:, 2:4] = (-_absnormal_f16(rng, nb, 0.1)).view(np.uint8).reshape(nb, 2)
        o = 4
    out[:, o:] = rng.integers(0, 256, size=(nb, nbytes - o), dtype=np.uint8)
    return out.reshape(-1)


def q5_k_weights(N: int, K: int, seed: int, d_scale: float = 0.02,
                 dmin_scale: float = 0.01) -> np.ndarray:
    nb = N * (K // 256)
    rng = np.random.Generator(np.random.PCG64(seed))
    out = np.empty((nb, 176), dtype=np.uint8)
    out[:, 0:2] = _absnormal_f16(rng, nb, d_scale).view(np.uint8).reshape(nb, 2)
    out[:, 2:4] = _absnormal_f16(rng, nb, dmin_scale).view(np.uint8).reshape(nb, 2)
    out[:, 4:16] = rng.integers(0, 256, size=(nb, 12), dtype=np.uint8)
    out[:, 16:48] = rng.integers(0, 256, size=(nb, 32), dtype=np.uint8)
    out[:, 48:176] = rng.integers(0, 256, size=(nb, 128), dtype=np.uint8)
    return out.reshape(-1)


def float_weights(N: int, K: int, seed: int, bf16: bool, w_scale: float = 0.02) -> np.ndarray:
    """F16 or BF16: N x K elements, row-major, little-endian."""
    rng = np.random.default_rng(seed)
    v = (rng.standard_normal(N * K) * w_scale).astype(np.float32)
    bits = (v.view(np.uint32) >> 16).astype(np.uint16) if bf16 else v.astype(np.float16).view(np.uint16)
    return bits.astype("<u2").view(np.uint8).copy()


def weights(qtype: int, N: int, K: int, seed: int) -> np.ndarray:
    """Raw GGUF bytes of an N x K weight, rows contiguous, blocks along K."""
    if qtype in (F16, BF16):
        return float_weights(N, K, seed, qtype == BF16)
    if qtype == Q4_0:
        return q4_0_weights(N, K, seed)
    if qtype == Q4_1:
        return q32_min_weights(N, K, seed, 20, True, False, 0.02)
    if qtype == Q5_0:
        return q32_min_weights(N, K, seed, 22, False, True, 0.01)
    if qtype == Q5_1:
        return q32_min_weights(N, K, seed, 24, True, True, 0.01)
    if qtype == Q5_K:
        return q5_k_weights(N, K, seed)
    if qtype == Q8_0:
        return q8_0_weights(N, K, seed)
    if qtype == Q4_K:
        return q4_k_weights(N, K, seed)
    if qtype == Q6_K:
        return q6_k_weights(N, K, seed)
    raise ValueError(f"unsupported GGUF type {qtype}")


def activations(rows: int, K: int, seed: int, x_scale: float = 1.0) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((rows, K), dtype=np.float32)
    if x_scale != 1.0:
        x *= np.float32(x_scale)
    return x


# The five hot-path workloads.  ``B`` lists the decode batch sizes, ``M`` the
# prefill row counts; seeds: weights first, then activations.
WORKLOADS = {
    "q8_0_matvec_896x896": dict(qtype=Q8_0, N=896, K=896, B=(1,), M=(), w_seed=101,
                                x_seed=0, x_scale=1.0),
    "q4_k_matvec_18944x3584": dict(qtype=Q4_K, N=18944, K=3584, B=(1,), M=(), w_seed=102,
                                   x_seed=202, x_scale=1.0),
    "q6_k_matvec_3584x18944": dict(qtype=Q6_K, N=3584, K=18944, B=(1, 2, 4, 8), M=(),
                                   w_seed=103, x_seed=203, x_scale=1.0),
    "q4_k_mmq_512x18944x3584": dict(qtype=Q4_K, N=18944, K=3584, B=(), M=(512,), w_seed=102,
                                    x_seed=204, x_scale=1.0),
    "q6_k_lm_head_151936x3584": dict(qtype=Q6_K, N=151936, K=3584, B=(1,), M=(2048,),
                                     w_seed=105, x_seed=205, x_scale=0.5),
}
