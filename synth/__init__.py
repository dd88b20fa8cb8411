"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module holds no arithmetic of the method: it only draws random bytes and
random values and stores them in the fields of the weight formats.  Both the
CPU oracle and the GPU path consume the very same buffers.

Recipe (the workload definitions fix the value distributions):
  Q4_K weights   per 144-byte super-block: d and dmin uniform in [1e-3, 4e-3]
                 in float64, rounded to fp16 (round-to-nearest-even); the 12
                 packed scale bytes and the 128 nibble bytes uniform random
                 bytes.  Every one of the 96 packed scale bits feeds exactly
                 one 6-bit value, so uniform bytes give independent 6-bit
                 scales/mins uniform in 0..63, and uniform bytes give nibbles
                 uniform in 0..15.
  Q6_K weights   per 210-byte block: the 128 ql and 64 qh bytes uniform random
                 bytes (every bit of the 1536 code bits feeds exactly one code,
                 so the 6-bit codes are uniform in 0..63); the 16 int8 scales
                 uniform random bytes (uniform in -128..127); d uniform in
                 [1e-5, 8e-5] rounded to fp16, so that both subnormal and
                 normal fp16 d occur (GGML puts the block's largest scale near
                 127, which leaves d small: weights of magnitude ~0.05 give d
                 ~1e-5).
  W4A16 weights  uniform random 32-bit words (so every 4-bit code is uniform
                 in 0..15 whatever the bit interleave), fp16 scales uniform in
                 [1e-3, 4e-3], uint8 zero points uniform in 0..15.
  activations    N(0, 1) in float32, rounded to bf16 (Q4_K path) or fp16
                 (W4A16 path) with round-to-nearest-even.
"""
from __future__ import annotations

import numpy as np

Q4K_BLOCK_BYTES = 144  # bytes per 256-weight super-block (0.5625 byte per weight)
Q4K_BLOCK_K = 256
Q6K_BLOCK_BYTES = 210  # ql[128], qh[64], int8 scales[16], fp16 d


def _fp16_bits(values: np.ndarray) -> np.ndarray:
    return values.astype(np.float16).view(np.uint16)


def q4k_weights(N: int, K: int, seed: int, lo: float = 1e-3, hi: float = 4e-3) -> np.ndarray:
    """GGML Q4_K rows: uint8 array [N, K/256*144]; super-block b of row n at byte 144*b."""
    if K % Q4K_BLOCK_K:
        raise ValueError("K must be a multiple of 256")
    rng = np.random.default_rng(seed)
    nb = N * (K // Q4K_BLOCK_K)
    blk = np.empty((nb, Q4K_BLOCK_BYTES), np.uint8)
    d = _fp16_bits(rng.uniform(lo, hi, nb))
    dmin = _fp16_bits(rng.uniform(lo, hi, nb))
    blk[:, 0:2] = d.astype("<u2").view(np.uint8).reshape(nb, 2)
    blk[:, 2:4] = dmin.astype("<u2").view(np.uint8).reshape(nb, 2)
    blk[:, 4:144] = rng.integers(0, 256, size=(nb, 140), dtype=np.uint8)
    return blk.reshape(N, (K // Q4K_BLOCK_K) * Q4K_BLOCK_BYTES)


def q6k_weights(N: int, K: int, seed: int, lo: float = 1e-5, hi: float = 8e-5) -> np.ndarray:
    """GGML Q6_K rows: uint8 array [N, K/256*210]; block b of row n at byte 210*b."""
    if K % Q4K_BLOCK_K:
        raise ValueError("K must be a multiple of 256")
    rng = np.random.default_rng(seed)
    nb = N * (K // Q4K_BLOCK_K)
    blk = np.empty((nb, Q6K_BLOCK_BYTES), np.uint8)
    blk[:, 0:208] = rng.integers(0, 256, size=(nb, 208), dtype=np.uint8)
    d = _fp16_bits(rng.uniform(lo, hi, nb))
    blk[:, 208:210] = d.astype("<u2").view(np.uint8).reshape(nb, 2)
    return blk.reshape(N, (K // Q4K_BLOCK_K) * Q6K_BLOCK_BYTES)


def w4a16_weights(N: int, K: int, group: int, seed: int, lo: float = 1e-3, hi: float = 4e-3):
    """(wq uint32 [N, K/8], scales fp16 [N, K/group], zeros uint8 [N, K/group])."""
    if K % 8 or K % group:
        raise ValueError("K must be a multiple of 8 and of the group size")
    rng = np.random.default_rng(seed)
    wq = rng.integers(0, 2**32, size=(N, K // 8), dtype=np.uint64).astype(np.uint32)
    scales = rng.uniform(lo, hi, size=(N, K // group)).astype(np.float16)
    zeros = rng.integers(0, 16, size=(N, K // group), dtype=np.uint8)
    return wq, scales, zeros


def _normal_f32(M: int, K: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.standard_normal((M, K), dtype=np.float32)


def activations_bf16(M: int, K: int, seed: int) -> np.ndarray:
    """N(0,1) activations rounded to bf16; returned as uint16 bit patterns [M, K]."""
    import torch

    x = torch.from_numpy(_normal_f32(M, K, seed)).to(torch.bfloat16)
    return x.view(torch.int16).numpy().view(np.uint16)


def activations_f16(M: int, K: int, seed: int) -> np.ndarray:
    """N(0,1) activations rounded to fp16 [M, K]."""
    return _normal_f32(M, K, seed).astype(np.float16)


# The workloads (shapes and seeds) every test and the benchmark draw from.
QWEN3_8B_LAYER = (  # (name, K, N) of the four projections of one layer
    ("qkv", 4096, 6144),
    ("o", 4096, 4096),
    ("gate_up", 4096, 24576),
    ("down", 12288, 4096),
)
