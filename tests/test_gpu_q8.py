"""Quantized activations (8-bit codes per block of 32) and the Q4_K product with
them, through the C ABI, against the oracle.

* q8_quantize: the whole record buffer, byte for byte, against the documented
  layout filled from the oracle's codes, scales and sums (the codes are integers
  decided in fp32 on both sides, so they must match exactly), for ragged token
  counts (padding tokens zero), hand-worked blocks, values over a wide exponent
  range and rounding ties; a non-finite activation is reported as QWP_ERR_RANGE.
* q4k_q8_gemm: every element within the fp32 bound of its integer-dot
  arithmetic, (K/32 + 4) * 2^-24 * sum_k (|d*sc*q| + |dmin*m|) * |d_x*q_x|, of the
  oracle's fp64 product with the dequantized activations; bitwise reproducible;
  the vocabulary-sized shape on sampled rows; and the end-to-end quantization
  error against the unquantized product within half a code per activation.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import quantized_weight_prefill_gb300 as qwp
import synth
from helpers import q8_records_reference

pytestmark = pytest.mark.gpu

DEV = "cuda"
RANGE = -7
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert qwp.device_status() == 0, "a kernel reported an error"


def _to_dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def _wide_bf16(M, K, seed):
    """bf16 values over a wide exponent range, with zero blocks and exact halves."""
    rng = np.random.default_rng(seed)
    mant = rng.integers(0, 128, size=(M, K))
    expo = rng.integers(110, 140, size=(M, K))
    sign = rng.integers(0, 2, size=(M, K))
    bits = ((sign << 15) | (expo << 7) | mant).astype(np.uint16)
    if K >= 64:
        bits[0, 32:64] = 0                                      # a zero block
        bits[M - 1, :32] = 0x3F80 * np.ones(32, np.uint16)      # a block of ones
    return bits


@pytest.mark.parametrize("M,K,seed", [(1, 256, 1), (5, 512, 2), (8, 4096, 3), (9, 256, 4), (33, 1024, 5),
                                      (105, 4096, 6)])
def test_q8_quantize_records_bit_exact(M, K, seed):
    xb = synth.activations_bf16(M, K, seed=seed) if seed % 2 else _wide_bf16(M, K, seed)
    buf = qwp.q8_quantize(_to_dev_bf16(xb)).cpu().numpy()
    assert buf.size == qwp.q8_activation_bytes(M, K) == -(-M // 8) * (K // 256) * 2560
    q, d, s = oracle.q8_quantize(xb, K)
    assert np.array_equal(buf, q8_records_reference(q, d, s))


def test_q8_quantize_handbuilt_blocks():
    """The hand-worked blocks of tests/golden/q8_handbuilt.json, one per token."""
    with open(os.path.join(GOLDEN, "q8_handbuilt.json")) as f:
        cases = json.load(f)["cases"]
    rows = []
    for c in cases:
        vals = np.concatenate([np.full(int(n), v, np.float32) for v, n in c["x"]])
        row = np.tile(vals, 8)  # 256 values: the block repeated
        rows.append((row.view(np.uint32) >> 16).astype(np.uint16))
    xb = np.stack(rows)
    buf = qwp.q8_quantize(_to_dev_bf16(xb)).cpu().numpy().reshape(1, 1, 8, 320)
    for t, c in enumerate(cases):
        expect = np.concatenate([np.full(int(n), v, np.int64) for v, n in c["q"]])
        stored = buf[0, 0, t, :256].view(np.int8).reshape(32, 8)
        codes = np.empty_like(stored)
        codes[:, [0, 4, 1, 5, 2, 6, 3, 7]] = stored
        assert np.array_equal(codes.reshape(8, 32).astype(np.int64), np.tile(expect, (8, 1))), c["name"]
        assert np.all(buf[0, 0, t, 256:288].view(np.float32) == np.float32(c["d"]))
        assert np.all(buf[0, 0, t, 288:320].view(np.float32) == np.float32(c["s"]))


def test_q8_quantize_nonfinite_is_reported():
    xb = synth.activations_bf16(2, 256, seed=11)
    xb[1, 7] = 0x7FC0  # NaN
    qwp.q8_quantize(_to_dev_bf16(xb))
    assert qwp.device_status() == RANGE
    assert qwp.device_status() == 0


def _gemm_case(M, N, K, seed, xb=None):
    blocks = synth.q4k_weights(N, K, seed=seed)
    w = qwp.q4k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
    if xb is None:
        xb = synth.activations_bf16(M, K, seed=seed + 1)
    xq = qwp.q8_quantize(_to_dev_bf16(xb))
    return blocks, w, xb, xq


def _check_q8_bound(y, ref, mag2, K, what):
    tol = (K / 32 + 4) * 2.0 ** -24 * mag2 + 1e-30
    err = np.abs(y.astype(np.float64) - ref)
    bad = err > tol
    assert not bad.any(), f"{what}: {bad.sum()} elements out of bound, worst ratio {np.max(err / tol):.3g}"


@pytest.mark.parametrize("M,N,K", [(1, 1, 256), (1, 4096, 4096), (2, 300, 512), (5, 1000, 2048), (8, 4096, 4096),
                                   (8, 129, 12288), (3, 24576, 4096)])
def test_q4k_q8_gemm_against_oracle(M, N, K):
    blocks, w, xb, xq = _gemm_case(M, N, K, seed=M * 7 + N + K)
    y1 = qwp.q4k_q8_gemm(w, xq, M, N, K).cpu().numpy()
    y2 = qwp.q4k_q8_gemm(w, xq, M, N, K).cpu().numpy()
    q, d, _ = oracle.q8_quantize(xb, K)
    ref, mag2 = oracle.q4k_q8_gemm(blocks, q, d, N, K)
    _check_q8_bound(y1, ref, mag2, K, f"M{M} N{N} K{K}")
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32)), "not bitwise reproducible"


def test_q4k_q8_gemm_vocab_shape_sampled_rows():
    """One token against a vocabulary-sized matrix (N = 152064, K = 4096): the
    first, last and two middle 128-row tiles of y against the oracle."""
    M, N, K = 1, 152064, 4096
    blocks, w, xb, xq = _gemm_case(M, N, K, seed=77)
    y = qwp.q4k_q8_gemm(w, xq, M, N, K).cpu().numpy()
    rows = np.r_[0:128, 76032:76160, 100000:100128, N - 128:N]
    q, d, _ = oracle.q8_quantize(xb, K)
    ref, mag2 = oracle.q4k_q8_gemm(blocks.reshape(N, -1)[rows], q, d, len(rows), K)
    _check_q8_bound(y[:, rows], ref, mag2, K, "M1 N152064 K4096")


def test_q4k_q8_gemm_cancelling_blocks_and_wide_activations():
    """Blocks whose two terms cancel exactly (w == 0) give 0 whatever x is; x over
    a wide exponent range, with zero blocks."""
    M, N, K = 4, 40, 1024
    nb = N * (K // 256)
    rng = np.random.default_rng(13)
    blk = np.zeros((nb, 144), np.uint8)
    dbits = rng.uniform(1e-3, 4e-3, nb).astype(np.float16).view(np.uint16)
    blk[:, 0:2] = dbits.astype("<u2").view(np.uint8).reshape(nb, 2)
    blk[:, 2:4] = blk[:, 0:2]
    lo6 = rng.integers(1, 256, size=(nb, 4), dtype=np.uint8)
    blk[:, 4:8] = lo6
    blk[:, 8:12] = lo6
    nib = rng.integers(1, 16, size=(nb, 4), dtype=np.uint8)
    blk[:, 12:16] = nib | (nib << 4)
    blk[:, 16:] = 0x11
    blocks = blk.reshape(N, -1)
    assert not oracle.q4k_dequant(blocks, N, K).any()
    w = qwp.q4k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
    xb = _wide_bf16(M, K, seed=14)
    xq = qwp.q8_quantize(_to_dev_bf16(xb))
    y = qwp.q4k_q8_gemm(w, xq, M, N, K).cpu().numpy()
    q, d, _ = oracle.q8_quantize(xb, K)
    ref, mag2 = oracle.q4k_q8_gemm(blocks, q, d, N, K)
    assert not ref.any()
    _check_q8_bound(y, ref, mag2, K, "cancelling blocks")


def test_q4k_q8_gemm_quantization_error_is_half_a_code():
    """Against the unquantized product: |y - x.W| <= sum_k |W_k| * d_k / 2 (half a
    code per activation) plus the fp32 bound -- the accuracy this path trades."""
    M, N, K = 3, 512, 4096
    blocks, w, xb, xq = _gemm_case(M, N, K, seed=21)
    y = qwp.q4k_q8_gemm(w, xq, M, N, K).cpu().numpy().astype(np.float64)
    exact, _ = oracle.q4k_gemm(blocks, xb, N, K)
    q, d, _ = oracle.q8_quantize(xb, K)
    _, mag2 = oracle.q4k_q8_gemm(blocks, q, d, N, K)
    W = oracle.q4k_dequant(blocks, N, K)
    half = np.repeat(d.astype(np.float64), 32, axis=1) / 2 * (1 + 2.0 ** -20)
    bound = half @ np.abs(W).T + (K / 32 + 4) * 2.0 ** -24 * mag2
    assert np.all(np.abs(y - exact) <= bound)
    # and the quantization error is real: the path does not reproduce x.W to fp32
    assert np.abs(y - exact).max() > 1e-6 * np.abs(exact).max()


def test_q4k_q8_gemm_more_than_eight_tokens_is_refused():
    blocks, w, xb, xq = _gemm_case(9, 64, 256, seed=31)
    with pytest.raises(qwp.QwpError) as e:
        qwp.q4k_q8_gemm(w, xq, 9, 64, 256)
    assert e.value.code == -2
