"""The skinny-N kernel (Q4_K, N <= 64 weight rows, M >= 256 tokens) against the oracle.

Through the C ABI: bf16 and fp16 activations, weight counts from 1 to 64 (MMA N
padded to 16, 32, 48, 64), token tiles of 2 to 128 rows (cut to fill whole
waves) with a ragged last tile, K split over clusters of 1, 2, 4 and 8 CTAs
(reduction slices that do not divide the tile), the workload's stress shape (M=4096, N=32, K=4096; sampled token
rows), blocks whose terms cancel, bitwise reproducibility, the no-alloc entry
point and bf16 activations beyond fp16's range (taken as they are).  Every element must
meet |y - y_oracle| <= 1e-3 * sum|x*w| + 1e-5.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_weight_prefill_gb300 as qwp
import synth
from helpers import check_bound

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert qwp.device_status() == 0, "a kernel reported an error"


def _setup(M, N, K, seed):
    blocks = synth.q4k_weights(N, K, seed=seed)
    w = qwp.q4k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
    xb = synth.activations_bf16(M, K, seed=seed + 1)
    x = torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).to(DEV).view(torch.bfloat16)
    return blocks, w, xb, x


# (M, N, K): N over 1..64, ragged M, K giving every cluster size 1, 2, 4, 8.
SHAPES = [(256, 32, 4096), (300, 1, 256), (1000, 7, 512), (513, 16, 1024), (777, 33, 2048),
          (4096, 64, 4096), (2048, 48, 12288), (20000, 32, 512), (640, 17, 8192), (5000, 5, 2048)]


def test_shapes_take_the_skinny_kernel_with_every_split():
    splits = set()
    for M, N, K in SHAPES:
        p = qwp.gemm_plan("q4k", M, N, K)
        assert p["kernel"] == "skinny", (M, N, K, p)
        tm = p["token_tile"]
        assert 1 <= tm <= 128 and p["clusters"] == -(-M // tm) and (K // 256) % p["splits"] == 0
        assert (p["clusters"] - 1) * tm < M  # no empty tile
        splits.add(p["splits"])
    assert {1, 2, 4, 8} <= splits, sorted(splits)
    assert qwp.gemm_plan("q4k", 255, 32, 4096)["kernel"] == "prefill"
    assert qwp.gemm_plan("q4k", 4096, 65, 4096)["kernel"] == "prefill"
    assert qwp.gemm_plan("q6k", 4096, 32, 4096)["kernel"] == "prefill"


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_skinny_bf16_against_oracle(M, N, K):
    blocks, w, xb, x = _setup(M, N, K, seed=M + N + K)
    y1 = qwp.q4k_gemm(w, x, N).cpu().numpy()
    y2 = qwp.q4k_gemm(w, x, N).cpu().numpy()
    ref, mag = oracle.q4k_gemm(blocks, xb, N, K)
    check_bound(y1, ref, mag, f"skinny M{M} N{N} K{K} plan {qwp.gemm_plan('q4k', M, N, K)}")
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32)), "not bitwise reproducible"


@pytest.mark.parametrize("M,N,K", [(256, 32, 4096), (777, 33, 2048), (1000, 7, 512), (4096, 32, 4096)])
def test_skinny_f16_against_oracle(M, N, K):
    blocks = synth.q4k_weights(N, K, seed=M + 5)
    w = qwp.q4k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
    xh = synth.activations_f16(M, K, seed=M + 6)
    y = qwp.q4k_gemm_f16(w, torch.from_numpy(xh).to(DEV), N).cpu().numpy()
    ref, mag = oracle.gemm(oracle.half_to_f64(xh.view(np.uint16)), oracle.q4k_dequant(blocks, N, K))
    check_bound(y, ref, mag, f"skinny fp16 M{M} N{N} K{K}")


def test_skinny_stress_shape_sampled_rows():
    """The workload's skinny gate projection: M=4096, N=32, K=4096; token rows 0-127,
    1920-2175 and the last 128 (spanning several token tiles and their boundaries,
    the ragged last tile included) against the oracle."""
    M, N, K = 4096, 32, 4096
    blocks, w, xb, x = _setup(M, N, K, seed=601)
    y = qwp.q4k_gemm(w, x, N).cpu().numpy()
    rows = np.r_[0:128, 1920:2048, 2048:2176, M - 128:M]
    ref, mag = oracle.q4k_gemm(blocks, xb[rows], N, K)
    check_bound(y[rows], ref, mag, "skinny M4096 N32 K4096")


def test_skinny_exact_cancellation_gives_zero():
    """d == dmin, sc_j == m_j (mirrored scale bytes), every nibble 1: W == 0, so y == 0."""
    M, N, K = 512, 24, 2048
    nb = N * (K // 256)
    rng = np.random.default_rng(7)
    blk = np.zeros((nb, 144), np.uint8)
    d = rng.uniform(1e-3, 4e-3, nb).astype(np.float16).view(np.uint16)
    blk[:, 0:2] = d.astype("<u2").view(np.uint8).reshape(nb, 2)
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
    xb = synth.activations_bf16(M, K, seed=8) & np.uint16(0x7FFF)
    x = torch.from_numpy(xb.view(np.int16)).to(DEV).view(torch.bfloat16)
    y = qwp.q4k_gemm(w, x, N).cpu().numpy()
    assert np.array_equal(y, np.zeros_like(y)), f"max |y| {np.abs(y).max():.3g} for an all-zero W"


def test_skinny_noalloc_two_calls():
    """q4k_gemm_noalloc takes the same kernel (it needs no scratch): two calls in a row."""
    N, K = 32, 4096
    blocks = synth.q4k_weights(N, K, seed=611)
    w = qwp.q4k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
    for M, seed in ((1024, 612), (300, 613)):
        xb = synth.activations_bf16(M, K, seed=seed)
        x = torch.from_numpy(xb.view(np.int16)).to(DEV).view(torch.bfloat16)
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
        qwp.q4k_gemm_noalloc(w, x, N, out=y)
        ref, mag = oracle.q4k_gemm(blocks, xb, N, K)
        check_bound(y.cpu().numpy(), ref, mag, f"skinny noalloc M{M}")


def test_skinny_bf16_beyond_fp16_range_is_exact():
    """bf16 activations go to the tensor core unconverted (weights as a bf16 hi + lo
    pair), so values beyond fp16's range (1e5, 3e6) and below its subnormals (1e-9)
    are taken as they are: the result meets the bound and no range error is set."""
    M, N, K = 256, 16, 512
    blocks, w, xb, x = _setup(M, N, K, seed=621)
    big = np.array([1.0e5, -3.0e6, 1.0e-9, -2.5e-8], np.float32).view(np.uint32) >> 16
    for (r, c), v in zip([(5, 17), (100, 300), (200, 3), (255, 511)], big):
        xb[r, c] = np.uint16(v)
    x = torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).to(DEV).view(torch.bfloat16)
    y = qwp.q4k_gemm(w, x, N).cpu().numpy()
    assert qwp.device_status() == 0
    ref, mag = oracle.q4k_gemm(blocks, xb, N, K)
    check_bound(y, ref, mag, "skinny bf16 beyond fp16 range")
