"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

* repacks byte-exact against the documented layouts,
* dequant entry points bit-exact against the oracle's fp64 values rounded to fp32,
* GEMMs within |y - y_oracle| <= 1e-3 * sum|x*w| + 1e-5 elementwise, on tiny
  shapes with ragged tails, on every workload shape (sampled token rows at the
  large ones) and on edge cases (empty, misaligned, guard bands).
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_weight_prefill_gb300 as qwp
import synth
from helpers import (check_bound, q4k_oracle_rows, q4k_tiled_reference, q6k_oracle_rows, q6k_tiled_reference,
                     sample_rows, w4a16_oracle_rows, w4a16_tiled_reference)

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _q4k_on_gpu(N, K, seed):
    blocks = synth.q4k_weights(N, K, seed=seed)
    w = qwp.q4k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
    return blocks, w


def _q6k_on_gpu(N, K, seed):
    blocks = synth.q6k_weights(N, K, seed=seed)
    w = qwp.q6k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
    return blocks, w


def _bf16_on_gpu(xb):
    return torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).to(DEV).view(torch.bfloat16)


def _w4_on_gpu(N, K, g, seed):
    wq, s, z = synth.w4a16_weights(N, K, g, seed=seed)
    wt = qwp.w4a16_repack(torch.from_numpy(wq.view(np.int32)).to(DEV))
    return (wq, s, z), (wt, torch.from_numpy(s).to(DEV), torch.from_numpy(z).to(DEV))


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert qwp.device_status() == 0, "a kernel reported a timeout"


# --- repack and dequant ------------------------------------------------------------

@pytest.mark.parametrize("N,K", [(1, 256), (5, 512), (128, 256), (130, 768), (300, 1024)])
def test_q4k_repack_layout(N, K):
    blocks, w = _q4k_on_gpu(N, K, seed=N + K)
    assert np.array_equal(w.cpu().numpy(), q4k_tiled_reference(blocks, N, K))


@pytest.mark.parametrize("N,K", [(1, 64), (5, 128), (130, 512), (257, 1024)])
def test_w4a16_repack_layout(N, K):
    (wq, _, _), (wt, _, _) = _w4_on_gpu(N, K, 64, seed=N + K)
    assert np.array_equal(wt.cpu().numpy().view(np.uint32).reshape(-1), w4a16_tiled_reference(wq, N, K))


@pytest.mark.parametrize("N,K", [(1, 256), (7, 512), (130, 1024), (4096, 12288)])
def test_q4k_dequant_bit_exact(N, K):
    blocks, w = _q4k_on_gpu(N, K, seed=3 * N + K)
    got = qwp.q4k_dequant(w, N, K).cpu().numpy()
    ref = oracle.q4k_dequant(blocks, N, K).astype(np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_q4k_dequant_extreme_scales_bit_exact():
    """Subnormal, tiny and large fp16 d/dmin still give the correctly rounded fp32 value."""
    N, K = 64, 512
    blocks = synth.q4k_weights(N, K, seed=77).reshape(-1, 144).copy()
    rng = np.random.default_rng(78)
    special = np.array([0x0001, 0x03FF, 0x0400, 0x1400, 0x3C00, 0x5BFF, 0x7BFF, 0x8001, 0xBC00],
                       np.uint16)
    d = rng.choice(special, size=blocks.shape[0])
    dm = rng.choice(special, size=blocks.shape[0])
    blocks[:, 0:2] = d.astype("<u2").view(np.uint8).reshape(-1, 2)
    blocks[:, 2:4] = dm.astype("<u2").view(np.uint8).reshape(-1, 2)
    w = qwp.q4k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
    got = qwp.q4k_dequant(w, N, K).cpu().numpy()
    ref = oracle.q4k_dequant(blocks.reshape(-1), N, K).astype(np.float32)
    # Every value is bit-identical; only the sign of an exact zero may differ (d < 0, q = m = 0).
    got, ref = got + np.float32(0), ref + np.float32(0)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("N,K,g", [(1, 64, 64), (9, 256, 128), (130, 512, 128), (4096, 12288, 128)])
def test_w4a16_dequant_bit_exact(N, K, g):
    (wq, s, z), (wt, sd, zd) = _w4_on_gpu(N, K, g, seed=5 * N + K)
    got = qwp.w4a16_dequant(wt, sd, zd, N, K, g).cpu().numpy()
    ref = oracle.w4a16_dequant(wq, s, z, N, K, g).astype(np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


# --- GEMM: tiny shapes with ragged tails ------------------------------------------

TINY = [(1, 1, 256), (7, 5, 256), (16, 128, 512), (33, 130, 768), (105, 256, 1024),
        (200, 384, 512), (300, 136, 256), (257, 129, 512), (64, 1000, 256)]


@pytest.mark.parametrize("M,N,K", TINY)
def test_q4k_gemm_tiny(M, N, K):
    blocks, w = _q4k_on_gpu(N, K, seed=M * 7 + N)
    xb = synth.activations_bf16(M, K, seed=M + 1)
    y = qwp.q4k_gemm(w, _bf16_on_gpu(xb), N).cpu().numpy()
    ref, mag = oracle.q4k_gemm(blocks, xb, N, K)
    check_bound(y, ref, mag, f"q4k M{M} N{N} K{K}")


@pytest.mark.parametrize("M,N,K", [(1, 1, 256), (33, 130, 768), (105, 256, 1024), (300, 136, 256)])
def test_q4k_gemm_f16_activations(M, N, K):
    """The fp16-activation entry point (no conversion pass) against the oracle."""
    blocks, w = _q4k_on_gpu(N, K, seed=M * 5 + N)
    xh = synth.activations_f16(M, K, seed=M + 3)
    y = qwp.q4k_gemm_f16(w, torch.from_numpy(xh).to(DEV), N).cpu().numpy()
    wf = oracle.q4k_dequant(blocks, N, K)
    ref, mag = oracle.gemm(oracle.half_to_f64(xh.view(np.uint16)), wf)
    check_bound(y, ref, mag, f"q4k f16 M{M} N{N} K{K}")


def _x_conversion(M, N, K, fmt="q4k"):
    """Where a bf16-x call of this shape on the prefill kernel converts x: "epilogue"
    (every CTA runs at most one unit with two accumulators and converts at most
    32 KB of x, or 64 KB of at most 16 token rows: the epilogue warps convert each
    x slot), "mma" (one token: the MMA warp converts the token row), else "kernel"
    (a conversion kernel first)."""
    p = qwp.gemm_plan(fmt, M, N, K)
    assert p["kernel"] == "prefill"
    k_cta = -(-(K // 64) // p["splits"]) * 64
    rows = min(p["token_tile"], M)
    small = rows * k_cta * 2 <= 32768 or (rows <= 16 and rows * k_cta * 2 <= 65536)
    if p["units_per_cluster"] == 1 and p["token_tile"] <= 128 and small:
        return "epilogue"
    return "mma" if M == 1 else "kernel"


@pytest.mark.parametrize("M,N,K,where", [(1, 2048, 2048, "epilogue"), (1, 40000, 1024, "mma"),
                                         (1, 19456, 4096, "epilogue"), (1, 700, 8192, "epilogue"),
                                         (2, 3000, 1024, "epilogue"), (32, 2048, 2048, "epilogue"),
                                         (105, 4096, 4096, "kernel"), (16, 1000, 768, "epilogue"),
                                         (13, 700, 8192, "epilogue"), (24, 1000, 1536, "epilogue"),
                                         (8, 4096, 12288, "epilogue"), (32, 4096, 4096, "kernel"),
                                         (8, 40000, 1024, "kernel"), (300, 40000, 256, "kernel")])
def test_q4k_bf16_x_conversion_paths(M, N, K, where):
    """bf16 x on the prefill kernel, each way of converting it to the fp16 MMA
    operand: by the epilogue warps in shared memory (one unit per CTA, also with
    split-K and ragged token rows), by the MMA warp (one token, CTAs with several
    units), or by a conversion kernel first; every element within the bound."""
    prev = qwp.set_decode_policy(qwp.DECODE_NEVER)
    try:
        assert _x_conversion(M, N, K) == where, qwp.gemm_plan("q4k", M, N, K)
        blocks, w = _q4k_on_gpu(N, K, seed=M * 3 + N)
        xb = synth.activations_bf16(M, K, seed=M + 9)
        y = qwp.q4k_gemm(w, _bf16_on_gpu(xb), N).cpu().numpy()
    finally:
        qwp.set_decode_policy(prev)
    ref, mag = oracle.q4k_gemm(blocks, xb, N, K)
    check_bound(y, ref, mag, f"q4k bf16 M{M} N{N} K{K} ({where}) plan {qwp.gemm_plan('q4k', M, N, K)}")


@pytest.mark.parametrize("M,N,K,where", [(8, 128, 256, "epilogue"), (1, 40000, 256, "mma"),
                                         (8, 40000, 256, "kernel"), (32, 2048, 2048, "epilogue")])
def test_q4k_bf16_activation_beyond_fp16_range_is_reported(M, N, K, where):
    """An activation that overflows fp16 is reported as QWP_ERR_RANGE whichever way
    x is converted, and the next call is clean."""
    prev = qwp.set_decode_policy(qwp.DECODE_NEVER)
    try:
        assert _x_conversion(M, N, K) == where
        blocks, w = _q4k_on_gpu(N, K, seed=31)
        xb = synth.activations_bf16(M, K, seed=32).copy()
        r = min(3, M - 1)
        xb[r, K - 17] = 0x4880  # bf16 262144.0, beyond fp16's largest finite value
        qwp.q4k_gemm(w, _bf16_on_gpu(xb), N)
        assert qwp.device_status() == -7
        xb[r, K - 17] = 0x3F80  # 1.0
        y = qwp.q4k_gemm(w, _bf16_on_gpu(xb), N).cpu().numpy()
        assert qwp.device_status() == 0
    finally:
        qwp.set_decode_policy(prev)
    ref, mag = oracle.q4k_gemm(blocks, xb, N, K)
    check_bound(y, ref, mag, "after a range error")


@pytest.mark.parametrize("M,N,K,g", [(1, 1, 64, 64), (7, 5, 256, 128), (33, 130, 768, 64),
                                     (105, 256, 1024, 128), (300, 136, 512, 256), (257, 200, 320, 64)])
def test_w4a16_gemm_tiny(M, N, K, g):
    (wq, s, z), (wt, sd, zd) = _w4_on_gpu(N, K, g, seed=M * 11 + N)
    xh = synth.activations_f16(M, K, seed=M + 2)
    y = qwp.w4a16_gemm(wt, sd, zd, torch.from_numpy(xh).to(DEV), N, g).cpu().numpy()
    ref, mag = oracle.w4a16_gemm(wq, s, z, xh, N, K, g)
    check_bound(y, ref, mag, f"w4a16 M{M} N{N} K{K} g{g}")


def test_w4a16_more_units_than_ctas_with_short_last_stage():
    """157 row tiles on at most one CTA per SM: CTAs run several units in turn, and K = 320
    leaves a last weight stage of one block (the other transform warps only release it)."""
    M, N, K, g = 33, 20000, 320, 64
    (wq, s, z), (wt, sd, zd) = _w4_on_gpu(N, K, g, seed=77)
    xh = synth.activations_f16(M, K, seed=78)
    y = qwp.w4a16_gemm(wt, sd, zd, torch.from_numpy(xh).to(DEV), N, g).cpu().numpy()
    ref, mag = oracle.w4a16_gemm(wq, s, z, xh, N, K, g)
    check_bound(y, ref, mag, f"w4a16 M{M} N{N} K{K} g{g}")


@pytest.mark.parametrize("N,K,g", [(1, 64, 64), (130, 512, 128), (4096, 4096, 128)])
def test_w4a16_symmetric_dequant_bit_exact(N, K, g):
    """No zero points: w = s * (q - 8)."""
    (wq, s, _), (wt, sd, _) = _w4_on_gpu(N, K, g, seed=9 * N + K)
    got = qwp.w4a16_dequant(wt, sd, None, N, K, g).cpu().numpy()
    ref = oracle.w4a16_dequant(wq, s, None, N, K, g).astype(np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("M,N,K,g", [(1, 1, 64, 64), (33, 130, 768, 64), (105, 256, 1024, 128),
                                     (257, 200, 320, 64)])
def test_w4a16_symmetric_gemm_tiny(M, N, K, g):
    (wq, s, _), (wt, sd, _) = _w4_on_gpu(N, K, g, seed=M * 13 + N)
    xh = synth.activations_f16(M, K, seed=M + 3)
    y = qwp.w4a16_gemm(wt, sd, None, torch.from_numpy(xh).to(DEV), N, g).cpu().numpy()
    ref, mag = oracle.w4a16_gemm(wq, s, None, xh, N, K, g)
    check_bound(y, ref, mag, f"w4a16 sym M{M} N{N} K{K} g{g}")


@pytest.mark.parametrize("symmetric", [False, True])
@pytest.mark.parametrize("M,N,K,g", [(1, 1, 64, 64), (7, 5, 256, 128), (105, 256, 1024, 128),
                                     (300, 136, 512, 256)])
def test_w4a16_bf16_gemm_tiny(M, N, K, g, symmetric):
    (wq, s, z), (wt, sd, zd) = _w4_on_gpu(N, K, g, seed=M * 17 + N)
    if symmetric:
        z = zd = None
    xb = synth.activations_bf16(M, K, seed=M + 4)
    y = qwp.w4a16_gemm_bf16(wt, sd, zd, _bf16_on_gpu(xb), N, g).cpu().numpy()
    ref, mag = oracle.w4a16_gemm_bf16(wq, s, z, xb, N, K, g)
    check_bound(y, ref, mag, f"w4a16 bf16 sym={symmetric} M{M} N{N} K{K} g{g}")


def test_w4a16_bf16_activation_beyond_fp16_range_is_reported():
    """An activation that overflows fp16 is reported as QWP_ERR_RANGE, and the next call is clean."""
    M, N, K, g = 8, 128, 256, 128
    (wq, s, z), (wt, sd, zd) = _w4_on_gpu(N, K, g, seed=31)
    xb = synth.activations_bf16(M, K, seed=32).copy()
    xb[3, 17] = 0x4880  # bf16 262144.0, beyond fp16's largest finite value
    qwp.w4a16_gemm_bf16(wt, sd, zd, _bf16_on_gpu(xb), N, g)
    assert qwp.device_status() == -7
    xb[3, 17] = 0x3F80  # 1.0
    y = qwp.w4a16_gemm_bf16(wt, sd, zd, _bf16_on_gpu(xb), N, g).cpu().numpy()
    assert qwp.device_status() == 0
    ref, mag = oracle.w4a16_gemm_bf16(wq, s, z, xb, N, K, g)
    check_bound(y, ref, mag, "w4a16 bf16 after a range error")


# --- Q6_K ------------------------------------------------------------------------------

@pytest.mark.parametrize("N,K", [(1, 256), (5, 512), (130, 256), (300, 768)])
def test_q6k_repack_layout(N, K):
    blocks, w = _q6k_on_gpu(N, K, seed=N + K)
    assert w.numel() == qwp.q6k_repacked_bytes(N, K)
    assert np.array_equal(w.cpu().numpy(), q6k_tiled_reference(blocks, N, K))


@pytest.mark.parametrize("N,K", [(1, 256), (9, 512), (130, 512), (4096, 4096)])
def test_q6k_dequant_bit_exact(N, K):
    blocks, w = _q6k_on_gpu(N, K, seed=3 * N + K)
    got = qwp.q6k_dequant(w, N, K).cpu().numpy()
    ref = oracle.q6k_dequant(blocks, N, K).astype(np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("M,N,K", TINY)
def test_q6k_gemm_tiny(M, N, K):
    blocks, w = _q6k_on_gpu(N, K, seed=M * 7 + N)
    xb = synth.activations_bf16(M, K, seed=M + 5)
    y = qwp.q6k_gemm(w, _bf16_on_gpu(xb), N).cpu().numpy()
    ref, mag = oracle.q6k_gemm(blocks, xb, N, K)
    check_bound(y, ref, mag, f"q6k M{M} N{N} K{K}")


@pytest.mark.parametrize("M,N,K", [(1, 3, 256), (40, 200, 512), (257, 129, 768)])
def test_q6k_gemm_f16_activations(M, N, K):
    blocks, w = _q6k_on_gpu(N, K, seed=M + 3 * N)
    xh = synth.activations_f16(M, K, seed=M + 6)
    y = qwp.q6k_gemm_f16(w, torch.from_numpy(xh).to(DEV), N).cpu().numpy()
    ref, mag = oracle.gemm(oracle.half_to_f64(xh.view(np.uint16)), oracle.q6k_dequant(blocks, N, K))
    check_bound(y, ref, mag, f"q6k f16 M{M} N{N} K{K}")


def test_q6k_more_units_than_ctas():
    """253 row tiles (the last one of 100 rows, padded to 104) over at most one CTA per SM."""
    M, N, K = 24, 32356, 256
    blocks, w = _q6k_on_gpu(N, K, seed=91)
    xb = synth.activations_bf16(M, K, seed=92)
    y = qwp.q6k_gemm(w, _bf16_on_gpu(xb), N).cpu().numpy()
    ref, mag = oracle.q6k_gemm(blocks, xb, N, K)
    check_bound(y, ref, mag, f"q6k M{M} N{N} K{K}")


@pytest.mark.parametrize("M,name,K,N", [(105, "attn_v", 4096, 1024), (105, "ffn_down", 12288, 4096),
                                        (2048, "ffn_down", 12288, 4096), (658, "attn_v", 4096, 1024)])
def test_q6k_qwen3_8b_projections(M, name, K, N):
    """The projections a Q4_K_M checkpoint stores in Q6_K, at the workload token counts
    (every element at M=105, sampled rows beyond)."""
    blocks, w = _q6k_on_gpu(N, K, seed=K + N + M)
    xb = synth.activations_bf16(M, K, seed=M + 17)
    y = qwp.q6k_gemm(w, _bf16_on_gpu(xb), N)
    rows = np.arange(M) if M <= 128 else sample_rows(M, seed=M)
    ys = y[torch.from_numpy(rows).to(DEV)].cpu().numpy()
    ref, mag = q6k_oracle_rows(blocks, xb[rows], N, K)
    check_bound(ys, ref, mag, f"q6k {name} M{M} N{N} K{K}")


# --- GEMM: the workload shapes -------------------------------------------------------

def _q4k_workload(M, N, K, seed, rows=None):
    blocks, w = _q4k_on_gpu(N, K, seed=seed)
    xb = synth.activations_bf16(M, K, seed=seed + 1000)
    y = qwp.q4k_gemm(w, _bf16_on_gpu(xb), N)
    sel = np.arange(M) if rows is None else rows
    ys = y[torch.from_numpy(sel).to(DEV)].cpu().numpy()
    ref, mag = q4k_oracle_rows(blocks, xb[sel], N, K)
    return check_bound(ys, ref, mag, f"q4k M{M} N{N} K{K}")


def test_q4k_skinny_m_full():
    """M=32 tokens, N=2048, K=2048: every output element."""
    _q4k_workload(32, 2048, 2048, seed=1)


@pytest.mark.parametrize("name,K,N", synth.QWEN3_8B_LAYER)
def test_q4k_qwen3_8b_layer_m105(name, K, N):
    """The 105-token layer the benchmark times: every output element of every projection."""
    _q4k_workload(105, N, K, seed={"qkv": 2, "o": 3, "gate_up": 4, "down": 5}[name])


@pytest.mark.parametrize("M", [658, 2048])
@pytest.mark.parametrize("name,K,N", synth.QWEN3_8B_LAYER)
def test_q4k_qwen3_8b_layer_large_m(M, name, K, N):
    _q4k_workload(M, N, K, seed=M + len(name), rows=sample_rows(M, seed=M))


@pytest.mark.parametrize("M,N,K", [(4096, 32, 4096), (8192, 12288, 4096)])
def test_q4k_stress(M, N, K):
    _q4k_workload(M, N, K, seed=M + N, rows=sample_rows(M, seed=N))


@pytest.mark.parametrize("K,N,arm", [(4096, 12288, "f16"), (12288, 4096, "f16"),
                                     (4096, 12288, "f16_symmetric"), (12288, 4096, "bf16"),
                                     (4096, 12288, "bf16_symmetric")])
def test_w4a16_m2048(K, N, arm):
    M, g = 2048, 128
    (wq, s, z), (wt, sd, zd) = _w4_on_gpu(N, K, g, seed=K + 5)
    if arm.endswith("symmetric"):
        z = zd = None
    rows = sample_rows(M, seed=K)
    if arm.startswith("bf16"):
        xb = synth.activations_bf16(M, K, seed=K + 6)
        y = qwp.w4a16_gemm_bf16(wt, sd, zd, _bf16_on_gpu(xb), N, g)
        ref, mag = w4a16_oracle_rows(wq, s, z, xb[rows], N, K, g, bf16=True)
    else:
        xh = synth.activations_f16(M, K, seed=K + 6)
        y = qwp.w4a16_gemm(wt, sd, zd, torch.from_numpy(xh).to(DEV), N, g)
        ref, mag = w4a16_oracle_rows(wq, s, z, xh[rows], N, K, g)
    ys = y[torch.from_numpy(rows).to(DEV)].cpu().numpy()
    check_bound(ys, ref, mag, f"w4a16 {arm} M{M} N{N} K{K}")


# --- edge cases -----------------------------------------------------------------------

def test_empty_problems_are_noops():
    blocks, w = _q4k_on_gpu(8, 256, seed=9)
    y = torch.full((0, 8), float("nan"), device=DEV)
    qwp.q4k_gemm(w, torch.empty(0, 256, dtype=torch.bfloat16, device=DEV), 8, out=y)
    y2 = torch.full((4, 0), 1.0, device=DEV)
    qwp.q4k_gemm(w, torch.zeros(4, 256, dtype=torch.bfloat16, device=DEV), 0, out=y2)


def test_guard_band_untouched():
    """Output writes stay inside [M, N] even with ragged row and token tiles."""
    M, N, K = 37, 131, 512
    blocks, w = _q4k_on_gpu(N, K, seed=12)
    xb = synth.activations_bf16(M, K, seed=13)
    buf = torch.full((M * N + 4096,), float("nan"), device=DEV)
    y = buf[:M * N].view(M, N)
    qwp.q4k_gemm(w, _bf16_on_gpu(xb), N, out=y)
    assert torch.isnan(buf[M * N:]).all()
    ref, mag = oracle.q4k_gemm(blocks, xb, N, K)
    check_bound(y.cpu().numpy(), ref, mag, "guard band")


def test_misaligned_and_bad_shapes_rejected():
    blocks, w = _q4k_on_gpu(8, 256, seed=14)
    x = torch.zeros(5, 256, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(qwp.QwpError) as e:  # output starting 4 bytes into an allocation
        qwp.q4k_gemm(w, x, 8, out=torch.empty(5 * 8 + 1, device=DEV)[1:].view(5, 8))
    assert e.value.code == -3
    with pytest.raises(qwp.QwpError) as e:
        qwp.q4k_gemm(w, torch.zeros(4, 300, dtype=torch.bfloat16, device=DEV), 8)
    assert e.value.code == -2


def test_repeat_calls_are_deterministic():
    M, N, K = 96, 256, 1024
    blocks, w = _q4k_on_gpu(N, K, seed=15)
    x = _bf16_on_gpu(synth.activations_bf16(M, K, seed=16))
    y1 = qwp.q4k_gemm(w, x, N)
    y2 = qwp.q4k_gemm(w, x, N)
    assert torch.equal(y1, y2)
