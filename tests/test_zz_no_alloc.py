"""q4k_gemm_noalloc (the Q4_K GEMM whose activation scratch is a fixed array in
the library) against the CPU oracle and against q4k_gemm (pool scratch), through
the C ABI.

Two calls in a row with different activations and token counts must each meet
the GEMM tolerance against the oracle and against q4k_gemm, so a stale copy of x
left in the array by the first call cannot pass; M*K at the limit runs, one
token row beyond it is rejected before any work.  Collected last so that it also
runs after every other test in the same process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import quantized_weight_prefill_gb300 as qwp
import synth
from helpers import check_bound

DEV = "cuda"
SCRATCH_LIMIT = -8


def _bf16_on_gpu(xb):
    return torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).to(DEV).view(torch.bfloat16)


def test_noalloc_rejects_beyond_the_limit_before_any_cuda_call():
    lib = qwp.library()
    p = ctypes.c_void_p(0x1000)
    K = 1024
    m_max = qwp.NOALLOC_MAX_X_ELEMS // K
    assert lib.q4k_gemm_noalloc(p, p, p, m_max + 1, 8, K, None) == SCRATCH_LIMIT
    assert lib.qwp_status_string(SCRATCH_LIMIT).decode() == "QWP_ERR_SCRATCH_LIMIT"
    assert lib.q4k_gemm_noalloc(p, p, p, 0, 8, K, None) == 0
    assert lib.q4k_gemm_noalloc(p, p, p, 4, 8, 100, None) == -2


@pytest.mark.gpu
def test_noalloc_matches_q4k_gemm_on_two_calls_in_a_row():
    N, K = 384, 1024
    blocks = synth.q4k_weights(N, K, seed=901)
    w = qwp.q4k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
    for call, (M, seed) in enumerate([(300, 902), (77, 903)]):
        xb = synth.activations_bf16(M, K, seed=seed)
        x = _bf16_on_gpu(xb)
        y_ref = qwp.q4k_gemm(w, x, N)
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
        qwp.q4k_gemm_noalloc(w, x, N, out=y)
        torch.cuda.synchronize()
        assert qwp.device_status() == 0
        ref, mag = oracle.q4k_gemm(blocks, xb, N, K)
        check_bound(y.cpu().numpy(), ref, mag, f"q4k_gemm_noalloc call {call + 1} (M={M}) against the oracle")
        check_bound(y.cpu().numpy(), y_ref.cpu().numpy().astype(np.float64), mag,
                    f"q4k_gemm_noalloc call {call + 1} (M={M}) against q4k_gemm")


@pytest.mark.gpu
def test_noalloc_at_the_limit_and_one_row_beyond():
    N, K = 136, 1024
    M = qwp.NOALLOC_MAX_X_ELEMS // K
    blocks = synth.q4k_weights(N, K, seed=904)
    w = qwp.q4k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
    xb = synth.activations_bf16(M, K, seed=905)
    x = _bf16_on_gpu(xb)
    y_ref = qwp.q4k_gemm(w, x, N)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
    qwp.q4k_gemm_noalloc(w, x, N, out=y)
    torch.cuda.synchronize()
    assert qwp.device_status() == 0
    rows = np.r_[0:16, M - 16:M]
    ref, mag = oracle.q4k_gemm(blocks, xb[rows], N, K)
    check_bound(y[rows].cpu().numpy(), ref, mag, "q4k_gemm_noalloc at M*K = limit, against the oracle")
    check_bound(y[rows].cpu().numpy(), y_ref[rows].cpu().numpy().astype(np.float64), mag,
                "q4k_gemm_noalloc at M*K = limit, against q4k_gemm")
    assert torch.isfinite(y).all()

    x_big = torch.zeros(M + 1, K, dtype=torch.bfloat16, device=DEV)
    y_big = torch.full((M + 1, N), 7.0, dtype=torch.float32, device=DEV)
    with pytest.raises(qwp.QwpError) as e:
        qwp.q4k_gemm_noalloc(w, x_big, N, out=y_big)
    assert e.value.code == SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert bool((y_big == 7.0).all()), "a rejected call must not touch y"


@pytest.mark.gpu
@pytest.mark.parametrize("policy,M,N,K", [(0, 1, 65600, 512), (2, 7, 2500, 8192)])
def test_noalloc_decode_shaped(policy, M, N, K):
    """Decode-shaped calls keep the decode kernel's partial sums in the library's
    second fixed array: two calls in a row (different activations) each meet the
    bound against the oracle, by default (one token, wide matrix) and with the
    decode kernel forced (seven tokens)."""
    prev = qwp.set_decode_policy(policy)
    try:
        assert qwp.decode_selected("q4k", M, N, K)
        blocks = synth.q4k_weights(N, K, seed=906 + M)
        w = qwp.q4k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
        for call, seed in enumerate((907, 908)):
            xb = synth.activations_bf16(M, K, seed=seed)
            y = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
            qwp.q4k_gemm_noalloc(w, _bf16_on_gpu(xb), N, out=y)
            torch.cuda.synchronize()
            assert qwp.device_status() == 0
            ref, mag = oracle.q4k_gemm(blocks, xb, N, K)
            check_bound(y.cpu().numpy(), ref, mag, f"q4k_gemm_noalloc decode-shaped call {call + 1} (M={M})")
    finally:
        qwp.set_decode_policy(prev)

