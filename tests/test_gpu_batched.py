"""The strided batch of Q4_K products (q4k_gemm_batched / _f16) against the oracle.

Every problem of the batch is checked element by element at the workload bound
(including problems of one token, ragged token and row tiles, and a batch whose
units exceed the persistent grid so that CTAs run units of several problems),
and the rows around each problem's y are checked untouched.
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


def _batch(B, M, N, K, seed, f16=False):
    blocks = [synth.q4k_weights(N, K, seed=seed + p) for p in range(B)]
    w = torch.cat([qwp.q4k_repack(torch.from_numpy(b.reshape(-1)).to(DEV), N, K) for b in blocks])
    if f16:
        xs = [synth.activations_f16(M, K, seed=seed + 100 + p) for p in range(B)]
        x = torch.from_numpy(np.stack(xs)).to(DEV)
    else:
        xs = [synth.activations_bf16(M, K, seed=seed + 100 + p) for p in range(B)]
        x = torch.from_numpy(np.ascontiguousarray(np.stack(xs)).view(np.int16)).to(DEV).view(torch.bfloat16)
    return blocks, w, xs, x


@pytest.mark.parametrize("B,M,N,K", [(3, 32, 2048, 2048), (4, 105, 640, 1024), (5, 1, 300, 512), (2, 7, 130, 768),
                                     (8, 32, 2048, 2048), (40, 16, 1024, 512)])
def test_batched_bf16_against_oracle(B, M, N, K):
    blocks, w, xs, x = _batch(B, M, N, K, seed=B * 11 + M)
    # y inside a NaN guard of 64 floats each side; a problem's y need not start on
    # 16 bytes (M*N*4 is not a multiple of 16 for M7 N130), only the batch's does
    flat = torch.full((B * M * N + 128,), float("nan"), dtype=torch.float32, device=DEV)
    y = flat[64:64 + B * M * N].view(B, M, N)
    qwp.q4k_gemm_batched(w, x, N, out=y)
    g = flat.cpu().numpy()
    assert np.isnan(g[:64]).all() and np.isnan(g[64 + B * M * N:]).all(), "wrote outside the batch"
    g = g[64:64 + B * M * N].reshape(B, M, N)
    for p in range(B):
        ref, mag = oracle.q4k_gemm(blocks[p], xs[p], N, K)
        check_bound(g[p], ref, mag, f"problem {p} of B{B} M{M} N{N} K{K}")


@pytest.mark.parametrize("B,M,N,K", [(3, 32, 2048, 2048), (6, 9, 256, 1024)])
def test_batched_f16_against_oracle(B, M, N, K):
    blocks, w, xs, x = _batch(B, M, N, K, seed=B * 13 + M, f16=True)
    y = qwp.q4k_gemm_batched(w, x, N).cpu().numpy()
    for p in range(B):
        wf = oracle.q4k_dequant(blocks[p], N, K)
        ref, mag = oracle.gemm(oracle.half_to_f64(xs[p].view(np.uint16)), wf)
        check_bound(y[p], ref, mag, f"f16 problem {p}")


def test_batched_equals_single_calls_bitwise():
    """Each problem of a batch gets the same units as a single call would only when
    the plans agree; its result must at least equal a single call on the same
    problem to the workload bound, and two batched calls are bitwise identical."""
    B, M, N, K = 4, 32, 2048, 2048
    blocks, w, xs, x = _batch(B, M, N, K, seed=77)
    y1 = qwp.q4k_gemm_batched(w, x, N).cpu().numpy()
    y2 = qwp.q4k_gemm_batched(w, x, N).cpu().numpy()
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
    nb = w.numel() // B
    for p in range(B):
        ys = qwp.q4k_gemm(w[p * nb:(p + 1) * nb], x[p], N).cpu().numpy()
        ref, mag = oracle.q4k_gemm(blocks[p], xs[p], N, K)
        check_bound(ys, ref, mag, f"single {p}")
        check_bound(y1[p], ref, mag, f"batched {p}")
