"""The prefill kernel's bounded waits, made to run out on purpose.

A main-loop wait limit of a few nanoseconds (qwp_set_wait_timeout_ns) makes the
first wait that does not succeed at once give up.  The kernel must then record
QWP_ERR_TIMEOUT in the device status word, let every CTA wait for its own copies
and MMAs in flight (those waits keep their 2 s bound), release its tensor memory
and exit; while the status word holds the timeout, later launches must skip
their work (y untouched); reading the status clears it, and the next call is
correct again.  Nothing here faults or hangs the GPU: no wait, arrive or copy is
removed, only the limit of the waits is shortened.  Run on plans without
split-K (no cluster), with one and with two accumulators, so that no copy or
remote access of another CTA can outlive a CTA.
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
TIMEOUT = -6


@pytest.mark.parametrize("M,N,K", [(128, 19456, 4096), (2048, 4096, 4096)])
def test_short_wait_limit_times_out_cleanly(M, N, K):
    assert qwp.device_status() == 0
    plan = qwp.gemm_plan("q4k", M, N, K)
    assert plan["kernel"] == "prefill" and plan["splits"] == 1, plan
    blocks = synth.q4k_weights(N, K, seed=M + 31)
    w = qwp.q4k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
    xb = synth.activations_bf16(M, K, seed=M + 32)
    x = torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).to(DEV).view(torch.bfloat16)
    torch.cuda.synchronize()

    qwp.set_wait_timeout_ns(8)
    try:
        y = torch.zeros(M, N, dtype=torch.float32, device=DEV)
        qwp.q4k_gemm(w, x, N, out=y)
        torch.cuda.synchronize()
    finally:
        qwp.set_wait_timeout_ns(qwp.DEFAULT_WAIT_TIMEOUT_NS)

    # While the timeout is recorded, a launch skips its work.
    y2 = torch.full((M, N), 7.0, dtype=torch.float32, device=DEV)
    qwp.q4k_gemm(w, x, N, out=y2)
    torch.cuda.synchronize()
    assert bool((y2 == 7.0).all()), "a launch after a recorded timeout wrote y"

    assert qwp.device_status() == TIMEOUT
    assert qwp.device_status() == 0, "reading the status clears it"

    y3 = qwp.q4k_gemm(w, x, N).cpu().numpy()
    assert qwp.device_status() == 0
    rows = np.r_[0:128, N - 128:N]
    ref, mag = oracle.gemm(oracle.bf16_to_f64(xb), oracle.q4k_dequant(blocks.reshape(N, -1)[rows], len(rows), K))
    check_bound(y3[:, rows], ref, mag, f"after the timeout, M{M} N{N} K{K}")
