"""Every launch plan of the prefill kernel against the oracle, through the C ABI.

The planner picks a split-K factor S (the cluster size: S CTAs each reduce a
K range of every unit and sum the partials through distributed shared memory)
and the number of clusters; with more units than clusters each cluster loops
over several units, which changes how the partials are handed over (a partial
buffer of its own, the last unit through the idle rings).  The shapes below are
chosen so that, on GB300, every factor the planner uses occurs with one unit per
cluster and with several (qwp_gemm_plan reports the plan); each is compared with
the oracle on all tokens and a sample of weight rows (first, last and random
128-row tiles, so that every split of every sampled unit is checked), under
|y - y_oracle| <= 1e-3 * sum|x*w| + 1e-5.
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

# (M, N, K): found with the planner's cost model and GB300's resident-cluster counts.
SHAPES = [(16, 10112, 1024), (16, 29312, 1024), (16, 4736, 1024), (16, 23168, 1024), (16, 4736, 2048),
          (16, 10112, 2048), (16, 128, 1024), (16, 19712, 1024), (16, 3200, 8192), (16, 6272, 8192),
          (16, 2048, 4096), (16, 14720, 12288), (16, 128, 2048), (105, 24576, 4096), (105, 4096, 12288),
          (100, 1000, 8192), (128, 2500, 4096)]


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert qwp.device_status() == 0, "a kernel reported an error"


def test_shapes_cover_every_split_factor():
    keys = set()
    for M, N, K in SHAPES:
        p = qwp.gemm_plan("q4k", M, N, K)
        assert p["kernel"] == "prefill" and p["units"] == -(-N // 128) * -(-M // p["token_tile"])
        assert p["splits"] * p["clusters"] <= 152 and p["units_per_cluster"] == -(-p["units"] // p["clusters"])
        keys.add((p["splits"], p["units_per_cluster"] > 1))
    assert {(1, False), (1, True), (2, False), (2, True), (3, False), (3, True), (4, False), (4, True),
            (6, False), (6, True), (8, False)} <= keys, sorted(keys)


def _weight_rows(N: int, seed: int) -> np.ndarray:
    """First and last 128-row tiles and up to six random tiles in between."""
    tiles = -(-N // 128)
    pick = {0, tiles - 1}
    if tiles > 2:
        rng = np.random.default_rng(seed)
        pick |= set(rng.choice(np.arange(1, tiles - 1), size=min(6, tiles - 2), replace=False).tolist())
    rows = np.concatenate([np.arange(128 * t, min(N, 128 * t + 128)) for t in sorted(pick)])
    return rows


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_plan_parity(M, N, K):
    blocks = synth.q4k_weights(N, K, seed=M + N + K)
    w = qwp.q4k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
    xb = synth.activations_bf16(M, K, seed=N + 3)
    x = torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).to(DEV).view(torch.bfloat16)
    y = qwp.q4k_gemm(w, x, N).cpu().numpy()
    rows = _weight_rows(N, seed=K)
    ref, mag = oracle.gemm(oracle.bf16_to_f64(xb), oracle.q4k_dequant(blocks.reshape(N, -1)[rows], len(rows), K))
    plan = qwp.gemm_plan("q4k", M, N, K)
    check_bound(y[:, rows], ref, mag, f"M{M} N{N} K{K} plan {plan}")
