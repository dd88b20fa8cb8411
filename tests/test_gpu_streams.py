"""Stream-ordered scratch and launch chaining.

bf16-activation prefill calls and decode-shaped calls take their scratch from a
stream-ordered pool (a block freed after one call may be the next call's block),
and every kernel is launched with programmatic stream serialization, so it may
start while the kernel before it still runs.  Checked here against the oracle:
calls alternating between two streams with different shapes and kernels (prefill
and decode), back-to-back calls on one stream that each overwrite an fp16 copy of
x the call before them read, and a captured graph replayed between eager calls
on its stream.
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


def _case(M, N, K, seed):
    blocks = synth.q4k_weights(N, K, seed=seed)
    w = qwp.q4k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
    xb = synth.activations_bf16(M, K, seed=seed + 1)
    x = torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).to(DEV).view(torch.bfloat16)
    ref, mag = oracle.q4k_gemm(blocks, xb, N, K)
    return w, x, ref, mag


def test_two_streams_alternating_with_growing_scratch():
    cases = [_case(64, 512, 1024, 11), _case(300, 384, 4096, 12), _case(1, 70000, 512, 13), _case(200, 640, 2048, 14)]
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    torch.cuda.synchronize()
    for rep in range(3):
        for i, (w, x, _, _) in enumerate(cases):
            s = s1 if (i + rep) % 2 == 0 else s2
            with torch.cuda.stream(s):
                y = torch.empty(x.shape[0], w.numel() // (x.shape[1] // 256 * 144), dtype=torch.float32, device=DEV)
                qwp.q4k_gemm(w, x, y.shape[1], out=y)
                outs.append((i, y))
    torch.cuda.synchronize()
    for i, y in outs:
        _, _, ref, mag = cases[i]
        check_bound(y.cpu().numpy(), ref, mag, f"case {i}")


def test_back_to_back_calls_reuse_the_block_in_order():
    """Each call's conversion overwrites the stream's fp16 copy of x that the call
    before it reads: 16 calls alternating two inputs, every result checked."""
    a = _case(105, 4096, 4096, 21)
    b = _case(105, 4096, 4096, 23)
    ys = []
    for i in range(16):
        w, x, _, _ = a if i % 2 == 0 else b
        ys.append(qwp.q4k_gemm(w, x, 4096))
    torch.cuda.synchronize()
    for i, y in enumerate(ys):
        _, _, ref, mag = a if i % 2 == 0 else b
        check_bound(y.cpu().numpy(), ref, mag, f"call {i}")


def test_graph_replayed_between_eager_calls():
    w1, x1, ref1, mag1 = _case(105, 6144, 4096, 31)
    w2, x2, ref2, mag2 = _case(105, 2048, 4096, 33)
    s = torch.cuda.Stream()
    y1 = torch.empty(105, 6144, dtype=torch.float32, device=DEV)
    with torch.cuda.stream(s):
        qwp.q4k_gemm(w1, x1, 6144, out=y1)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        qwp.q4k_gemm(w1, x1, 6144, out=y1)
    y2 = torch.empty(105, 2048, dtype=torch.float32, device=DEV)
    with torch.cuda.stream(s):
        for _ in range(3):
            y1.zero_()
            g.replay()
            qwp.q4k_gemm(w2, x2, 2048, out=y2)
    s.synchronize()
    check_bound(y1.cpu().numpy(), ref1, mag1, "graph")
    check_bound(y2.cpu().numpy(), ref2, mag2, "eager")
