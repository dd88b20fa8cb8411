"""GPU parity of the decode-shaped path through the C ABI.

Products with 1..8 tokens, K % 256 == 0 and at least 600 (128-row tile,
256-wide super-block) items can run the decode kernel (mma.sync over operands
unpacked in registers, a stream-K split whose shared tiles are finished by the
last CTA to arrive).  By default only those where it is the faster kernel do;
these tests set the QWP_DECODE_ALWAYS policy so that every shape here (ragged
row counts, every token count) takes it, and one test checks the default choice
end to end.  Every case is compared element by element with the CPU oracle under
the same bound as the prefill path: |y - y_oracle| <= 1e-3 * sum|x*w| + 1e-5.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_weight_prefill_gb300 as qwp
import synth
from helpers import check_bound, q4k_oracle_rows, q6k_oracle_rows

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _bf16(xb):
    return torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).to(DEV).view(torch.bfloat16)


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert qwp.device_status() == 0, "a kernel reported an error"


@pytest.fixture(autouse=True)
def _decode_kernel_forced():
    prev = qwp.set_decode_policy(qwp.DECODE_ALWAYS)
    yield
    qwp.set_decode_policy(prev)


# (M, N, K): tile items = ceil(N/128) * K/256, all >= 600; N % 128 != 0 except one.
SHAPES = [(1, 2500, 8192), (2, 1700, 12288), (5, 6000, 4096), (8, 3000, 8192), (3, 9000, 4096),
          (7, 800, 24576), (4, 4096, 4864), (6, 76850, 256)]


def _items(N, K):
    return -(-N // 128) * (K // 256)


def test_decode_shapes_take_the_decode_path():
    assert all(1 <= M <= 8 and K % 256 == 0 and _items(N, K) >= 600 for M, N, K in SHAPES)
    assert all(qwp.decode_selected("q4k", M, N, K) for M, N, K in SHAPES)


@pytest.mark.parametrize("M,N,K", [(1, 65600, 512), (1, 66000, 768), (2, 65600, 512)])
def test_default_policy_both_kernels(M, N, K):
    """Under the default policy these shapes take the decode kernel; forced onto the
    prefill kernel they give results within the same bound."""
    blocks = synth.q4k_weights(N, K, seed=M * 53 + N)
    w = qwp.q4k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
    xb = synth.activations_bf16(M, K, seed=M + 11)
    ref, mag = oracle.q4k_gemm(blocks, xb, N, K)
    for policy, decode in [(qwp.DECODE_AUTO, True), (qwp.DECODE_NEVER, False)]:
        qwp.set_decode_policy(policy)
        assert qwp.decode_selected("q4k", M, N, K) == decode
        y = qwp.q4k_gemm(w, _bf16(xb), N).cpu().numpy()
        check_bound(y, ref, mag, f"policy {policy} M{M} N{N} K{K}")


@pytest.mark.parametrize("fmt,M,N,decode", [("q6k", 1, 65600, True), ("q6k", 2, 65600, True),
                                             ("q6k", 1, 24640, False), ("w4a16", 1, 65600, True),
                                             ("w4a16", 2, 65600, True), ("w4a16", 1, 24640, True),
                                             ("w4a16", 2, 24640, False)])
def test_default_policy_per_format(fmt, M, N, decode):
    """The default choice per weight format on wide matrices (K = 512 or 1536, so
    that both take at least 600 tile items): Q6_K takes the decode kernel from N =
    65536, W4A16 from N = 24576 at one token and from 65536 at two; under either
    kernel (default, then forced onto the prefill kernel) the result meets the
    bound against the oracle."""
    K, g = (512 if N > 65536 else 1536), 128
    xb = synth.activations_bf16(M, K, seed=M + 17)
    if fmt == "q6k":
        blocks = synth.q6k_weights(N, K, seed=M * 59 + N)
        w = qwp.q6k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
        ref, mag = oracle.q6k_gemm(blocks, xb, N, K)
        run = lambda: qwp.q6k_gemm(w, _bf16(xb), N)
    else:
        wq, s, z = synth.w4a16_weights(N, K, g, seed=M * 61 + N)
        wt = qwp.w4a16_repack(torch.from_numpy(wq.view(np.int32)).to(DEV))
        sd, zd = torch.from_numpy(s).to(DEV), torch.from_numpy(z).to(DEV)
        ref, mag = oracle.w4a16_gemm_bf16(wq, s, z, xb, N, K, g)
        run = lambda: qwp.w4a16_gemm_bf16(wt, sd, zd, _bf16(xb), N, g)
    for policy, expect in [(qwp.DECODE_AUTO, decode), (qwp.DECODE_NEVER, False)]:
        qwp.set_decode_policy(policy)
        assert qwp.decode_selected(fmt, M, N, K) == expect
        check_bound(run().cpu().numpy(), ref, mag, f"{fmt} policy {policy} M{M} N{N} K{K}")


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_decode_q4k_bf16(M, N, K):
    blocks = synth.q4k_weights(N, K, seed=M * 31 + N)
    w = qwp.q4k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
    xb = synth.activations_bf16(M, K, seed=M + N)
    y = qwp.q4k_gemm(w, _bf16(xb), N).cpu().numpy()
    ref, mag = oracle.q4k_gemm(blocks, xb, N, K)
    check_bound(y, ref, mag, f"decode q4k M{M} N{N} K{K}")


@pytest.mark.parametrize("M,N,K", SHAPES[:5])
def test_decode_q4k_f16(M, N, K):
    blocks = synth.q4k_weights(N, K, seed=M * 37 + N)
    w = qwp.q4k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
    xh = synth.activations_f16(M, K, seed=M + 2 * N)
    y = qwp.q4k_gemm_f16(w, torch.from_numpy(xh).to(DEV), N).cpu().numpy()
    ref, mag = oracle.gemm(oracle.half_to_f64(xh.view(np.uint16)), oracle.q4k_dequant(blocks, N, K))
    check_bound(y, ref, mag, f"decode q4k f16 M{M} N{N} K{K}")


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_decode_q6k_bf16(M, N, K):
    blocks = synth.q6k_weights(N, K, seed=M * 41 + N)
    w = qwp.q6k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
    xb = synth.activations_bf16(M, K, seed=M + 3 * N)
    y = qwp.q6k_gemm(w, _bf16(xb), N).cpu().numpy()
    ref, mag = oracle.q6k_gemm(blocks, xb, N, K)
    check_bound(y, ref, mag, f"decode q6k M{M} N{N} K{K}")


@pytest.mark.parametrize("M,N,K", [(1, 2500, 8192), (8, 3000, 8192)])
def test_decode_q6k_f16(M, N, K):
    blocks = synth.q6k_weights(N, K, seed=M * 43 + N)
    w = qwp.q6k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
    xh = synth.activations_f16(M, K, seed=M + 5 * N)
    y = qwp.q6k_gemm_f16(w, torch.from_numpy(xh).to(DEV), N).cpu().numpy()
    ref, mag = oracle.gemm(oracle.half_to_f64(xh.view(np.uint16)), oracle.q6k_dequant(blocks, N, K))
    check_bound(y, ref, mag, f"decode q6k f16 M{M} N{N} K{K}")


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("symmetric", [False, True])
@pytest.mark.parametrize("M,N,K,g", [(1, 2500, 8192, 64), (4, 5000, 4096, 128), (8, 3000, 8192, 256),
                                     (7, 800, 24576, 128)])
def test_decode_w4a16(M, N, K, g, symmetric, bf16):
    wq, s, z = synth.w4a16_weights(N, K, g, seed=M * 47 + N + K)
    wt = qwp.w4a16_repack(torch.from_numpy(wq.view(np.int32)).to(DEV))
    sd = torch.from_numpy(s).to(DEV)
    zd = None if symmetric else torch.from_numpy(z).to(DEV)
    zo = None if symmetric else z
    if bf16:
        xb = synth.activations_bf16(M, K, seed=M + 7)
        y = qwp.w4a16_gemm_bf16(wt, sd, zd, _bf16(xb), N, g).cpu().numpy()
        ref, mag = oracle.w4a16_gemm_bf16(wq, s, zo, xb, N, K, g)
    else:
        xh = synth.activations_f16(M, K, seed=M + 7)
        y = qwp.w4a16_gemm(wt, sd, zd, torch.from_numpy(xh).to(DEV), N, g).cpu().numpy()
        ref, mag = oracle.w4a16_gemm(wq, s, zo, xh, N, K, g)
    check_bound(y, ref, mag, f"decode w4a16 sym={symmetric} bf16={bf16} M{M} N{N} K{K} g{g}")


@pytest.mark.parametrize("M", [1, 8])
@pytest.mark.parametrize("name,K,N", synth.QWEN3_8B_LAYER)
def test_decode_qwen3_8b_layer(M, name, K, N):
    """Every element of every layer projection at one and at eight tokens (o, with 512 tile
    items, takes the prefill kernel; the others the decode kernel)."""
    blocks = synth.q4k_weights(N, K, seed=K + N + M)
    w = qwp.q4k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
    xb = synth.activations_bf16(M, K, seed=M + 99)
    y = qwp.q4k_gemm(w, _bf16(xb), N).cpu().numpy()
    ref, mag = q4k_oracle_rows(blocks, xb, N, K)
    check_bound(y, ref, mag, f"decode q4k {name} M{M}")


@pytest.mark.parametrize("M,K,N", [(1, 12288, 4096), (8, 12288, 4096)])
def test_decode_q6k_projections(M, K, N):
    blocks = synth.q6k_weights(N, K, seed=K + N + M)
    w = qwp.q6k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
    xb = synth.activations_bf16(M, K, seed=M + 98)
    y = qwp.q6k_gemm(w, _bf16(xb), N).cpu().numpy()
    ref, mag = q6k_oracle_rows(blocks, xb, N, K)
    check_bound(y, ref, mag, f"decode q6k M{M} N{N} K{K}")


def test_decode_bf16_overflow_is_reported():
    """An activation beyond fp16's range, converted inside the decode kernel, is reported
    as QWP_ERR_RANGE; the next call is clean."""
    M, N, K = 4, 2500, 8192
    blocks = synth.q4k_weights(N, K, seed=5)
    w = qwp.q4k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
    xb = synth.activations_bf16(M, K, seed=6).copy()
    xb[2, 3000] = 0x4880  # bf16 262144.0
    qwp.q4k_gemm(w, _bf16(xb), N)
    assert qwp.device_status() == -7
    xb[2, 3000] = 0x3F80
    y = qwp.q4k_gemm(w, _bf16(xb), N).cpu().numpy()
    assert qwp.device_status() == 0
    ref, mag = oracle.q4k_gemm(blocks, xb, N, K)
    check_bound(y, ref, mag, "decode after a range error")


def test_decode_split_k_is_deterministic():
    """Shared tiles are summed in CTA order: repeated calls agree bit for bit."""
    M, N, K = 8, 1600, 12288
    blocks = synth.q4k_weights(N, K, seed=8)
    w = qwp.q4k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
    x = _bf16(synth.activations_bf16(M, K, seed=9))
    y0 = qwp.q4k_gemm(w, x, N).clone()
    for _ in range(5):
        assert torch.equal(qwp.q4k_gemm(w, x, N), y0)


def test_decode_leaves_other_tokens_untouched():
    """Only the M token rows of y are written (the kernel computes 8 token columns)."""
    M, N, K = 3, 2500, 8192
    blocks = synth.q4k_weights(N, K, seed=10)
    w = qwp.q4k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
    xb = synth.activations_bf16(M, K, seed=11)
    guard = torch.full((M + 5, N), 7.0, device=DEV)
    qwp.q4k_gemm(w, _bf16(xb), N, out=guard[:M])
    assert torch.all(guard[M:] == 7.0)
    ref, mag = oracle.q4k_gemm(blocks, xb, N, K)
    check_bound(guard[:M].cpu().numpy(), ref, mag, "decode guard")
