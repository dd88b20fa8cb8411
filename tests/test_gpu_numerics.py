"""GPU parity on the method's numerical edge cases, against the CPU oracle.

The workload's bound is per output element: |y - y_oracle| <= 1e-3 * sum_k|x_k*w_k| + 1e-5.
A weight whose two terms cancel (Q4_K d*sc*q close to dmin*m) leaves a tiny
sum_k|x*w|, so the tensor-core operand has to be the fp16 rounding of the exact
weight, not of its terms.  These cases are built so that any rounding of a term
(rather than of the weight) adds up coherently over K and breaks the bound:
  * Q4_K blocks with d == dmin and sc_j == m_j: nibbles of 1 give w == 0 exactly
    (y must be exactly 0); nibbles mostly 1 with dmin one fp16 step above d give
    weights a few units of d's last place wide next to full-size ones;
  * Q4_K blocks with subnormal, tiny and large d / dmin;
  * Q6_K blocks whose d*scale and d*scale*(q - 32) both round up by close to
    half a unit in the last place (two fp16 roundings would double the error);
  * W4A16 scales across fp16's range (subnormal to ~4000).
All-positive activations make the errors of every term line up.  Each case runs
on the prefill kernel (tokens >= 9) and on the decode kernel (1..8 tokens, policy
ALWAYS), whose operands are built by the same unpack.
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
    assert qwp.device_status() == 0, "a kernel reported a timeout or a range error"


@pytest.fixture
def decode_always():
    prev = qwp.set_decode_policy(qwp.DECODE_ALWAYS)
    yield
    qwp.set_decode_policy(prev)


def _bf16_on_gpu(xb):
    return torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).to(DEV).view(torch.bfloat16)


def _positive_bf16(M, K, seed):
    """|N(0,1)| activations as bf16 bits: every x_k > 0 (or +0), so errors of one sign add up."""
    return synth.activations_bf16(M, K, seed) & np.uint16(0x7FFF)


def _fp16_bits(v):
    return np.asarray(v, np.float64).astype(np.float16).view(np.uint16)


# --- Q4_K blocks with mirrored scale bytes -------------------------------------------

def _q4k_mirrored_blocks(N, K, seed, d_bits, dmin_bits, nibbles):
    """Q4_K rows whose packed scale bytes give sc_j == m_j for every sub-block: bytes
    4..7 repeat bytes 0..3 (the low six bits of sc_0..3 / m_0..3 and the top two bits
    of sc_4..7 / m_4..7) and bytes 8..11 hold equal nibbles (the low four bits of
    sc_4..7 / m_4..7).  d_bits, dmin_bits: fp16 bits per block; nibbles [blocks, 256]
    in K order (element 64c+l of a block in the low nibble of byte 32c+l for l < 32,
    in the high nibble of byte 32c+l-32 otherwise)."""
    nb = N * (K // 256)
    rng = np.random.default_rng(seed)
    blk = np.zeros((nb, 144), np.uint8)
    blk[:, 0:2] = np.asarray(d_bits, np.uint16).astype("<u2").view(np.uint8).reshape(nb, 2)
    blk[:, 2:4] = np.asarray(dmin_bits, np.uint16).astype("<u2").view(np.uint8).reshape(nb, 2)
    lo6 = rng.integers(1, 256, size=(nb, 4), dtype=np.uint8)
    blk[:, 4:8] = lo6
    blk[:, 8:12] = lo6
    nib = rng.integers(1, 16, size=(nb, 4), dtype=np.uint8)
    blk[:, 12:16] = nib | (nib << 4)
    q = np.asarray(nibbles, np.uint8).reshape(nb, 4, 64)
    blk[:, 16:] = (q[:, :, :32] | (q[:, :, 32:] << 4)).reshape(nb, 128)
    for b in range(min(nb, 8)):  # the construction really gives sc_j == m_j (decoded by the oracle)
        for j in range(8):
            sc, m = oracle.q4k_scale_min(blk[b, 4:16], j)
            assert sc == m
    return blk.reshape(N, -1)


def _run_q4k(blocks, xb, N, K):
    w = qwp.q4k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
    y = qwp.q4k_gemm(w, _bf16_on_gpu(xb), N).cpu().numpy()
    ref, mag = oracle.q4k_gemm(blocks, xb, N, K)
    return y, ref, mag


SHAPES = [(105, 1000, 2048), (40, 136, 512)]
DECODE_SHAPES = [(1, 4864, 4096), (5, 4864, 4096)]  # 38 row tiles x 16 super-blocks = 608 items


def _q4k_exact_cancel(N, K, seed):
    nb = N * (K // 256)
    rng = np.random.default_rng(seed)
    d = _fp16_bits(rng.uniform(1e-3, 4e-3, nb))
    return _q4k_mirrored_blocks(N, K, seed, d, d, np.ones((nb, 256), np.uint8))


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_q4k_exact_cancellation_gives_zero(M, N, K):
    """d == dmin, sc_j == m_j, every nibble 1: every weight is exactly 0, so y is 0."""
    blocks = _q4k_exact_cancel(N, K, seed=M + N)
    assert not oracle.q4k_dequant(blocks, N, K).any()
    for xb in (_positive_bf16(M, K, seed=11), synth.activations_bf16(M, K, seed=12)):
        y, ref, mag = _run_q4k(blocks, xb, N, K)
        assert not ref.any() and not mag.any()
        assert np.array_equal(y, np.zeros_like(y)), f"max |y| {np.abs(y).max():.3g} for an all-zero W"


@pytest.mark.parametrize("M,N,K", DECODE_SHAPES)
def test_q4k_exact_cancellation_gives_zero_decode(M, N, K, decode_always):
    assert qwp.decode_selected("q4k", M, N, K)
    blocks = _q4k_exact_cancel(N, K, seed=M + N)
    y, ref, mag = _run_q4k(blocks, _positive_bf16(M, K, seed=13), N, K)
    assert not ref.any()
    assert np.array_equal(y, np.zeros_like(y)), f"max |y| {np.abs(y).max():.3g} for an all-zero W"


def _q4k_near_cancel(N, K, seed):
    """dmin one fp16 step above d, sc_j == m_j, nibbles 1 with probability 0.9 else 0 or
    2: w = sc*(d*q - dmin) is -sc*ulp(d) at q = 1, about +-d*sc elsewhere."""
    nb = N * (K // 256)
    rng = np.random.default_rng(seed)
    d = _fp16_bits(rng.uniform(1e-3, 4e-3, nb))
    dmin = d + np.uint16(1)
    q = np.where(rng.random((nb, 256)) < 0.9, 1, rng.choice([0, 2], size=(nb, 256))).astype(np.uint8)
    return _q4k_mirrored_blocks(N, K, seed, d, dmin, q)


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_q4k_near_cancellation_within_bound(M, N, K):
    blocks = _q4k_near_cancel(N, K, seed=3 * M + N)
    for xb in (_positive_bf16(M, K, seed=21), synth.activations_bf16(M, K, seed=22)):
        y, ref, mag = _run_q4k(blocks, xb, N, K)
        r = check_bound(y, ref, mag, f"q4k near-cancel M{M} N{N} K{K}")
        print(f"worst err/bound {r:.3f}")


@pytest.mark.parametrize("M,N,K", DECODE_SHAPES)
def test_q4k_near_cancellation_within_bound_decode(M, N, K, decode_always):
    blocks = _q4k_near_cancel(N, K, seed=3 * M + N)
    y, ref, mag = _run_q4k(blocks, _positive_bf16(M, K, seed=23), N, K)
    check_bound(y, ref, mag, f"q4k near-cancel decode M{M} N{N} K{K}")


# fp16 bit patterns: smallest subnormal, largest subnormal, smallest normal, 2^-10,
# 1.0, 60.0 (d*15*63 stays below 65504), and for dmin also 900.0 (dmin*63 < 65504).
D_SPECIAL = np.array([0x0001, 0x03FF, 0x0400, 0x1400, 0x3C00, 0x5380], np.uint16)
DMIN_SPECIAL = np.array([0x0000, 0x0001, 0x03FF, 0x0400, 0x1400, 0x3C00, 0x5380, 0x6308], np.uint16)


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_q4k_extreme_d_dmin_within_bound(M, N, K):
    blocks = synth.q4k_weights(N, K, seed=M + 5).reshape(-1, 144).copy()
    rng = np.random.default_rng(M + 6)
    nb = blocks.shape[0]
    blocks[:, 0:2] = rng.choice(D_SPECIAL, nb).astype("<u2").view(np.uint8).reshape(nb, 2)
    blocks[:, 2:4] = rng.choice(DMIN_SPECIAL, nb).astype("<u2").view(np.uint8).reshape(nb, 2)
    blocks = blocks.reshape(N, -1)
    assert np.abs(oracle.q4k_dequant(blocks, N, K)).max() < 65504
    for xb in (_positive_bf16(M, K, seed=31), synth.activations_bf16(M, K, seed=32)):
        y, ref, mag = _run_q4k(blocks, xb, N, K)
        check_bound(y, ref, mag, f"q4k extreme d/dmin M{M} N{N} K{K}")


# --- Q6_K: both roundings of a two-step operand pushed up ------------------------------

def _q6k_adversarial(N, K, seed, d_lo, d_hi):
    """Q6_K rows with d, scale and codes chosen so that RN16(d*scale) and
    RN16(RN16(d*scale)*(q - 32)) both round up by more than 0.3 of a unit in the
    last place; all weights positive (q > 32, scale > 0)."""
    rng = np.random.default_rng(seed)
    d_cand = np.unique(_fp16_bits(rng.uniform(d_lo, d_hi, 4096)))
    d_val = d_cand.view(np.float16).astype(np.float64)
    sc = np.arange(1, 128, dtype=np.float64)
    prod = d_val[:, None] * sc[None, :]
    r1 = prod.astype(np.float16).astype(np.float64)
    ulp1 = np.spacing(np.abs(r1).astype(np.float16)).astype(np.float64)
    up1 = (r1 - prod) / ulp1
    qc = np.arange(1, 32, dtype=np.float64)
    picks = []
    for i, j in zip(*np.nonzero(up1 > 0.3)):
        t = r1[i, j] * qc
        r2 = t.astype(np.float16).astype(np.float64)
        ulp2 = np.spacing(r2.astype(np.float16)).astype(np.float64)
        good = qc[(r2 - t) / ulp2 > 0.3]
        if good.size:
            picks.append((d_cand[i], int(sc[j]), good.astype(np.int64)))
    assert len(picks) >= 16, "not enough adversarial (d, scale) pairs"
    nb = N * (K // 256)
    choice = rng.integers(0, len(picks), nb)
    codes = np.empty((nb, 256), np.int64)
    for i, (_, _, goodq) in enumerate(picks):
        sel = choice == i
        codes[sel] = 32 + rng.choice(goodq, size=(int(sel.sum()), 256))  # 6-bit codes 33..63
    # GGML Q6_K: element 128h + 32j + l keeps its low four bits in nibble j//2 of
    # ql[64h + l + 32(j%2)] and its high two bits at bits 2j of qh[32h + l]
    ql = np.zeros((nb, 128), np.int64)
    qh = np.zeros((nb, 64), np.int64)
    for e in range(256):
        h, j, l = e >> 7, (e >> 5) & 3, e & 31
        ql[:, 64 * h + l + 32 * (j & 1)] |= (codes[:, e] & 15) << (4 * (j >> 1))
        qh[:, 32 * h + l] |= (codes[:, e] >> 4) << (2 * j)
    blk = np.zeros((nb, 210), np.uint8)
    blk[:, 0:128] = ql
    blk[:, 128:192] = qh
    blk[:, 192:208] = np.array([picks[c][1] for c in choice], np.uint8)[:, None]
    blk[:, 208:210] = np.array([picks[c][0] for c in choice], np.uint16).astype("<u2").view(np.uint8).reshape(nb, 2)
    for e in range(256):  # the construction gives the intended codes (read back by the oracle)
        assert oracle.q6k_code(blk[0], e) == codes[0, e]
    blocks = blk.reshape(N, -1)
    assert (oracle.q6k_dequant(blocks[:8], 8, K) > 0).all()
    return blocks


def _run_q6k(blocks, xb, N, K):
    w = qwp.q6k_repack(torch.from_numpy(blocks.reshape(-1)).to(DEV), N, K)
    y = qwp.q6k_gemm(w, _bf16_on_gpu(xb), N).cpu().numpy()
    ref, mag = oracle.q6k_gemm(blocks, xb, N, K)
    return y, ref, mag


@pytest.mark.parametrize("d_lo,d_hi", [(2.0 ** -9, 2.0 ** -7), (1e-5, 6e-5)])
@pytest.mark.parametrize("M,N,K", [(105, 264, 2048), (2, 4864, 4096)])
def test_q6k_adversarial_rounding_within_bound(M, N, K, d_lo, d_hi):
    prev = qwp.set_decode_policy(qwp.DECODE_ALWAYS)
    try:
        blocks = _q6k_adversarial(N, K, seed=M + N, d_lo=d_lo, d_hi=d_hi)
        y, ref, mag = _run_q6k(blocks, _positive_bf16(M, K, seed=41), N, K)
    finally:
        qwp.set_decode_policy(prev)
    r = check_bound(y, ref, mag, f"q6k adversarial M{M} N{N} K{K} d in [{d_lo:.2g}, {d_hi:.2g}]")
    print(f"worst err/bound {r:.3f}")
    # one rounding of each weight (relative <= 2^-11) leaves the error below half the bound
    assert r < 0.6


# --- W4A16 across fp16's scale range ---------------------------------------------------

@pytest.mark.parametrize("symmetric", [False, True])
@pytest.mark.parametrize("M,N,K", [(105, 264, 1024), (1, 4864, 4096)])
def test_w4a16_extreme_scales_within_bound(M, N, K, symmetric):
    g = 128
    wq, s, z = synth.w4a16_weights(N, K, g, seed=M + 51)
    rng = np.random.default_rng(M + 52)
    # subnormal, smallest normal, around one, and up to 4000 (s * 15 < 65504)
    pool = np.array([2.0 ** -24, 3 * 2.0 ** -24, 2.0 ** -14, 0.37, 1.0, 97.0, 1500.0, 4000.0])
    s = rng.choice(pool, size=s.shape).astype(np.float16)
    zd = None if symmetric else torch.from_numpy(z).to(DEV)
    wt = qwp.w4a16_repack(torch.from_numpy(wq.view(np.int32)).to(DEV))
    xh = np.abs(synth.activations_f16(M, K, seed=M + 53))
    prev = qwp.set_decode_policy(qwp.DECODE_ALWAYS)
    try:
        y = qwp.w4a16_gemm(wt, torch.from_numpy(s).to(DEV), zd, torch.from_numpy(xh).to(DEV), N, g).cpu().numpy()
    finally:
        qwp.set_decode_policy(prev)
    ref, mag = oracle.w4a16_gemm(wq, s, None if symmetric else z, xh, N, K, g)
    check_bound(y, ref, mag, f"w4a16 extreme scales M{M} N{N} K{K} sym={symmetric}")
