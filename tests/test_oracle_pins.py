"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each test cites what it pins:
  * exhaustive IEEE decodes against numpy's independent conversions,
  * hand-built blocks whose values are worked out by hand from the pages
    (tests/golden/*.json, each case with its citation),
  * closed forms of the GEMM (unit vectors, one sub-block of ones),
  * brute force against numpy's float64 matmul at tiny shapes,
  * the bijection of the 96 packed scale bits onto sixteen 6-bit values.
A plausible slip in the oracle (a dropped term, a wrong sign, a swapped
nibble, a transposed operand, a wrong block offset) fails at least one.
"""
import json
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rle(pairs):
    out = []
    for v, c in pairs:
        out.extend([float(v)] * int(c))
    return np.array(out, np.float64)


def _q4k_block(spec):
    blk = np.zeros(144, np.uint8)
    d = int(spec["d"], 16)
    dmin = int(spec["dmin"], 16)
    blk[0], blk[1] = d & 255, d >> 8
    blk[2], blk[3] = dmin & 255, dmin >> 8
    blk[4:16] = np.frombuffer(bytes.fromhex(spec["scales"]), np.uint8)
    blk[16:144] = int(spec["qs_fill"], 16)
    for idx, val in spec["qs_set"].items():
        blk[16 + int(idx)] = int(val, 16)
    return blk


def _q4k_cases():
    with open(os.path.join(GOLDEN, "q4k_handbuilt.json")) as f:
        return json.load(f)["cases"]


def _q6k_block(spec):
    blk = np.zeros(210, np.uint8)
    blk[0:128] = int(spec["ql_fill"], 16)
    blk[128:192] = int(spec["qh_fill"], 16)
    for idx, val in spec["ql_set"].items():
        blk[int(idx)] = int(val, 16)
    for idx, val in spec["qh_set"].items():
        blk[128 + int(idx)] = int(val, 16)
    blk[192:208] = np.frombuffer(bytes.fromhex(spec["scales"]), np.uint8)
    d = int(spec["d"], 16)
    blk[208], blk[209] = d & 255, d >> 8
    return blk


def _q6k_cases():
    with open(os.path.join(GOLDEN, "q6k_handbuilt.json")) as f:
        return json.load(f)["cases"]


def _w4a16_cases():
    with open(os.path.join(GOLDEN, "w4a16_handbuilt.json")) as f:
        return json.load(f)["cases"]


# --- exact decodes ---------------------------------------------------------------

def test_half_decode_exhaustive():
    """All 65536 binary16 patterns against numpy's float16 -> float64 conversion."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.half_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zero is kept
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_bf16_decode_exhaustive():
    """All 65536 bfloat16 patterns: bf16 is the top half of an IEEE binary32."""
    bits = np.arange(65536, dtype=np.uint32)
    ours = oracle.bf16_to_f64(bits.astype(np.uint16))
    with np.errstate(invalid="ignore"):
        ref = (bits << 16).view(np.float32).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


# --- Q4_K dequant -----------------------------------------------------------------

@pytest.mark.parametrize("case", _q4k_cases(), ids=lambda c: c["name"])
def test_q4k_handbuilt_blocks(case):
    N, K = case["N"], case["K"]
    blocks = np.concatenate([_q4k_block(b) for b in case["blocks"]])
    w = oracle.q4k_dequant(blocks, N, K)
    for n in range(N):
        expect = _rle(case["expect"][n])
        assert expect.size == K
        assert np.array_equal(w[n], expect), case["source"]


def test_q4k_scale_bits_are_a_bijection():
    """Each of the 96 packed bits reaches exactly one 6-bit (scale or min) value, as one bit.

    Sixteen 6-bit values in 12 bytes leave no spare bit, so the unpack must be a
    permutation of bits: a dropped, duplicated or mis-shifted term breaks this.
    """
    hits = {}
    for byte in range(12):
        for bit in range(8):
            s = np.zeros(12, np.uint8)
            s[byte] = 1 << bit
            nonzero = []
            for j in range(8):
                sc, m = oracle.q4k_scale_min(s, j)
                for kind, v in (("sc", sc), ("m", m)):
                    if v:
                        nonzero.append((kind, j, v))
            assert len(nonzero) == 1, (byte, bit, nonzero)
            kind, j, v = nonzero[0]
            assert v & (v - 1) == 0 and v < 64
            key = (kind, j, v.bit_length() - 1)
            assert key not in hits
            hits[key] = (byte, bit)
    assert len(hits) == 96


def test_q4k_low_six_bits_for_first_four_subblocks():
    """Sub-blocks 0..3: scale = low 6 bits of bytes 0..3, min = low 6 bits of bytes 4..7."""
    s = np.array([0xC5, 0x3F, 0x40, 0x81, 0x12, 0xE7, 0x00, 0x7F, 0, 0, 0, 0], np.uint8)
    expect = [(0x05, 0x12), (0x3F, 0x27), (0x00, 0x00), (0x01, 0x3F)]
    for j in range(4):
        assert oracle.q4k_scale_min(s, j) == expect[j]


def test_q4k_random_values_in_range_and_exact_form():
    """Random blocks: every weight equals d*sc*q - dmin*m for some sc, m in 0..63, q in 0..15."""
    N, K = 3, 512
    blocks = synth.q4k_weights(N, K, seed=11)
    w = oracle.q4k_dequant(blocks, N, K)
    raw = blocks.reshape(N, K // 256, 144)
    d = raw[:, :, 0:2].copy().view("<u2")[..., 0].view(np.float16).astype(np.float64)
    dmin = raw[:, :, 2:4].copy().view("<u2")[..., 0].view(np.float16).astype(np.float64)
    for n in range(N):
        for b in range(K // 256):
            sub = w[n, 256 * b:256 * (b + 1)].reshape(8, 32)
            for j in range(8):
                sc, m = oracle.q4k_scale_min(raw[n, b, 4:16], j)
                q = (sub[j] + dmin[n, b] * m) / (d[n, b] * sc) if sc else None
                if q is not None:
                    assert np.allclose(q, np.round(q), atol=1e-9)
                    assert q.min() >= -1e-9 and q.max() <= 15 + 1e-9
                else:
                    assert np.all(sub[j] == -dmin[n, b] * m)


def test_q4k_rejects_bad_shape():
    with pytest.raises(ValueError):
        oracle.q4k_dequant(np.zeros(144, np.uint8), 1, 128)


# --- Q6_K dequant -----------------------------------------------------------------

@pytest.mark.parametrize("case", _q6k_cases(), ids=lambda c: c["name"])
def test_q6k_handbuilt_blocks(case):
    N, K = case["N"], case["K"]
    blocks = np.concatenate([_q6k_block(b) for b in case["blocks"]])
    w = oracle.q6k_dequant(blocks, N, K)
    for n in range(N):
        expect = _rle(case["expect"][n])
        assert expect.size == K
        assert np.array_equal(w[n], expect), case["source"]


def test_q6k_code_bits_are_a_bijection():
    """Each of the 1536 code bits (ql, qh) reaches exactly one weight, as one power of two.

    256 six-bit codes in 192 bytes leave no spare bit, so the decode must be a
    permutation of bits with bit weights 1..32: a dropped, duplicated, mis-shifted
    or mis-indexed term breaks this.  Low-nibble bytes must give weights 1..8, qh
    bytes weights 16 and 32.
    """
    base = np.zeros(210, np.uint8)
    base[192:208] = 1        # every scale 1
    base[208:210] = (0x00, 0x3C)  # d = 1.0
    w0 = oracle.q6k_dequant(base, 1, 256)[0]
    assert np.array_equal(w0, np.full(256, -32.0))
    hits = set()
    for byte in range(192):
        for bit in range(8):
            blk = base.copy()
            blk[byte] = 1 << bit
            diff = oracle.q6k_dequant(blk, 1, 256)[0] - w0
            nz = np.flatnonzero(diff)
            assert nz.size == 1, (byte, bit, nz)
            v = diff[nz[0]]
            assert v > 0 and v == 2.0 ** round(np.log2(v)) and v <= 32, (byte, bit, v)
            k = int(round(np.log2(v)))
            assert (k < 4) == (byte < 128), (byte, bit, k)
            key = (int(nz[0]), k)
            assert key not in hits
            hits.add(key)
    assert len(hits) == 1536


def test_q6k_each_scale_covers_16_consecutive_weights():
    """Scale byte s multiplies exactly elements 16s..16s+15 (one-hot scales, codes 0)."""
    for s in range(16):
        blk = np.zeros(210, np.uint8)
        blk[192 + s] = 3
        blk[208:210] = (0x00, 0x3C)
        w = oracle.q6k_dequant(blk, 1, 256)[0]
        nz = np.flatnonzero(w)
        assert np.array_equal(nz, np.arange(16 * s, 16 * s + 16))
        assert np.all(w[nz] == -96.0)  # 1 * 3 * (0 - 32)


def test_q6k_code_accessor_matches_dequant_and_covers_all_codes():
    """Random blocks: the one-code accessor agrees with the dequant, and with d = 1 and
    unit scales every code 0..63 appears (uniform random bytes)."""
    blk = synth.q6k_weights(1, 256, seed=3).reshape(210).copy()
    blk[192:208] = 1
    blk[208:210] = (0x00, 0x3C)
    w = oracle.q6k_dequant(blk, 1, 256)[0]
    codes = np.array([oracle.q6k_code(blk, e) for e in range(256)])
    assert np.array_equal(w, codes - 32.0)
    many = synth.q6k_weights(64, 256, seed=4).copy()
    many[:, 192:208] = 1
    many[:, 208:210] = (0x00, 0x3C)
    allw = oracle.q6k_dequant(many, 64, 256)
    assert set(np.unique(allw + 32).astype(int)) == set(range(64))


def test_q6k_gemm_closed_form_one_hot_and_ones():
    """x = e_k picks column k of W; x = ones sums a row (one_scale_per_16: sum = 128)."""
    case = {c["name"]: c for c in _q6k_cases()}["one_scale_per_16_weights"]
    blk = _q6k_block(case["blocks"][0])
    x = np.zeros((2, 256), np.float32)
    x[0, 37] = 1.0
    x[1, :] = 1.0
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)  # exact: 0 and 1 are bf16
    y, a = oracle.q6k_gemm(blk, xb, 1, 256)
    assert y[0, 0] == -3.0         # element 37 is in sub-block 2 (scale 3): w = -sc = -3
    assert y[1, 0] == 128.0        # -(1 - 2 + 3 - ... - 16) * 16 = 128
    assert a[1, 0] == 16.0 * sum(range(1, 17))


def test_q6k_rejects_bad_shape():
    with pytest.raises(ValueError):
        oracle.q6k_dequant(np.zeros(210, np.uint8), 1, 300)


# --- W4A16 dequant ----------------------------------------------------------------

@pytest.mark.parametrize("case", _w4a16_cases(), ids=lambda c: c["name"])
def test_w4a16_handbuilt(case):
    K, g = case["K"], case["group"]
    words = np.full(K // 8, int(case["words_fill"], 16), np.uint32)
    for i, wv in enumerate(case["words"]):
        words[i] = int(wv, 16)
    scales = np.array([int(s, 16) for s in case["scales"]], np.uint16)
    zeros = np.array(case["zeros"], np.uint8)
    w = oracle.w4a16_dequant(words[None], scales[None], zeros[None], 1, K, g)
    assert np.array_equal(w[0], _rle(case["expect"])), case["source"]


def test_w4a16_symmetric_handbuilt():
    """zeros=None is the symmetric form w = s*(q - 8).  Word 0x76543210 holds, in K order,
    the codes 0,4,1,5,2,6,3,7 (val[2p] at bits 4p, val[2p+1] at bits 16+4p), worked by hand."""
    K, g = 64, 64
    words = np.full(K // 8, 0x88888888, np.uint32)  # code 8 everywhere: w = 0
    words[0] = 0x76543210
    words[7] = 0xFFFF0000  # elements 56..63: codes 0,15,0,15,0,15,0,15
    for sbits, s in ((0x3C00, 1.0), (0x3800, 0.5)):
        w = oracle.w4a16_dequant(words[None], np.array([[sbits]], np.uint16), None, 1, K, g)[0]
        expect = np.zeros(K)
        expect[0:8] = s * (np.array([0, 4, 1, 5, 2, 6, 3, 7]) - 8)
        expect[56:64] = s * (np.array([0, 15, 0, 15, 0, 15, 0, 15]) - 8)
        assert np.array_equal(w, expect)


def test_w4a16_bf16_gemm_one_hot():
    """bf16 activations: x = e_k picks column k of W; x = 2^-3 scales it exactly."""
    N, K, g = 3, 128, 64
    wq, s, z = synth.w4a16_weights(N, K, g, seed=11)
    w = oracle.w4a16_dequant(wq, s, z, N, K, g)
    for k in (0, 37, 127):
        xb = np.zeros((1, K), np.uint16)
        xb[0, k] = 0x3E00  # bf16 0.125
        y, a = oracle.w4a16_gemm_bf16(wq, s, z, xb, N, K, g)
        assert np.array_equal(y[0], 0.125 * w[:, k]) and np.array_equal(a[0], 0.125 * np.abs(w[:, k]))


# --- the pages' exact fp16 identity (used by the kernels' unpack) ----------------

def test_fp16_magic_identity():
    """fp16 0x6400|n is exactly 1024+n, and (1024+n) - (1024+zp) == n - zp exactly."""
    n = np.arange(16, dtype=np.uint16)
    v = (0x6400 | n).view(np.float16)
    assert np.array_equal(v.astype(np.float64), 1024.0 + n)
    for zp in range(16):
        sub = (v - np.float16(1024 + zp)).astype(np.float64)
        assert np.array_equal(sub, n.astype(np.float64) - zp)


def test_bf16_and_fp32_magic_identities():
    """bf16 0x4300|n is 128+n and fp32 0x4B000000|n is 2^23+n, for every nibble n."""
    n = np.arange(16, dtype=np.uint32)
    bf = ((0x4300 | n) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(bf, 128.0 + n)
    f32 = (0x4B000000 | n).view(np.float32).astype(np.float64)
    assert np.array_equal(f32, 2.0 ** 23 + n)


# --- GEMM -------------------------------------------------------------------------

@pytest.mark.parametrize("M,N,K", [(1, 1, 256), (2, 3, 256), (3, 16, 512), (7, 5, 256), (16, 9, 512)])
def test_gemm_brute_force_against_numpy(M, N, K):
    rng = np.random.default_rng(M * 1000 + N * 10 + K)
    x = rng.standard_normal((M, K))
    w = rng.standard_normal((N, K))
    y, a = oracle.gemm(x, w)
    ref = x @ w.T
    ref_abs = np.abs(x) @ np.abs(w).T
    assert y.shape == (M, N)
    assert np.allclose(y, ref, rtol=0, atol=1e-12 * ref_abs.max())
    assert np.allclose(a, ref_abs, rtol=1e-13, atol=0)
    assert np.all(a >= np.abs(y) - 1e-12)


def test_gemm_unit_vector_picks_weight_column():
    """x = e_k gives y[:, n] = w[n][k] exactly."""
    N, K = 6, 256
    blocks = synth.q4k_weights(N, K, seed=5)
    w = oracle.q4k_dequant(blocks, N, K)
    for k in (0, 31, 32, 100, 255):
        x = np.zeros((1, K))
        x[0, k] = 1.0
        y, _ = oracle.gemm(x, w)
        assert np.array_equal(y[0], w[:, k])


def test_q4k_gemm_closed_form_one_subblock():
    """x = 1 on sub-block j only: y = d*sc_j*sum(q) - 32*dmin*m_j (worked example block)."""
    case = [c for c in _q4k_cases() if c["name"] == "worked_example_power_of_two_scales"][0]
    blk = _q4k_block(case["blocks"][0])
    x = np.zeros((1, 256), np.float64)
    x[0, 0:32] = 1.0
    # bf16 bit pattern of 1.0 is 0x3F80
    xb = np.where(x > 0, 0x3F80, 0).astype(np.uint16)
    y, a = oracle.q4k_gemm(blk, xb, 1, 256)
    # d = 2^-10, sc_0 = 3, sum q = 7; dmin = 2^-9, m_0 = 5
    assert y[0, 0] == 2.0 ** -10 * 3 * 7 - 32 * 2.0 ** -9 * 5
    assert a[0, 0] == abs(2.0 ** -10 * 3 * 7 - 2.0 ** -9 * 5) + 31 * 2.0 ** -9 * 5


def test_q4k_gemm_closed_form_random_blocks():
    """Same closed form on random blocks, every sub-block of every row."""
    N, K = 4, 512
    blocks = synth.q4k_weights(N, K, seed=21)
    raw = blocks.reshape(N, K // 256, 144)
    for b in range(K // 256):
        for j in range(8):
            xb = np.zeros((1, K), np.uint16)
            xb[0, 256 * b + 32 * j:256 * b + 32 * j + 32] = 0x3F80
            y, _ = oracle.q4k_gemm(blocks, xb, N, K)
            for n in range(N):
                d = float(raw[n, b, 0:2].copy().view("<u2").view(np.float16)[0])
                dmin = float(raw[n, b, 2:4].copy().view("<u2").view(np.float16)[0])
                sc, m = oracle.q4k_scale_min(raw[n, b, 4:16], j)
                qs = raw[n, b, 16:144].astype(np.int64)
                c, hi = divmod(j, 2)
                q = (qs[32 * c:32 * c + 32] >> 4) if hi else (qs[32 * c:32 * c + 32] & 15)
                expect = d * sc * q.sum() - 32 * dmin * m
                assert abs(y[0, n] - expect) <= 1e-12 * (abs(expect) + 1)


def test_w4a16_gemm_against_numpy():
    N, K, g = 5, 256, 128
    wq, s, z = synth.w4a16_weights(N, K, g, seed=3)
    x = synth.activations_f16(3, K, seed=4)
    y, _ = oracle.w4a16_gemm(wq, s, z, x, N, K, g)
    w = oracle.w4a16_dequant(wq, s, z, N, K, g)
    assert np.allclose(y, x.astype(np.float64) @ w.T, rtol=0, atol=1e-12)


# --- generators -------------------------------------------------------------------

def test_synth_value_ranges():
    blocks = synth.q4k_weights(4, 1024, seed=1).reshape(-1, 144)
    d = blocks[:, 0:2].copy().view("<u2").view(np.float16).astype(np.float64)
    assert d.min() >= 1e-3 * (1 - 2 ** -11) and d.max() <= 4e-3 * (1 + 2 ** -11)
    xb = synth.activations_bf16(8, 256, seed=2)
    x = oracle.bf16_to_f64(xb)
    assert abs(x.mean()) < 0.1 and 0.9 < x.std() < 1.1
    wq, s, z = synth.w4a16_weights(4, 256, 128, seed=3)
    assert z.max() <= 15 and s.astype(np.float64).min() >= 1e-3 * (1 - 2 ** -11)
    q6 = synth.q6k_weights(64, 1024, seed=4).reshape(-1, 210)
    d6 = q6[:, 208:210].copy().view("<u2").view(np.float16).astype(np.float64)
    assert d6.min() >= 1e-5 * (1 - 2 ** -10) and d6.max() <= 8e-5 * (1 + 2 ** -11)
    assert (d6 < 2.0 ** -14).any() and (d6 >= 2.0 ** -14).any()  # subnormal and normal fp16 d


# ---------------------------------------------------------------- activation quantization


def _q8_cases():
    with open(os.path.join(GOLDEN, "q8_handbuilt.json")) as f:
        return json.load(f)["cases"]


def _bf16_bits(values):
    """Exact bfloat16 bits of values that bfloat16 represents exactly."""
    f = np.asarray(values, np.float32)
    bits = (f.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((bits.astype(np.uint32) << 16).view(np.float32), f), "not a bfloat16 value"
    return bits


@pytest.mark.parametrize("case", _q8_cases(), ids=lambda c: c["name"])
def test_q8_handbuilt_blocks(case):
    """Blocks worked out by hand (tests/golden/q8_handbuilt.json), also as the
    second block of a row and with the row mirrored (q(-x) = -q(x))."""
    x = _bf16_bits(_rle(case["x"]))
    expect_q = _rle(case["q"]).astype(np.int64)
    row = np.concatenate([_bf16_bits(np.full(32, 3.0)), x])
    q, d, s = oracle.q8_quantize(row.reshape(1, 64), 64)
    assert np.array_equal(q[0, 32:].astype(np.int64), expect_q)
    assert d[0, 1] == np.float32(case["d"]) and s[0, 1] == case["s"]
    q2, d2, s2 = oracle.q8_quantize((x ^ np.uint16(0x8000)).reshape(1, 32), 32)
    assert np.array_equal(q2[0].astype(np.int64), -expect_q) and d2[0, 0] == np.float32(case["d"])
    assert s2[0, 0] == -case["s"]


def test_q8_invariants_on_wide_range_values():
    """Every block: |q| <= 127, the largest |q| is 127 (unless the block is zero),
    s = sum q, and d * q is within d/2 (plus fp32 rounding) of x."""
    rng = np.random.default_rng(5)
    M, K = 6, 1024
    mant = rng.integers(0, 128, size=(M, K))
    expo = rng.integers(100, 150, size=(M, K))  # 2^-27 .. 2^22
    sign = rng.integers(0, 2, size=(M, K))
    bits = ((sign << 15) | (expo << 7) | mant).astype(np.uint16)
    bits[2, 64:96] = 0  # one zero block
    q, d, s = oracle.q8_quantize(bits, K)
    x = oracle.bf16_to_f64(bits)
    qb = q.reshape(M, K // 32, 32).astype(np.int64)
    assert np.abs(qb).max() <= 127
    amax = np.abs(x.reshape(M, K // 32, 32)).max(axis=2)
    assert np.array_equal(np.abs(qb).max(axis=2) == 127, amax > 0)
    assert np.array_equal(qb.sum(axis=2), s.astype(np.int64))
    err = np.abs(x - oracle.q8_dequant(q, d))
    half = np.repeat(d.astype(np.float64), 32, axis=1) / 2
    assert np.all(err <= half * (1 + 2.0 ** -20))
    assert np.all(np.abs(d.astype(np.float64) * 127 - amax) <= amax * 2.0 ** -23)


def test_q8_rejects_nonfinite_and_bad_shape():
    bits = np.zeros((1, 32), np.uint16)
    bits[0, 3] = 0x7F80  # +inf
    with pytest.raises(ValueError):
        oracle.q8_quantize(bits, 32)
    with pytest.raises(ValueError):
        oracle.q8_quantize(np.zeros((1, 48), np.uint16), 48)


@pytest.mark.parametrize("case", _q4k_cases(), ids=lambda c: c["name"])
def test_q4k_terms_handbuilt(case):
    """w = a - b with a = d*sc*q and b = dmin*m: the hand-built blocks with dmin = 0
    have b = 0 and a = w, those with d = 0 have a = 0 and b = -w."""
    blocks = np.stack([_q4k_block(b) for b in case["blocks"]]).reshape(case["N"], -1)
    a, b = oracle.q4k_terms(blocks, case["N"], case["K"])
    w = np.concatenate([_rle(e) for e in case["expect"]]).reshape(case["N"], case["K"])
    assert np.array_equal(a - b, w)
    spec = case["blocks"][0]
    if int(spec["dmin"], 16) == 0:
        assert not b.any() and np.array_equal(a, w)
    if int(spec["d"], 16) == 0:
        assert not a.any() and np.array_equal(b, -w)


def test_q4k_terms_worked_example():
    """d = 2^-10, dmin = 2^-9, sc_0 = 3, m_0 = 5, q(element 0) = 7: a = 21/1024 and
    b = 10/1024 for element 0; a = 0, b = 10/1024 for the rest of sub-block 0."""
    case = next(c for c in _q4k_cases() if c["name"] == "worked_example_power_of_two_scales")
    a, b = oracle.q4k_terms(_q4k_block(case["blocks"][0]).reshape(1, -1), 1, 256)
    assert a[0, 0] == 21 / 1024 and b[0, 0] == 10 / 1024
    assert not a[0, 1:32].any() and np.all(b[0, 1:32] == 10 / 1024) and not b[0, 32:].any()


def test_q4k_q8_gemm_equals_unquantized_product_on_the_code_grid():
    """Activations already on the code grid (each block's largest |x| is 127/64 and
    every x a multiple of 1/64) quantize exactly, so the product with quantized
    activations is the unquantized oracle product, bit for bit; the bound magnitude
    over the two weight terms is at least the one over the weights."""
    rng = np.random.default_rng(9)
    M, N, K = 3, 7, 512
    codes = rng.integers(-127, 128, size=(M, K))
    codes[:, ::32] = 127 * np.where(rng.integers(0, 2, size=(M, K // 32)) > 0, 1, -1)
    bits = _bf16_bits(codes / 64.0).reshape(M, K)
    blocks = synth.q4k_weights(N, K, seed=10)
    q, d, s = oracle.q8_quantize(bits, K)
    assert np.array_equal(q.astype(np.int64), codes) and np.all(d == np.float32(1 / 64))
    y, mag2 = oracle.q4k_q8_gemm(blocks, q, d, N, K)
    y0, mag = oracle.q4k_gemm(blocks, bits, N, K)
    assert np.array_equal(y, y0)
    assert np.all(mag2 >= mag)
