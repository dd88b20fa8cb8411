"""Shared test helpers: moving the seeded inputs to the GPU, the chunked oracle,
the error-bound check, and a numpy statement of the documented repack layouts
(used only to check the CUDA repack byte for byte)."""
from __future__ import annotations

import numpy as np

import oracle

TOL_REL = 1e-3
TOL_ABS = 1e-5


# --- documented tile-major layouts (numpy restatement, test side) ----------------

def q4k_tiled_reference(blocks: np.ndarray, N: int, K: int) -> np.ndarray:
    """Tile-major Q4_K order: per 128-row tile and super-block, a 16-byte header plane
    and four nibble planes [h][row][16 bytes]; word v of a row's 64-wide chunk holds
    chunk elements 8v+t, element t=2p in bits 4p..4p+3 and t=2p+1 in bits 16+4p..19+4p."""
    nb = K // 256
    raw = blocks.reshape(N, nb, 144)
    out = np.zeros(N * nb * 144, np.uint8)
    for t0 in range(0, N, 128):
        R = min(128, N - t0)
        for b in range(nb):
            base = t0 * nb * 144 + b * R * 144
            grp = out[base:base + R * 144]
            grp[:16 * R] = raw[t0:t0 + R, b, :16].reshape(-1)
            qs = raw[t0:t0 + R, b, 16:].astype(np.uint32)            # [R, 128]
            for c in range(4):
                lo = qs[:, 32 * c:32 * c + 32] & 15                     # elements 0..31
                hi = qs[:, 32 * c:32 * c + 32] >> 4                     # elements 32..63
                elems = np.concatenate([lo, hi], axis=1)                # [R, 64]
                words = np.zeros((R, 8), np.uint32)
                for t in range(8):
                    shift = 16 + 4 * (t // 2) if t % 2 else 4 * (t // 2)
                    words |= elems[:, t::8] << shift
                plane = words.reshape(R, 2, 4).transpose(1, 0, 2)        # [h][row][4 words]
                start = 16 * R + 32 * R * c
                grp[start:start + 32 * R] = plane.astype("<u4").reshape(-1).view(np.uint8)
    return out


def q6k_codes(blocks: np.ndarray, N: int, K: int) -> np.ndarray:
    """The 6-bit codes [N, K] of GGML Q6_K rows, read through the oracle's dequant with
    every scale set to 1 and d to 1.0 (w = q - 32)."""
    raw = blocks.reshape(N, K // 256, 210).copy()
    raw[:, :, 192:208] = 1
    raw[:, :, 208], raw[:, :, 209] = 0x00, 0x3C
    return (oracle.q6k_dequant(raw.reshape(-1), N, K) + 32).astype(np.uint32)


def q6k_high_bit(t: int) -> int:
    p, o = (t & 7) >> 1, t & 1
    return 4 + 2 * p + 16 * o if t < 8 else (12 + 2 * p + 16 * o) & 31


def q6k_tiled_reference(blocks: np.ndarray, N: int, K: int) -> np.ndarray:
    """Tile-major Q6_K order: the last tile padded to a multiple of 8 rows; per tile and
    super-block a d plane [row][2 B], a scale plane [row][16 B], four low planes
    [h][row][16 B] (interleaved nibbles as in Q4_K) and four high planes [row][16 B]
    (word u: high bits of chunk elements 16u+t at q6k_high_bit(t))."""
    nb = K // 256
    raw = blocks.reshape(N, nb, 210)
    codes = q6k_codes(blocks, N, K).reshape(N, nb, 256)
    full = N // 128 * 128
    stored = full + ((N - full + 7) // 8 * 8)
    out = np.zeros(stored * nb * 210, np.uint8)
    for t0 in range(0, N, 128):
        R = min(128, N - t0)
        Rp = (R + 7) // 8 * 8
        for b in range(nb):
            base = t0 * nb * 210 + b * Rp * 210
            grp = out[base:base + Rp * 210]
            grp[:2 * R] = raw[t0:t0 + R, b, 208:210].reshape(-1)
            grp[2 * Rp:2 * Rp + 16 * R] = raw[t0:t0 + R, b, 192:208].reshape(-1)
            q = codes[t0:t0 + R, b]                                    # [R, 256]
            for c in range(4):
                lo = q[:, 64 * c:64 * c + 64] & 15
                words = np.zeros((R, 8), np.uint32)
                for t in range(8):
                    shift = 16 + 4 * (t // 2) if t % 2 else 4 * (t // 2)
                    words |= lo[:, t::8] << shift
                plane = np.zeros((2, Rp, 4), np.uint32)
                plane[:, :R] = words.reshape(R, 2, 4).transpose(1, 0, 2)
                start = 18 * Rp + 32 * Rp * c
                grp[start:start + 32 * Rp] = plane.astype("<u4").reshape(-1).view(np.uint8)
                hi = q[:, 64 * c:64 * c + 64] >> 4
                hw = np.zeros((Rp, 4), np.uint32)
                for t in range(16):
                    hw[:R] |= hi[:, t::16] << q6k_high_bit(t)
                start = 146 * Rp + 16 * Rp * c
                grp[start:start + 16 * Rp] = hw.astype("<u4").reshape(-1).view(np.uint8)
    return out


def q6k_oracle_rows(blocks: np.ndarray, xb_rows: np.ndarray, N: int, K: int, chunk: int = 2048):
    """Oracle y and sum|x*w| of the Q6_K GEMM for the given bf16 activation rows."""
    x = oracle.bf16_to_f64(xb_rows).reshape(-1, K)
    raw = blocks.reshape(N, -1)
    ys, ms = [], []
    for n0 in range(0, N, chunk):
        n1 = min(N, n0 + chunk)
        w = oracle.q6k_dequant(raw[n0:n1], n1 - n0, K)
        y, a = oracle.gemm(x, w)
        ys.append(y)
        ms.append(a)
    return np.concatenate(ys, axis=1), np.concatenate(ms, axis=1)


def w4a16_tiled_reference(wq: np.ndarray, N: int, K: int) -> np.ndarray:
    """Tile-major W4A16 order: per 128-row tile and 64-wide K-block, a plane [h][row][4 words]."""
    words = wq.view(np.uint32).reshape(N, K // 8)
    out = np.zeros(N * K // 8, np.uint32)
    for t0 in range(0, N, 128):
        R = min(128, N - t0)
        for j in range(K // 64):
            blk = words[t0:t0 + R, 8 * j:8 * j + 8].reshape(R, 2, 4).transpose(1, 0, 2)
            base = (t0 * K // 2 + j * R * 32) // 4
            out[base:base + 8 * R] = blk.reshape(-1)
    return out


# --- oracle on row samples ---------------------------------------------------------

def q4k_oracle_rows(blocks: np.ndarray, xb_rows: np.ndarray, N: int, K: int, chunk: int = 2048):
    """Oracle y and sum|x*w| for the given bf16 activation rows, dequantizing W in row chunks."""
    x = oracle.bf16_to_f64(xb_rows).reshape(-1, K)
    raw = blocks.reshape(N, -1)
    ys, ms = [], []
    for n0 in range(0, N, chunk):
        n1 = min(N, n0 + chunk)
        w = oracle.q4k_dequant(raw[n0:n1], n1 - n0, K)
        y, a = oracle.gemm(x, w)
        ys.append(y)
        ms.append(a)
    return np.concatenate(ys, axis=1), np.concatenate(ms, axis=1)


def w4a16_oracle_rows(wq, s, z, xh_rows, N: int, K: int, group: int, chunk: int = 2048, bf16: bool = False):
    """Oracle rows of the W4A16 GEMM (z None: symmetric; bf16: x holds bf16 bits, else fp16)."""
    bits = np.asarray(xh_rows).view(np.uint16)
    x = (oracle.bf16_to_f64(bits) if bf16 else oracle.half_to_f64(bits)).reshape(-1, K)
    ys, ms = [], []
    for n0 in range(0, N, chunk):
        n1 = min(N, n0 + chunk)
        w = oracle.w4a16_dequant(wq[n0:n1], s[n0:n1], None if z is None else z[n0:n1], n1 - n0, K, group)
        y, a = oracle.gemm(x, w)
        ys.append(y)
        ms.append(a)
    return np.concatenate(ys, axis=1), np.concatenate(ms, axis=1)


def sample_rows(M: int, count: int = 64, seed: int = 0) -> np.ndarray:
    """First 16, last 16 and random rows in between (all rows if M is small)."""
    if M <= count:
        return np.arange(M)
    rng = np.random.default_rng(seed)
    head = np.arange(16)
    tail = np.arange(M - 16, M)
    mid = rng.choice(np.arange(16, M - 16), size=count - 32, replace=False)
    return np.unique(np.concatenate([head, mid, tail]))


def check_bound(y_gpu: np.ndarray, y_ref: np.ndarray, mag: np.ndarray, what: str) -> float:
    """Assert |y_gpu - y_ref| <= 1e-3 * sum|x*w| + 1e-5 elementwise; return the worst err/bound."""
    err = np.abs(y_gpu.astype(np.float64) - y_ref)
    bound = TOL_REL * mag + TOL_ABS
    ratio = float((err / bound).max()) if err.size else 0.0
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {err.size} outside the bound, "
                           f"worst err/bound {ratio:.3f}, first at {np.argwhere(bad)[0].tolist()}")
    assert np.isfinite(y_gpu).all(), f"{what}: non-finite output"
    return ratio



# --- documented quantized-activation record layout (numpy restatement) -----------

Q8_PERM = np.array([0, 4, 1, 5, 2, 6, 3, 7])  # stored byte i of a run of 8 holds element Q8_PERM[i]


def q8_records_reference(q: np.ndarray, d: np.ndarray, s: np.ndarray) -> np.ndarray:
    """The record buffer for codes q [M, K] int8, scales d [M, K/32] fp32 and sums
    s [M, K/32]: tokens in groups of 8 (zero-padded), one 2560-byte record per
    (group, 256-wide super-block), 320 bytes per token: the 256 codes with each run
    of 8 stored in the order e0 e4 e1 e5 e2 e6 e3 e7, 8 fp32 scales, 8 fp32 sums."""
    M, K = q.shape
    G, nsb = -(-M // 8), K // 256
    codes = np.zeros((G * 8, K), np.int8)
    codes[:M] = q
    dd = np.zeros((G * 8, K // 32), np.float32)
    dd[:M] = d
    ss = np.zeros((G * 8, K // 32), np.float32)
    ss[:M] = s
    runs = codes.reshape(G * 8, K // 8, 8)[:, :, Q8_PERM].reshape(G, 8, nsb, 256)
    rec = np.zeros((G, nsb, 8, 320), np.uint8)
    rec[..., :256] = runs.transpose(0, 2, 1, 3).view(np.uint8)
    rec[..., 256:288] = dd.reshape(G, 8, nsb, 8).transpose(0, 2, 1, 3).view(np.uint8).reshape(G, nsb, 8, 32)
    rec[..., 288:320] = ss.reshape(G, 8, nsb, 8).transpose(0, 2, 1, 3).view(np.uint8).reshape(G, nsb, 8, 32)
    return rec.reshape(-1)
