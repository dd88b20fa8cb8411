"""CPU oracle for the quantized-weight prefill GEMM -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The library path
(``quantized_weight_prefill_gb300``) never imports it, and the two share no
code: this package wraps ``qwp_oracle.c`` (plain C, fp64, naive loops) with
ctypes and numpy.

Functions (each follows the passage cited in ``qwp_oracle.c``):
  half_to_f64 / bf16_to_f64   exact IEEE decode of stored 16-bit values
  q4k_scale_min               the 6-bit (scale, min) pair of one sub-block
  q4k_dequant                 GGML Q4_K super-blocks -> fp64 weights [N, K]
  q6k_code / q6k_dequant      GGML Q6_K blocks: one 6-bit code / fp64 weights [N, K]
  w4a16_dequant               interleaved int4 words + fp16 scales + zeros -> fp64
  gemm                        y = x @ w.T and a = |x| @ |w|.T, both fp64, naive loops
  q4k_gemm / q6k_gemm / w4a16_gemm   decode + dequant + gemm in one call
  q4k_terms                   the two exact terms a = d*sc*q, b = dmin*m of each Q4_K weight
  q8_quantize / q8_dequant    activation quantization to 8-bit codes per block of 32
  q4k_q8_gemm                 the Q4_K product with quantized activations, and its bound

Parity pins: see ``tests/test_oracle_pins.py``.  The exact GGML bit layout of
the 6-bit scale/min packing is not printed on the source pages and is
"parity unpinned" beyond the invariants tested there (every one of the 96
packed bits reaches exactly one 6-bit value).  The same holds for the Q6_K bit
layout (the pages name Q6_K but print no layout): the pins check that the 1536
code bits of a block reach each of the 256 codes exactly six times, one bit per
power of two, that each int8 scale covers exactly 16 consecutive weights, and
hand-worked blocks of the GGML reading.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.library_path()
        if not os.path.exists(path) or _build.is_stale():
            _build.build()
        lib = ctypes.CDLL(path)
        d = ctypes.c_double
        i64 = ctypes.c_int64
        p = ctypes.c_void_p
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_half_to_double.restype = d
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = d
        lib.oracle_half_array_to_double.argtypes = [p, i64, p]
        lib.oracle_bf16_array_to_double.argtypes = [p, i64, p]
        lib.oracle_q4k_scale_min.argtypes = [p, ctypes.c_int, p, p]
        lib.oracle_q4k_scale_min.restype = None
        lib.oracle_q4k_dequant.argtypes = [p, i64, i64, p]
        lib.oracle_q6k_code.argtypes = [p, ctypes.c_int]
        lib.oracle_q6k_dequant.argtypes = [p, i64, i64, p]
        lib.oracle_w4a16_dequant.argtypes = [p, p, p, i64, i64, i64, p]
        lib.oracle_gemm.argtypes = [p, p, i64, i64, i64, p, p]
        lib.oracle_q4k_terms.argtypes = [p, i64, i64, p, p]
        lib.oracle_q8_quantize.argtypes = [p, i64, i64, p, p, p]
        lib.oracle_num_threads.argtypes = []
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def half_to_f64(bits) -> np.ndarray:
    """Exact value of IEEE binary16 bit patterns (uint16 array) as float64."""
    arr = np.asarray(bits)
    src = np.ascontiguousarray(arr.view(np.uint16) if arr.dtype == np.float16
                               else arr.astype(np.uint16, copy=False))
    out = np.empty(src.shape, np.float64)
    flat = src.reshape(-1)
    o = out.reshape(-1)
    # -2 only flags Inf/NaN inputs; their decoded values are still written.
    rc = _load().oracle_half_array_to_double(_ptr(flat), flat.size, _ptr(o))
    if rc not in (0, -2):
        _check(rc, "half decode")
    return out


def bf16_to_f64(bits) -> np.ndarray:
    """Exact value of bfloat16 bit patterns (uint16 array) as float64."""
    src = np.ascontiguousarray(np.asarray(bits).astype(np.uint16, copy=False))
    out = np.empty(src.shape, np.float64)
    flat = src.reshape(-1)
    o = out.reshape(-1)
    rc = _load().oracle_bf16_array_to_double(_ptr(flat), flat.size, _ptr(o))
    if rc not in (0, -2):
        _check(rc, "bf16 decode")
    return out


def q4k_scale_min(scales12: np.ndarray, j: int) -> tuple[int, int]:
    s = np.ascontiguousarray(np.asarray(scales12, dtype=np.uint8).reshape(12))
    sc = ctypes.c_int()
    m = ctypes.c_int()
    _load().oracle_q4k_scale_min(_ptr(s), int(j), ctypes.byref(sc), ctypes.byref(m))
    return sc.value, m.value


def q4k_dequant(blocks: np.ndarray, N: int, K: int) -> np.ndarray:
    """GGML Q4_K rows (N * K/256 * 144 bytes) -> exact fp64 weights [N, K]."""
    b = np.ascontiguousarray(np.asarray(blocks, dtype=np.uint8).reshape(-1))
    if b.size != N * (K // 256) * 144 or K % 256:
        raise ValueError("Q4_K buffer size does not match N, K")
    w = np.empty((N, K), np.float64)
    _check(_load().oracle_q4k_dequant(_ptr(b), N, K, _ptr(w)), "q4k_dequant")
    return w


def q6k_code(block: np.ndarray, e: int) -> int:
    """The 6-bit code (0..63) of element e of one 210-byte GGML Q6_K block."""
    b = np.ascontiguousarray(np.asarray(block, dtype=np.uint8).reshape(210))
    return int(_load().oracle_q6k_code(_ptr(b), int(e)))


def q6k_dequant(blocks: np.ndarray, N: int, K: int) -> np.ndarray:
    """GGML Q6_K rows (N * K/256 * 210 bytes) -> exact fp64 weights [N, K]."""
    b = np.ascontiguousarray(np.asarray(blocks, dtype=np.uint8).reshape(-1))
    if b.size != N * (K // 256) * 210 or K % 256:
        raise ValueError("Q6_K buffer size does not match N, K")
    w = np.empty((N, K), np.float64)
    _check(_load().oracle_q6k_dequant(_ptr(b), N, K, _ptr(w)), "q6k_dequant")
    return w


def w4a16_dequant(wq: np.ndarray, scales: np.ndarray, zeros,
                  N: int, K: int, group: int) -> np.ndarray:
    """Interleaved int4 words [N, K/8] + fp16 scales/uint8 zeros [N, K/group] -> fp64 [N, K].
    zeros=None: the symmetric form (zero point 8)."""
    q = np.ascontiguousarray(np.asarray(wq).view(np.uint32).reshape(N, K // 8))
    s = np.ascontiguousarray(np.asarray(scales).view(np.uint16).reshape(N, K // group))
    z = None if zeros is None else np.ascontiguousarray(np.asarray(zeros, dtype=np.uint8).reshape(N, K // group))
    w = np.empty((N, K), np.float64)
    _check(_load().oracle_w4a16_dequant(_ptr(q), _ptr(s), _ptr(z) if z is not None else None, N, K, group,
                                        _ptr(w)), "w4a16_dequant")
    return w


def gemm(x: np.ndarray, w: np.ndarray, with_abs: bool = True):
    """y = x @ w.T (fp64, naive loops) and a = sum_k |x*w|; x [M,K], w [N,K]."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    M, K = x.shape
    N, K2 = w.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    y = np.empty((M, N), np.float64)
    a = np.empty((M, N), np.float64) if with_abs else None
    _check(_load().oracle_gemm(_ptr(x), _ptr(w), M, N, K, _ptr(y),
                               _ptr(a) if a is not None else None), "gemm")
    return (y, a) if with_abs else y


def q4k_gemm(blocks: np.ndarray, x_bf16_bits: np.ndarray, N: int, K: int, with_abs: bool = True):
    """Plain definition of the Q4_K prefill GEMM: y[M,N] = x[M,K] . W[N,K]^T in fp64."""
    w = q4k_dequant(blocks, N, K)
    x = bf16_to_f64(x_bf16_bits)
    return gemm(x.reshape(-1, K), w, with_abs)


def q6k_gemm(blocks: np.ndarray, x_bf16_bits: np.ndarray, N: int, K: int, with_abs: bool = True):
    """Plain definition of the Q6_K prefill GEMM: y[M,N] = x[M,K] . W[N,K]^T in fp64 (bf16 x)."""
    w = q6k_dequant(blocks, N, K)
    x = bf16_to_f64(x_bf16_bits)
    return gemm(x.reshape(-1, K), w, with_abs)


def w4a16_gemm(wq, scales, zeros, x_f16, N: int, K: int, group: int, with_abs: bool = True):
    """Plain definition of the W4A16 GEMM in fp64 (fp16 activations; zeros=None: symmetric)."""
    w = w4a16_dequant(wq, scales, zeros, N, K, group)
    x = half_to_f64(np.asarray(x_f16).view(np.uint16))
    return gemm(x.reshape(-1, K), w, with_abs)


def w4a16_gemm_bf16(wq, scales, zeros, x_bf16, N: int, K: int, group: int, with_abs: bool = True):
    """The W4A16 GEMM with bf16 activations, in fp64."""
    w = w4a16_dequant(wq, scales, zeros, N, K, group)
    x = bf16_to_f64(np.asarray(x_bf16).view(np.uint16))
    return gemm(x.reshape(-1, K), w, with_abs)


def q4k_terms(blocks: np.ndarray, N: int, K: int):
    """The exact terms (a, b), both fp64 [N, K], of every Q4_K weight w = a - b:
    a = d * sc_j * q and b = dmin * m_j."""
    blk = np.ascontiguousarray(np.asarray(blocks, dtype=np.uint8).reshape(-1))
    if blk.size != N * (K // 256) * 144 or K % 256:
        raise ValueError("Q4_K buffer size does not match N, K")
    a = np.empty((N, K), np.float64)
    b = np.empty((N, K), np.float64)
    _check(_load().oracle_q4k_terms(_ptr(blk), N, K, _ptr(a), _ptr(b)), "q4k_terms")
    return a, b


def q8_quantize(x_bf16_bits: np.ndarray, K: int):
    """bf16 activations [M, K] -> (q int8 [M, K], d float32 [M, K/32], s int32 [M, K/32]):
    per block of 32, d = amax/127, q = round(x * (1/d)) half away from zero, s = sum q,
    all in fp32 (see qwp_oracle.c)."""
    src = np.ascontiguousarray(np.asarray(x_bf16_bits).astype(np.uint16, copy=False).reshape(-1, K))
    M = src.shape[0]
    q = np.empty((M, K), np.int8)
    d = np.empty((M, K // 32), np.float32)
    s = np.empty((M, K // 32), np.int32)
    _check(_load().oracle_q8_quantize(_ptr(src), M, K, _ptr(q), _ptr(d), _ptr(s)), "q8_quantize")
    return q, d, s


def q8_dequant(q: np.ndarray, d: np.ndarray) -> np.ndarray:
    """The value each code stands for, d * q, in fp64 (exact)."""
    q = np.asarray(q, dtype=np.int8)
    M, K = q.shape
    return q.astype(np.float64) * np.repeat(np.asarray(d, dtype=np.float64).reshape(M, K // 32), 32, axis=1)


def q4k_q8_gemm(blocks: np.ndarray, q: np.ndarray, d: np.ndarray, N: int, K: int):
    """Plain definition of the Q4_K product with quantized activations, fp64:
    y[m, n] = sum_k W[n, k] * d[m, k/32] * q[m, k]; with it the bound magnitude
    sum_k (|a[n, k]| + |b[n, k]|) * |d * q| over the weights' two terms."""
    xh = q8_dequant(q, d)
    w = q4k_dequant(blocks, N, K)
    y = gemm(xh, w, with_abs=False)
    a, b = q4k_terms(blocks, N, K)
    mag2 = gemm(np.abs(xh), np.abs(a) + np.abs(b), with_abs=False)
    return y, mag2
