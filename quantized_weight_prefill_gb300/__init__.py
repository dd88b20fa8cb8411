"""Batched-prefill GEMM over 4-bit quantized weights (Q4_K, W4A16) on GB300.

Thin Python binding over the C ABI of ``libqwp.so`` (declared in
``include/qwp.h``).  Every function here only marshals arguments: it checks
that tensors live on the GPU with the right dtype and layout, allocates the
output with torch when none is given, and passes raw pointers, sizes and the
current CUDA stream to the library.  All arithmetic runs in the library's CUDA
kernels; there is no CPU fallback, and a missing library raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

__all__ = [
    "QwpError", "library", "q4k_repacked_bytes", "q4k_repack", "q4k_dequant", "q4k_gemm", "q4k_gemm_f16",
    "q4k_gemm_noalloc", "NOALLOC_MAX_X_ELEMS",
    "q6k_repacked_bytes", "q6k_repack", "q6k_dequant", "q6k_gemm", "q6k_gemm_f16",
    "w4a16_repacked_bytes", "w4a16_repack", "w4a16_dequant", "w4a16_gemm", "w4a16_gemm_bf16",
    "device_status", "set_decode_policy", "decode_selected", "DECODE_AUTO", "DECODE_NEVER", "DECODE_ALWAYS",
    "gemm_plan", "set_wait_timeout_ns", "DEFAULT_WAIT_TIMEOUT_NS",
    "EXPORTED_SYMBOLS",
]

# Every symbol include/qwp.h declares.
EXPORTED_SYMBOLS = (
    "qwp_status_string", "q4k_repacked_bytes", "q4k_repack", "q4k_dequant", "q4k_gemm", "q4k_gemm_f16",
    "q4k_gemm_noalloc", "q6k_repacked_bytes", "q6k_repack", "q6k_dequant", "q6k_gemm", "q6k_gemm_f16",
    "w4a16_repacked_bytes", "w4a16_repack", "w4a16_dequant", "w4a16_gemm", "w4a16_gemm_bf16",
    "qwp_device_status", "qwp_set_decode_policy", "qwp_decode_selected", "qwp_gemm_plan",
    "qwp_set_wait_timeout_ns", "q8_activation_bytes", "q8_quantize", "q4k_q8_gemm",
    "q4k_gemm_batched", "q4k_gemm_batched_f16",
)

# Decode-kernel dispatch policies (enum qwp_decode_policy in the header).
DECODE_AUTO, DECODE_NEVER, DECODE_ALWAYS = 0, 1, 2

# Largest M*K that q4k_gemm_noalloc accepts (QWP_NOALLOC_MAX_X_ELEMS in the header).
NOALLOC_MAX_X_ELEMS = 8388608

_lib = None


class QwpError(RuntimeError):
    def __init__(self, code: int, name: str, what: str):
        super().__init__(f"{what}: {name} ({code})")
        self.code = code
        self.name = name


def library() -> ctypes.CDLL:
    """The loaded libqwp.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError(
                f"{_build.LIB} is missing: build it with `python -c \"import __graft_entry__ as g; "
                "g.build()\"` (nvcc, sm_103a); there is no fallback path")
        lib = ctypes.CDLL(_build.LIB)
        i64, p, sz = ctypes.c_int64, ctypes.c_void_p, ctypes.POINTER(ctypes.c_size_t)
        lib.qwp_status_string.argtypes = [ctypes.c_int]
        lib.qwp_status_string.restype = ctypes.c_char_p
        lib.q4k_repacked_bytes.argtypes = [i64, i64, sz]
        lib.w4a16_repacked_bytes.argtypes = [i64, i64, sz]
        lib.q6k_repacked_bytes.argtypes = [i64, i64, sz]
        lib.q6k_repack.argtypes = [p, p, i64, i64, p]
        lib.q6k_dequant.argtypes = [p, p, i64, i64, p]
        lib.q6k_gemm.argtypes = [p, p, p, i64, i64, i64, p]
        lib.q6k_gemm_f16.argtypes = [p, p, p, i64, i64, i64, p]
        lib.q4k_repack.argtypes = [p, p, i64, i64, p]
        lib.q4k_dequant.argtypes = [p, p, i64, i64, p]
        lib.q4k_gemm.argtypes = [p, p, p, i64, i64, i64, p]
        lib.q4k_gemm_f16.argtypes = [p, p, p, i64, i64, i64, p]
        lib.q4k_gemm_noalloc.argtypes = [p, p, p, i64, i64, i64, p]
        lib.w4a16_repack.argtypes = [p, p, i64, i64, p]
        lib.w4a16_dequant.argtypes = [p, p, p, p, i64, i64, i64, p]
        lib.w4a16_gemm.argtypes = [p, p, p, p, p, i64, i64, i64, i64, p]
        lib.w4a16_gemm_bf16.argtypes = [p, p, p, p, p, i64, i64, i64, i64, p]
        lib.qwp_device_status.argtypes = [p]
        lib.qwp_set_decode_policy.argtypes = [ctypes.c_int]
        lib.qwp_decode_selected.argtypes = [ctypes.c_int, i64, i64, i64]
        lib.qwp_gemm_plan.argtypes = [ctypes.c_int, i64, i64, i64, p]
        lib.qwp_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
        lib.q8_activation_bytes.argtypes = [i64, i64, sz]
        lib.q8_quantize.argtypes = [p, p, i64, i64, p]
        lib.q4k_q8_gemm.argtypes = [p, p, p, i64, i64, i64, p]
        lib.q4k_gemm_batched.argtypes = [p, p, p, i64, i64, i64, i64, p]
        lib.q4k_gemm_batched_f16.argtypes = [p, p, p, i64, i64, i64, i64, p]
        for name in EXPORTED_SYMBOLS:
            if name != "qwp_status_string":
                getattr(lib, name).restype = ctypes.c_int
        _lib = lib
    return _lib


def _check(rc: int, what: str):
    if rc != 0:
        raise QwpError(rc, library().qwp_status_string(rc).decode(), what)


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _dev(t: torch.Tensor, dtype, name: str) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def q4k_repacked_bytes(N: int, K: int) -> int:
    out = ctypes.c_size_t()
    _check(library().q4k_repacked_bytes(N, K, ctypes.byref(out)), "q4k_repacked_bytes")
    return out.value


def w4a16_repacked_bytes(N: int, K: int) -> int:
    out = ctypes.c_size_t()
    _check(library().w4a16_repacked_bytes(N, K, ctypes.byref(out)), "w4a16_repacked_bytes")
    return out.value


def q4k_repack(w_ggml: torch.Tensor, N: int, K: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """GGML Q4_K rows (uint8, N*K/256*144 bytes) -> tile-major repacked bytes."""
    _dev(w_ggml, torch.uint8, "w_ggml")
    nbytes = q4k_repacked_bytes(N, K)
    if w_ggml.numel() != nbytes:
        raise ValueError("w_ggml size does not match N, K")
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=w_ggml.device)
    _dev(out, torch.uint8, "out")
    _check(library().q4k_repack(_ptr(w_ggml), _ptr(out), N, K, _stream(w_ggml)), "q4k_repack")
    return out


def q4k_dequant(w_tiled: torch.Tensor, N: int, K: int, out: torch.Tensor | None = None) -> torch.Tensor:
    _dev(w_tiled, torch.uint8, "w_tiled")
    if out is None:
        out = torch.empty(N, K, dtype=torch.float32, device=w_tiled.device)
    _dev(out, torch.float32, "out")
    _check(library().q4k_dequant(_ptr(w_tiled), _ptr(out), N, K, _stream(w_tiled)), "q4k_dequant")
    return out


def q4k_gemm(w_tiled: torch.Tensor, x: torch.Tensor, N: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """y[M, N] (fp32) = x[M, K] (bf16) . W^T with W the repacked Q4_K matrix."""
    _dev(w_tiled, torch.uint8, "w_tiled")
    _dev(x, torch.bfloat16, "x")
    M, K = x.shape
    if out is None:
        out = torch.empty(M, N, dtype=torch.float32, device=x.device)
    _dev(out, torch.float32, "out")
    _check(library().q4k_gemm(_ptr(w_tiled), _ptr(x), _ptr(out), M, N, K, _stream(x)), "q4k_gemm")
    return out


def q4k_gemm_f16(w_tiled: torch.Tensor, x: torch.Tensor, N: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """y[M, N] (fp32) = x[M, K] (fp16) . W^T with W the repacked Q4_K matrix."""
    _dev(w_tiled, torch.uint8, "w_tiled")
    _dev(x, torch.float16, "x")
    M, K = x.shape
    if out is None:
        out = torch.empty(M, N, dtype=torch.float32, device=x.device)
    _dev(out, torch.float32, "out")
    _check(library().q4k_gemm_f16(_ptr(w_tiled), _ptr(x), _ptr(out), M, N, K, _stream(x)), "q4k_gemm_f16")
    return out


def q4k_gemm_batched(w_tiled: torch.Tensor, x: torch.Tensor, N: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """A strided batch of Q4_K products in one launch: x [B, M, K] (bf16 or fp16),
    w_tiled the B repacked matrices back to back (B * q4k_repacked_bytes(N, K) bytes),
    y [B, M, N] fp32."""
    _dev(w_tiled, torch.uint8, "w_tiled")
    if x.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError("x must be bfloat16 or float16")
    _dev(x, x.dtype, "x")
    B, M, K = x.shape
    if w_tiled.numel() != B * q4k_repacked_bytes(N, K):
        raise ValueError("w_tiled must hold B repacked matrices of N x K")
    if out is None:
        out = torch.empty(B, M, N, dtype=torch.float32, device=x.device)
    _dev(out, torch.float32, "out")
    if tuple(out.shape) != (B, M, N):
        raise ValueError("out must be [B, M, N]")
    fn = library().q4k_gemm_batched if x.dtype == torch.bfloat16 else library().q4k_gemm_batched_f16
    _check(fn(_ptr(w_tiled), _ptr(x), _ptr(out), B, M, N, K, _stream(x)), "q4k_gemm_batched")
    return out


def q4k_gemm_noalloc(w_tiled: torch.Tensor, x: torch.Tensor, N: int, out: torch.Tensor) -> torch.Tensor:
    """q4k_gemm into a caller-provided ``out`` [M, N] fp32; the library allocates nothing
    (x's fp16 copy goes to a fixed array of NOALLOC_MAX_X_ELEMS values)."""
    _dev(w_tiled, torch.uint8, "w_tiled")
    _dev(x, torch.bfloat16, "x")
    _dev(out, torch.float32, "out")
    M, K = x.shape
    if tuple(out.shape) != (M, N):
        raise ValueError("out must be [M, N]")
    _check(library().q4k_gemm_noalloc(_ptr(w_tiled), _ptr(x), _ptr(out), M, N, K, _stream(x)),
           "q4k_gemm_noalloc")
    return out


def q8_activation_bytes(M: int, K: int) -> int:
    out = ctypes.c_size_t()
    _check(library().q8_activation_bytes(M, K, ctypes.byref(out)), "q8_activation_bytes")
    return out.value


def q8_quantize(x: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """bf16 activations [M, K] -> the quantized-activation records (uint8,
    q8_activation_bytes(M, K) bytes): 8-bit codes per block of 32, fp32 scales."""
    _dev(x, torch.bfloat16, "x")
    M, K = x.shape
    nbytes = q8_activation_bytes(M, K)
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=x.device)
    _dev(out, torch.uint8, "out")
    if out.numel() < nbytes:
        raise ValueError("out is smaller than q8_activation_bytes(M, K)")
    _check(library().q8_quantize(_ptr(x), _ptr(out), M, K, _stream(x)), "q8_quantize")
    return out


def q4k_q8_gemm(w_tiled: torch.Tensor, xq: torch.Tensor, M: int, N: int, K: int,
                out: torch.Tensor | None = None) -> torch.Tensor:
    """y[M, N] (fp32) = the Q4_K product with quantized activations xq (from
    q8_quantize of an [M, K] x), 1 <= M <= 8."""
    _dev(w_tiled, torch.uint8, "w_tiled")
    _dev(xq, torch.uint8, "xq")
    if xq.numel() < q8_activation_bytes(M, K):
        raise ValueError("xq is smaller than q8_activation_bytes(M, K)")
    if out is None:
        out = torch.empty(M, N, dtype=torch.float32, device=xq.device)
    _dev(out, torch.float32, "out")
    _check(library().q4k_q8_gemm(_ptr(w_tiled), _ptr(xq), _ptr(out), M, N, K, _stream(xq)), "q4k_q8_gemm")
    return out


def q6k_repacked_bytes(N: int, K: int) -> int:
    out = ctypes.c_size_t()
    _check(library().q6k_repacked_bytes(N, K, ctypes.byref(out)), "q6k_repacked_bytes")
    return out.value


def q6k_repack(w_ggml: torch.Tensor, N: int, K: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """GGML Q6_K rows (uint8, N*K/256*210 bytes) -> tile-major repacked bytes (q6k_repacked_bytes)."""
    _dev(w_ggml, torch.uint8, "w_ggml")
    if K % 256 or w_ggml.numel() != N * (K // 256) * 210:
        raise ValueError("w_ggml size does not match N, K")
    nbytes = q6k_repacked_bytes(N, K)
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=w_ggml.device)
    _dev(out, torch.uint8, "out")
    if out.numel() != nbytes:
        raise ValueError("out must hold q6k_repacked_bytes(N, K) bytes")
    _check(library().q6k_repack(_ptr(w_ggml), _ptr(out), N, K, _stream(w_ggml)), "q6k_repack")
    return out


def q6k_dequant(w_tiled: torch.Tensor, N: int, K: int, out: torch.Tensor | None = None) -> torch.Tensor:
    _dev(w_tiled, torch.uint8, "w_tiled")
    if out is None:
        out = torch.empty(N, K, dtype=torch.float32, device=w_tiled.device)
    _dev(out, torch.float32, "out")
    _check(library().q6k_dequant(_ptr(w_tiled), _ptr(out), N, K, _stream(w_tiled)), "q6k_dequant")
    return out


def _q6k_gemm_call(entry, x_dtype, w_tiled, x, N, out):
    _dev(w_tiled, torch.uint8, "w_tiled")
    _dev(x, x_dtype, "x")
    M, K = x.shape
    if out is None:
        out = torch.empty(M, N, dtype=torch.float32, device=x.device)
    _dev(out, torch.float32, "out")
    _check(getattr(library(), entry)(_ptr(w_tiled), _ptr(x), _ptr(out), M, N, K, _stream(x)), entry)
    return out


def q6k_gemm(w_tiled: torch.Tensor, x: torch.Tensor, N: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """y[M, N] (fp32) = x[M, K] (bf16) . W^T with W the repacked Q6_K matrix."""
    return _q6k_gemm_call("q6k_gemm", torch.bfloat16, w_tiled, x, N, out)


def q6k_gemm_f16(w_tiled: torch.Tensor, x: torch.Tensor, N: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """y[M, N] (fp32) = x[M, K] (fp16) . W^T with W the repacked Q6_K matrix."""
    return _q6k_gemm_call("q6k_gemm_f16", torch.float16, w_tiled, x, N, out)


def w4a16_repack(wq: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """Interleaved int4 words [N, K/8] (int32) -> tile-major repacked words (same size)."""
    _dev(wq, torch.int32, "wq")
    N, K8 = wq.shape
    if out is None:
        out = torch.empty_like(wq)
    _dev(out, torch.int32, "out")
    _check(library().w4a16_repack(_ptr(wq), _ptr(out), N, K8 * 8, _stream(wq)), "w4a16_repack")
    return out


def w4a16_dequant(wq_tiled, scales, zeros, N: int, K: int, group: int, out=None) -> torch.Tensor:
    """Exact fp32 s*(q - zp) of a repacked W4A16 matrix; zeros=None is the symmetric form (zp = 8)."""
    _dev(wq_tiled, torch.int32, "wq_tiled")
    _dev(scales, torch.float16, "scales")
    if zeros is not None:
        _dev(zeros, torch.uint8, "zeros")
    if out is None:
        out = torch.empty(N, K, dtype=torch.float32, device=wq_tiled.device)
    _dev(out, torch.float32, "out")
    _check(library().w4a16_dequant(_ptr(wq_tiled), _ptr(scales), _ptr(zeros), _ptr(out), N, K, group,
                                   _stream(wq_tiled)), "w4a16_dequant")
    return out


def _w4a16_gemm_call(entry, x_dtype, wq_tiled, scales, zeros, x, N, group, out):
    _dev(wq_tiled, torch.int32, "wq_tiled")
    _dev(scales, torch.float16, "scales")
    if zeros is not None:
        _dev(zeros, torch.uint8, "zeros")
    _dev(x, x_dtype, "x")
    M, K = x.shape
    if out is None:
        out = torch.empty(M, N, dtype=torch.float32, device=x.device)
    _dev(out, torch.float32, "out")
    _check(getattr(library(), entry)(_ptr(wq_tiled), _ptr(scales), _ptr(zeros), _ptr(x), _ptr(out), M, N, K,
                                     group, _stream(x)), entry)
    return out


def w4a16_gemm(wq_tiled, scales, zeros, x: torch.Tensor, N: int, group: int, out=None) -> torch.Tensor:
    """y[M, N] (fp32) = x[M, K] (fp16) . W^T with W the repacked W4A16 matrix
    (zeros=None: symmetric, zero point 8)."""
    return _w4a16_gemm_call("w4a16_gemm", torch.float16, wq_tiled, scales, zeros, x, N, group, out)


def w4a16_gemm_bf16(wq_tiled, scales, zeros, x: torch.Tensor, N: int, group: int, out=None) -> torch.Tensor:
    """As w4a16_gemm with bf16 activations (converted to fp16 on the GPU first)."""
    return _w4a16_gemm_call("w4a16_gemm_bf16", torch.bfloat16, wq_tiled, scales, zeros, x, N, group, out)


def device_status(device=None) -> int:
    """Synchronize the current stream and return (and clear) the library's device status code."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return int(library().qwp_device_status(ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)))


def set_decode_policy(policy: int) -> int:
    """Set which decode-shaped products run on the decode kernel (DECODE_AUTO,
    DECODE_NEVER or DECODE_ALWAYS; process-wide) and return the previous policy."""
    rc = int(library().qwp_set_decode_policy(int(policy)))
    if rc < 0:
        _check(rc, "qwp_set_decode_policy")
    return rc


_PLAN_FORMATS = {"w4a16": 0, "q4k": 1, "q6k": 2}


def decode_selected(fmt: str, M: int, N: int, K: int) -> bool:
    """Whether a GEMM call of this weight format ("q4k", "q6k", "w4a16") and shape
    would run the decode kernel now."""
    rc = library().qwp_decode_selected(_PLAN_FORMATS[fmt], int(M), int(N), int(K))
    if rc < 0:
        _check(rc, "qwp_decode_selected")
    return bool(rc)


def gemm_plan(fmt: str, M: int, N: int, K: int) -> dict:
    """The launch a GEMM call of this shape gets on the current device: kernel
    ("prefill", "decode" or "skinny"), split-K factor, clusters, token tile, units
    and units per cluster (zero for the decode kernel; the skinny-N kernel reports
    its cluster size, token tiles, tokens per tile (<= 128), token tiles and 1)."""
    out = (ctypes.c_int32 * 6)()
    _check(library().qwp_gemm_plan(_PLAN_FORMATS[fmt], int(M), int(N), int(K), ctypes.cast(out, ctypes.c_void_p)),
           "qwp_gemm_plan")
    return {"kernel": {1: "prefill", 2: "decode", 3: "skinny"}[out[0]], "splits": out[1], "clusters": out[2],
            "token_tile": out[3], "units": out[4], "units_per_cluster": out[5]}


# The prefill kernel's default bound on a main-loop wait (qwp_set_wait_timeout_ns).
DEFAULT_WAIT_TIMEOUT_NS = 2_000_000_000


def set_wait_timeout_ns(ns: int) -> None:
    """Set the bound on the prefill kernel's main-loop waits (process-wide); calls
    launched afterwards use it."""
    _check(library().qwp_set_wait_timeout_ns(int(ns)), "qwp_set_wait_timeout_ns")
