"""The C-ABI library loads, exports every symbol include/qwp.h declares, and its
host-side argument checks return the documented codes (no GPU work is issued:
each call below is rejected before any CUDA call)."""
import ctypes
import os
import re

import pytest

import quantized_weight_prefill_gb300 as qwp
from quantized_weight_prefill_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qwp.h")

OK, INVALID, SHAPE, MISALIGNED = 0, -1, -2, -3


@pytest.fixture(scope="module")
def lib():
    if _build.is_stale():
        _build.build()
    return qwp.library()


def declared_functions():
    text = open(HEADER).read()
    return set(re.findall(r"^QWP_API\s+(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, re.M))


def test_header_declares_the_binding_symbols():
    assert declared_functions() == set(qwp.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    # and nothing else: internal helpers are hidden
    out = os.popen(f"nm -D --defined-only {_build.LIB}").read().split("\n")
    exported = {line.split()[-1] for line in out if " T " in line}
    assert exported == declared_functions()


def test_status_strings(lib):
    for code, name in [(0, "QWP_OK"), (-1, "QWP_ERR_INVALID_ARG"), (-2, "QWP_ERR_UNSUPPORTED_SHAPE"),
                       (-3, "QWP_ERR_MISALIGNED"), (-4, "QWP_ERR_CUDA"), (-5, "QWP_ERR_DEVICE"),
                       (-6, "QWP_ERR_TIMEOUT"), (-7, "QWP_ERR_RANGE")]:
        assert lib.qwp_status_string(code).decode() == name


def test_q8_activation_bytes(lib):
    assert qwp.q8_activation_bytes(1, 4096) == 16 * 2560
    assert qwp.q8_activation_bytes(8, 256) == 2560
    assert qwp.q8_activation_bytes(9, 512) == 2 * 2 * 2560
    assert qwp.q8_activation_bytes(0, 512) == 0
    assert lib.q8_activation_bytes(4, 100, ctypes.byref(ctypes.c_size_t())) == SHAPE
    assert lib.q8_activation_bytes(-1, 256, ctypes.byref(ctypes.c_size_t())) == INVALID


def test_repacked_bytes(lib):
    assert qwp.q4k_repacked_bytes(4096, 4096) == 4096 * 16 * 144
    assert qwp.q4k_repacked_bytes(3, 512) == 3 * 2 * 144
    assert qwp.w4a16_repacked_bytes(12288, 4096) == 12288 * 4096 // 2
    # Q6_K: the last tile is padded to a multiple of 8 rows
    assert qwp.q6k_repacked_bytes(4096, 12288) == 4096 * 48 * 210
    assert qwp.q6k_repacked_bytes(130, 256) == (128 + 8) * 210
    assert qwp.q6k_repacked_bytes(1, 512) == 8 * 2 * 210
    assert lib.q6k_repacked_bytes(4, 100, ctypes.byref(ctypes.c_size_t())) == SHAPE
    with pytest.raises(qwp.QwpError) as e:
        qwp.q4k_repacked_bytes(4, 100)
    assert e.value.code == SHAPE
    out = ctypes.c_size_t()
    assert lib.q4k_repacked_bytes(-1, 256, ctypes.byref(out)) == INVALID
    assert lib.q4k_repacked_bytes(1, 256, None) == INVALID


def _p(v):
    return ctypes.c_void_p(v)


def test_gemm_argument_checks_before_any_cuda_call(lib):
    a16 = _p(0x1000)
    # shape errors
    assert lib.q4k_gemm(a16, a16, a16, 8, 8, 100, None) == SHAPE
    assert lib.q4k_gemm(a16, a16, a16, -1, 8, 256, None) == INVALID
    assert lib.w4a16_gemm(a16, a16, a16, a16, a16, 8, 8, 256, 100, None) == INVALID   # group % 64
    assert lib.w4a16_gemm(a16, a16, a16, a16, a16, 8, 8, 320, 128, None) == SHAPE     # K % group
    # null and misaligned pointers
    assert lib.q4k_gemm(None, a16, a16, 8, 8, 256, None) == INVALID
    assert lib.q4k_gemm(_p(0x1004), a16, a16, 8, 8, 256, None) == MISALIGNED
    assert lib.q4k_gemm(a16, _p(0x1002), a16, 8, 8, 256, None) == MISALIGNED
    assert lib.w4a16_gemm(a16, None, a16, a16, a16, 8, 8, 256, 128, None) == INVALID
    assert lib.w4a16_gemm_bf16(a16, None, None, a16, a16, 8, 8, 256, 128, None) == INVALID  # scales required
    assert lib.w4a16_gemm_bf16(a16, a16, None, a16, a16, 8, 8, 256, 100, None) == INVALID   # group % 64
    assert lib.w4a16_gemm_bf16(a16, a16, None, a16, a16, 8, 8, 320, 128, None) == SHAPE     # K % group
    assert lib.w4a16_gemm_bf16(a16, a16, None, _p(0x1002), a16, 8, 8, 256, 128, None) == MISALIGNED
    assert lib.w4a16_gemm_bf16(None, None, None, None, None, 0, 8, 256, 128, None) == OK
    # empty problems are no-ops
    assert lib.q4k_gemm(None, None, None, 0, 8, 256, None) == OK
    assert lib.q4k_gemm(None, None, None, 8, 0, 256, None) == OK
    assert lib.q4k_gemm_f16(a16, a16, a16, 8, 8, 100, None) == SHAPE
    assert lib.q4k_gemm_f16(a16, _p(0x1008), a16, 8, 8, 256, None) == MISALIGNED
    assert lib.q6k_gemm(a16, a16, a16, 8, 8, 100, None) == SHAPE
    assert lib.q6k_gemm(None, a16, a16, 8, 8, 256, None) == INVALID
    assert lib.q6k_gemm_f16(a16, _p(0x1004), a16, 8, 8, 256, None) == MISALIGNED
    assert lib.q6k_gemm(None, None, None, 0, 8, 256, None) == OK
    assert lib.q6k_repack(a16, a16, 4, 256, None) == INVALID          # aliasing
    assert lib.q6k_dequant(a16, _p(0x2008), 4, 300, None) == SHAPE
    # repack / dequant checks
    assert lib.q4k_repack(a16, a16, 4, 256, None) == INVALID          # aliasing
    assert lib.q4k_repack(a16, _p(0x2008), 4, 256, None) == MISALIGNED
    assert lib.q4k_dequant(a16, a16, 4, 300, None) == SHAPE
    assert lib.w4a16_repack(a16, a16, 4, 96, None) == SHAPE
    assert lib.w4a16_dequant(a16, a16, a16, a16, 4, 256, 96, None) == INVALID
    # quantized activations
    assert lib.q8_quantize(a16, a16, 4, 100, None) == SHAPE
    assert lib.q8_quantize(a16, a16, -1, 256, None) == INVALID
    assert lib.q8_quantize(None, a16, 4, 256, None) == INVALID
    assert lib.q8_quantize(a16, _p(0x2008), 4, 256, None) == MISALIGNED
    assert lib.q8_quantize(None, None, 0, 256, None) == OK
    assert lib.q4k_q8_gemm(a16, a16, a16, 9, 8, 256, None) == SHAPE    # more than 8 tokens
    assert lib.q4k_q8_gemm(a16, a16, a16, 8, 8, 100, None) == SHAPE
    assert lib.q4k_q8_gemm(None, a16, a16, 8, 8, 256, None) == INVALID
    assert lib.q4k_q8_gemm(a16, _p(0x1008), a16, 8, 8, 256, None) == MISALIGNED
    assert lib.q4k_q8_gemm(None, None, None, 0, 8, 256, None) == OK
    # batched
    assert lib.q4k_gemm_batched(a16, a16, a16, -1, 8, 8, 256, None) == INVALID
    assert lib.q4k_gemm_batched(a16, a16, a16, 2, 8, 8, 100, None) == SHAPE
    assert lib.q4k_gemm_batched(a16, a16, a16, 70000, 8, 8, 256, None) == SHAPE
    assert lib.q4k_gemm_batched(None, a16, a16, 2, 8, 8, 256, None) == INVALID
    assert lib.q4k_gemm_batched_f16(a16, _p(0x1008), a16, 2, 8, 8, 256, None) == MISALIGNED
    assert lib.q4k_gemm_batched(None, None, None, 0, 8, 8, 256, None) == OK
    assert lib.q4k_gemm_batched_f16(None, None, None, 3, 0, 8, 256, None) == OK


def test_decode_policy_round_trip_and_automatic_rule(lib):
    """The dispatch between the decode and the prefill kernel is host logic: the
    automatic rule (at most two tokens; N >= 24576 for Q4_K, N >= 65536 for Q6_K,
    N >= 24576 at one token and N >= 65536 at two for W4A16; plus what the decode
    kernel needs: K % 256 == 0 and >= 600 tile items), the two forced policies,
    and the rejection of an unknown policy or format."""
    sel = qwp.decode_selected
    prev = qwp.set_decode_policy(qwp.DECODE_AUTO)
    try:
        for f in ("q4k", "q6k", "w4a16"):
            assert sel(f, 1, 152064, 4096) and sel(f, 1, 65536, 4096) and sel(f, 2, 65536, 4096)
            assert sel(f, 1, 65600, 512)                 # 513 x 2 = 1026 items
            assert not sel(f, 3, 152064, 4096)           # three tokens: the prefill kernel
            assert not sel(f, 1, 12288, 4096)            # narrow
            assert not sel(f, 1, 152064, 4000)           # K % 256 != 0
            assert not sel(f, 1, 65536, 256)             # 512 x 1 = 512 items
            assert not sel(f, 0, 152064, 4096)
        assert sel("q4k", 1, 24576, 4096) and sel("q4k", 2, 24576, 4096)
        assert not sel("q4k", 1, 24448, 4096)            # 191 row tiles
        assert not sel("q6k", 1, 24576, 4096) and not sel("q6k", 1, 65408, 4096)
        assert sel("w4a16", 1, 24576, 4096) and not sel("w4a16", 2, 24576, 4096)
        assert lib.qwp_decode_selected(3, 1, 152064, 4096) == INVALID
        assert lib.qwp_decode_selected(-1, 1, 152064, 4096) == INVALID
        assert qwp.set_decode_policy(qwp.DECODE_ALWAYS) == qwp.DECODE_AUTO
        for f in ("q4k", "q6k", "w4a16"):
            assert sel(f, 8, 4096, 12288) and sel(f, 5, 2500, 8192)
            assert not sel(f, 9, 24576, 4096)            # more than 8 tokens
            assert not sel(f, 1, 2048, 2048)             # 16 x 8 = 128 items
        assert qwp.set_decode_policy(qwp.DECODE_NEVER) == qwp.DECODE_ALWAYS
        assert not sel("q4k", 1, 152064, 4096)
        assert lib.qwp_set_decode_policy(3) == INVALID and lib.qwp_set_decode_policy(-1) == INVALID
        with pytest.raises(qwp.QwpError):
            qwp.set_decode_policy(7)
        assert qwp.set_decode_policy(qwp.DECODE_AUTO) == qwp.DECODE_NEVER
    finally:
        qwp.set_decode_policy(prev)


def test_gemm_plan_argument_checks(lib):
    """qwp_gemm_plan rejects bad arguments before touching the device; decode-shaped
    products are answered on the host."""
    out = (ctypes.c_int32 * 6)()
    p = ctypes.cast(out, ctypes.c_void_p)
    assert lib.qwp_gemm_plan(1, 105, 24576, 4096, None) == INVALID
    assert lib.qwp_gemm_plan(3, 105, 24576, 4096, p) == INVALID          # no such format
    assert lib.qwp_gemm_plan(1, 0, 24576, 4096, p) == INVALID
    assert lib.qwp_gemm_plan(1, 105, 24576, 4000, p) == SHAPE            # Q4_K: K % 256
    assert lib.qwp_gemm_plan(2, 105, 24576, 4032, p) == SHAPE            # Q6_K: K % 256
    assert lib.qwp_gemm_plan(0, 105, 24576, 4000, p) == SHAPE            # W4A16: K % 64
    assert lib.qwp_gemm_plan(1, 105, 1 << 31, 4096, p) == SHAPE
    prev = qwp.set_decode_policy(qwp.DECODE_ALWAYS)
    try:
        assert lib.qwp_gemm_plan(1, 1, 24576, 4096, p) == OK and list(out) == [2, 0, 0, 0, 0, 0]
    finally:
        qwp.set_decode_policy(prev)


def test_wait_limit_argument_checks(lib):
    """qwp_set_wait_timeout_ns is host-only: it rejects 0 and more than 60 s."""
    assert lib.qwp_set_wait_timeout_ns(0) == INVALID
    assert lib.qwp_set_wait_timeout_ns(61_000_000_000) == INVALID
    assert lib.qwp_set_wait_timeout_ns(qwp.DEFAULT_WAIT_TIMEOUT_NS) == OK
