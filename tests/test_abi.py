"""Host-side checks of the C ABI that need no GPU: the library builds, loads and
exports every entry point include/mq.h declares; size helpers and the
validation that runs before any CUDA call."""
import ctypes
import os
import re

import pytest

from quant_int8_quantized_gb300 import build as B
from quant_int8_quantized_gb300 import mq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    B.build()
    return mq.lib()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(mq_\w+)\s*\(", src))
    return names


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert {"mq_quantize_q8", "mq_rms_quant", "mq_swiglu_quant", "mq_gemm_q4k", "mq_gemm_q6k",
            "mq_gemv_q4k", "mq_gemv_q6k", "mq_gemv_q6k_packed"} <= names
    for n in names:
        assert hasattr(L, n), n
    assert names <= set(mq.EXPORTED) | names  # the binding wraps what it knows


def test_binding_covers_every_declared_symbol(L):
    assert declared_functions() <= set(mq.EXPORTED)


def test_size_helpers(L):
    tot, qs, d, s, ah, ax, af = mq.mq_plane_bytes(3314, 3584)
    assert (qs, d, s) == (3314 * 3584, 3314 * 112 * 4, 3314 * 112 * 4)
    assert (ah, ax, af) == (3314 * 3584 * 2, 3314 * 14 * 32, 14 * 3316 * 4)
    assert tot == qs + d + s + ah + ax + af
    assert mq.mq_q4k_row_bytes(3584) == 14 * 144
    assert mq.mq_q6k_row_bytes(18944) == 74 * 210
    assert mq.mq_q5k_row_bytes(5120) == 20 * 176
    assert mq.mq_q4_0_row_bytes(5120) == 160 * 18
    assert mq.mq_q4_1_row_bytes(5120) == 160 * 20


def test_status_strings(L):
    for code in range(7):
        assert mq.status_str(code).startswith("MQ_")
    assert "UNKNOWN" in mq.status_str(99)


def _plane(M, K, qs=1, d=1, s=1, ah=None, ax=None, af=None):
    return mq.CPlane(qs, d, s, ah, ax, af, M, K)


def test_validation_before_any_cuda_call(L):
    null = None
    # K not a positive multiple of 256
    p = _plane(4, 100)
    assert L.mq_quantize_q8(ctypes.c_void_p(16), 4, 100, ctypes.byref(p), null) == mq.MQ_ERR_SHAPE
    p = _plane(4, 0)
    assert L.mq_rms_quant(ctypes.c_void_p(16), ctypes.c_void_p(16), 4, 0, 1e-6, ctypes.byref(p), null) == mq.MQ_ERR_SHAPE
    # negative M
    p = _plane(-1, 256)
    assert L.mq_swiglu_quant(ctypes.c_void_p(16), ctypes.c_void_p(16), -1, 256, ctypes.byref(p), null) == mq.MQ_ERR_SHAPE
    # NULL plane
    assert L.mq_quantize_q8(ctypes.c_void_p(16), 4, 256, None, null) == mq.MQ_ERR_NULL
    # plane dims disagree with the call
    p = _plane(5, 256)
    assert L.mq_quantize_q8(ctypes.c_void_p(16), 4, 256, ctypes.byref(p), null) == mq.MQ_ERR_SHAPE
    # empty input is a no-op
    p = _plane(0, 256, 0, 0, 0)
    assert L.mq_quantize_q8(None, 0, 256, ctypes.byref(p), null) == mq.MQ_OK
    # NULL plane arrays / inputs, misaligned pointers
    p = _plane(4, 256, 0, 16, 16)
    assert L.mq_quantize_q8(ctypes.c_void_p(16), 4, 256, ctypes.byref(p), null) == mq.MQ_ERR_NULL
    p = _plane(4, 256, 16, 16, 16)
    assert L.mq_quantize_q8(None, 4, 256, ctypes.byref(p), null) == mq.MQ_ERR_NULL
    p = _plane(4, 256, 17, 16, 16)
    assert L.mq_quantize_q8(ctypes.c_void_p(16), 4, 256, ctypes.byref(p), null) == mq.MQ_ERR_ALIGN
    p = _plane(4, 256, 16, 16, 16)
    assert L.mq_quantize_q8(ctypes.c_void_p(20), 4, 256, ctypes.byref(p), null) == mq.MQ_ERR_ALIGN


def test_matmul_validation_before_any_cuda_call(L):
    null = None
    p = _plane(mq.MQ_GEMV_MAX_ROWS + 1, 512, 16, 16, 16)
    gemvs = (L.mq_gemv_q4k, L.mq_gemv_q6k, L.mq_gemv_q5k, L.mq_gemv_q4_0, L.mq_gemv_q4_1, L.mq_gemv_q6k_packed)
    for fn in gemvs:
        assert fn(ctypes.byref(p), ctypes.c_void_p(16), 8, ctypes.c_void_p(16), null) == mq.MQ_ERR_SHAPE  # M > 8
        assert fn(ctypes.byref(_plane(0, 512, 16, 16, 16)), ctypes.c_void_p(16), 8, ctypes.c_void_p(16), null) == mq.MQ_ERR_SHAPE
    p1 = _plane(1, 512, 16, 16, 16, 16, 16, 16)
    gemms = (L.mq_gemm_q4k, L.mq_gemm_q6k, L.mq_gemm_q4_0, L.mq_gemm_q4_1)
    for fn in gemms + gemvs:
        assert fn(None, ctypes.c_void_p(16), 8, ctypes.c_void_p(16), null) == mq.MQ_ERR_NULL
        assert fn(ctypes.byref(p1), None, 8, ctypes.c_void_p(16), null) == mq.MQ_ERR_NULL
        assert fn(ctypes.byref(p1), ctypes.c_void_p(16), 8, None, null) == mq.MQ_ERR_NULL
        assert fn(ctypes.byref(p1), ctypes.c_void_p(24), 8, ctypes.c_void_p(16), null) == mq.MQ_ERR_ALIGN
        assert fn(ctypes.byref(p1), ctypes.c_void_p(16), -1, ctypes.c_void_p(16), null) == mq.MQ_ERR_SHAPE
        assert fn(ctypes.byref(p1), ctypes.c_void_p(16), 0, None, null) == mq.MQ_OK      # N == 0: no-op
    bad = _plane(1, 300, 16, 16, 16)
    assert L.mq_gemm_q4k(ctypes.byref(bad), ctypes.c_void_p(16), 8, ctypes.c_void_p(16), null) == mq.MQ_ERR_SHAPE
    # the GEMM needs the operand arrays, the GEMV the q8 arrays; a group is all present or all
    # absent, and a misaligned array is rejected everywhere
    for fn in gemms:
        assert fn(ctypes.byref(_plane(4, 512, 16, 16, 16)), ctypes.c_void_p(16), 8, ctypes.c_void_p(16), null) == mq.MQ_ERR_NULL
        assert fn(ctypes.byref(_plane(4, 512, 16, 16, 16, 40, 16, 16)), ctypes.c_void_p(16), 8, ctypes.c_void_p(16), null) == mq.MQ_ERR_ALIGN
        assert fn(ctypes.byref(_plane(4, 512, 16, 16, 16, 16, None, 16)), ctypes.c_void_p(16), 8, ctypes.c_void_p(16), null) == mq.MQ_ERR_NULL
    for fn in gemvs:
        assert fn(ctypes.byref(_plane(1, 512, None, None, None, 16, 16, 16)), ctypes.c_void_p(16), 8, ctypes.c_void_p(16), null) == mq.MQ_ERR_NULL
    p8 = _plane(4, 256, 16, 16, 16, 16, 16, 24)
    assert L.mq_quantize_q8(ctypes.c_void_p(16), 4, 256, ctypes.byref(p8), null) == mq.MQ_ERR_ALIGN
    p9 = _plane(4, 256, None, None, None)
    assert L.mq_quantize_q8(ctypes.c_void_p(16), 4, 256, ctypes.byref(p9), null) == mq.MQ_ERR_NULL
    p10 = _plane(4, 256, 16, None, 16)
    assert L.mq_quantize_q8(ctypes.c_void_p(16), 4, 256, ctypes.byref(p10), null) == mq.MQ_ERR_NULL


def test_pair_and_static_gemm_validation_before_any_cuda_call(L):
    """mq_gemm_q4k_pair checks both problems (either one's bad argument is reported before
    anything runs); mq_gemm_q6k_static checks as mq_gemm_q6k does."""
    null = None
    p1 = _plane(1, 512, 16, 16, 16, 16, 16, 16)
    fn = L.mq_gemm_q4k_pair
    fn.restype = ctypes.c_int
    v = ctypes.c_void_p
    assert fn(None, v(16), 8, v(16), v(16), 8, v(16), null) == mq.MQ_ERR_NULL
    assert fn(ctypes.byref(p1), None, 8, v(16), v(16), 8, v(16), null) == mq.MQ_ERR_NULL
    assert fn(ctypes.byref(p1), v(16), 8, v(16), None, 8, v(16), null) == mq.MQ_ERR_NULL
    assert fn(ctypes.byref(p1), v(16), 8, v(16), v(16), 8, None, null) == mq.MQ_ERR_NULL
    assert fn(ctypes.byref(p1), v(16), 8, v(16), v(24), 8, v(16), null) == mq.MQ_ERR_ALIGN
    assert fn(ctypes.byref(p1), v(16), -1, v(16), v(16), 8, v(16), null) == mq.MQ_ERR_SHAPE
    assert fn(ctypes.byref(p1), v(16), 8, v(16), v(16), -1, v(16), null) == mq.MQ_ERR_SHAPE
    assert fn(ctypes.byref(_plane(1, 300, 16, 16, 16, 16, 16, 16)), v(16), 8, v(16), v(16), 8, v(16), null) == mq.MQ_ERR_SHAPE
    s = L.mq_gemm_q6k_static
    s.restype = ctypes.c_int
    assert s(None, v(16), 8, v(16), null) == mq.MQ_ERR_NULL
    assert s(ctypes.byref(p1), v(24), 8, v(16), null) == mq.MQ_ERR_ALIGN
    assert s(ctypes.byref(p1), v(16), -1, v(16), null) == mq.MQ_ERR_SHAPE
    assert s(ctypes.byref(p1), v(16), 0, None, null) == mq.MQ_OK      # N == 0: no-op
    assert mq.status_str(mq.MQ_ERR_SCRATCH).startswith("MQ_ERR_SCRATCH")
