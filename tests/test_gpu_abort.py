"""The GEMM's failure paths, exercised without a GPU fault: a test build of the library
(50 ms wait limit, switches that make CTA 0's TMA producer skip its first activation copy,
or the first K slice of an ordered split never pass its tile on) runs a GEMM whose bounded
waits must run out. The kernel must return, record the failure so that mq_device_status
reports MQ_ERR_DEVICE once (and clears it), and leave the context usable: the next GEMM,
with the switch off, is correct."""
import ctypes

import numpy as np
import pytest
import torch

from oracle import mq_oracle as O
from quant_int8_quantized_gb300 import build as B
from quant_int8_quantized_gb300 import mq, synth
from tests._gpu_util import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    require_gpu()
    path = B.build_variant("inject", ["MQ_TEST_INJECT", "MQ_WAIT_LIMIT_NS=50000000ull"])
    lib = ctypes.CDLL(path)
    vp, i, pp = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(mq.CPlane)
    for name, args in (("mq_quantize_q8", [vp, i, i, pp, vp]), ("mq_gemm_q4k", [pp, vp, i, vp, vp]),
                       ("mq_gemm_q6k", [pp, vp, i, vp, vp]), ("mq_prepack_q6k", [vp, i, i, vp, vp]),
                       ("mq_device_status", [vp]), ("mq_test_inject", [i])):
        getattr(lib, name).restype = i
        getattr(lib, name).argtypes = args
    return lib


def _gemm(L, p, w, N, out):
    cp = p.c()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.mq_gemm_q4k(ctypes.byref(cp), ctypes.c_void_p(w.data_ptr()), N, ctypes.c_void_p(out.data_ptr()), stream)


@pytest.mark.parametrize("M", [384, 16])   # full tiles; the short-tile form (16 tokens)
def test_gemm_wait_runs_out_and_is_reported_then_recovers(L, M):
    N, K = 640, 1024
    x = synth.normal((M, K), 0, f"ab.x{M}", device="cuda")
    w = synth.weights("q4k", N, K, 0, "ab.w", device="cuda")
    p = mq.Plane.empty(M, K)
    cp = p.c()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.mq_quantize_q8(ctypes.c_void_p(x.data_ptr()), M, K, ctypes.byref(cp), stream) == mq.MQ_OK
    out = torch.zeros((M, N), device="cuda")
    null = ctypes.c_void_p(0)
    assert L.mq_device_status(null) == mq.MQ_OK

    assert L.mq_test_inject(1) == mq.MQ_OK
    assert _gemm(L, p, w, N, out) == mq.MQ_OK          # the launch itself succeeds
    assert L.mq_device_status(null) == mq.MQ_ERR_DEVICE   # a bounded wait ran out
    assert L.mq_device_status(null) == mq.MQ_OK           # and the record was cleared

    assert L.mq_test_inject(0) == mq.MQ_OK
    out.fill_(float("nan"))
    assert _gemm(L, p, w, N, out) == mq.MQ_OK
    assert L.mq_device_status(null) == mq.MQ_OK
    ref, bound = O.gemm_rows(p.qs.cpu().numpy(), p.d.cpu().numpy(), w.cpu().numpy(), "q4k", N, K)
    got = out.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= bound)


def test_ordered_split_wait_runs_out_and_is_reported_then_recovers(L):
    """q6_K at 1000 x 3456 x 8192 (162 tiles on 152 SMs: the last 10 tiles run as ordered K
    slices): with the first slices' flags never passed on, the later slices give up after the
    wait limit; the next call, with the switch off, is correct on sampled rows."""
    M, N, K = 1000, 3456, 8192
    x = synth.normal((M, K), 0, "ab6.x", device="cuda")
    w_raw = synth.weights("q6k", N, K, 0, "ab6.w")
    wd = w_raw.cuda()
    wp = torch.empty((N, (K // 256) * 224), dtype=torch.uint8, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.mq_prepack_q6k(ctypes.c_void_p(wd.data_ptr()), N, K, ctypes.c_void_p(wp.data_ptr()), stream) == mq.MQ_OK
    p = mq.Plane.empty(M, K)
    cp = p.c()
    assert L.mq_quantize_q8(ctypes.c_void_p(x.data_ptr()), M, K, ctypes.byref(cp), stream) == mq.MQ_OK
    out = torch.zeros((M, N), device="cuda")
    null = ctypes.c_void_p(0)
    assert L.mq_device_status(null) == mq.MQ_OK

    def gemm():
        c = p.c()
        return L.mq_gemm_q6k(ctypes.byref(c), ctypes.c_void_p(wp.data_ptr()), N, ctypes.c_void_p(out.data_ptr()), stream)

    assert L.mq_test_inject(2) == mq.MQ_OK
    assert gemm() == mq.MQ_OK                          # the launches themselves succeed
    assert L.mq_device_status(null) == mq.MQ_ERR_DEVICE   # the slices' waits ran out
    assert L.mq_device_status(null) == mq.MQ_OK           # and the record was cleared

    assert L.mq_test_inject(0) == mq.MQ_OK
    for _ in range(2):
        out.fill_(float("nan"))
        assert gemm() == mq.MQ_OK
        assert L.mq_device_status(null) == mq.MQ_OK
        rows = np.r_[0, 500, np.arange(M - 12, M)]
        ref, bound = O.gemm_rows(p.qs.cpu().numpy(), p.d.cpu().numpy(), w_raw.numpy(), "q6k", N, K, rows=rows)
        got = out.cpu().numpy().astype(np.float64)[rows]
        assert np.all(np.abs(got - ref) <= bound)
