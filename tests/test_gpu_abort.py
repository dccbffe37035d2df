"""The GEMM's failure path, exercised without a GPU fault: a test build of the library
(50 ms wait limit, a switch that makes CTA 0's TMA producer skip its first activation
copy) runs a GEMM whose bounded waits must run out. The kernel must return, record the
failure so that mq_device_status reports MQ_ERR_DEVICE once (and clears it), and leave
the context usable: the next GEMM, with the switch off, is correct."""
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
