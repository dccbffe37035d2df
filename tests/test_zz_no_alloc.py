"""mq_gemm_q6k_static: the q6_K prefill GEMM for callers that cannot have device memory
allocated for them, such as a server whose device memory all belongs to its own pool, or code
that must not risk the device-wide synchronisation a cudaMalloc can cause. Its scratch (the
flags of an ordered split) is a fixed array inside the library.

Checked through the C ABI against mq_gemm_q6k on the same inputs, within the tolerance of the
other GEMM parity tests (1e-3 * sum_k |a||w| per element, from the oracle), on two calls in a
row. The shapes cover the path that uses the scratch (tile counts whose last round is cut into
ordered K slices: 504, 162 and 220 tiles on 152 SMs) and one that does not use it.

The file name sorts last, so a run that stops at its first failure has run every other test
before this one."""
import ctypes

import numpy as np
import pytest
import torch

from oracle import mq_oracle as O
from quant_int8_quantized_gb300 import mq, synth
from tests._gpu_util import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _call(name, plane, w, N, out):
    """One GEMM entry point, called through the C ABI on the current stream."""
    cp = plane.c()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return getattr(mq.lib(), name)(ctypes.byref(cp), ctypes.c_void_p(w.data_ptr()), int(N),
                                   ctypes.c_void_p(out.data_ptr()), stream)


@pytest.mark.parametrize("M,N,K", [(3314, 3584, 18944), (1000, 3456, 8192), (2000, 2560, 16384), (200, 768, 1024)])
def test_static_variant_matches_gemm_q6k(M, N, K):
    x = synth.normal((M, K), 0, f"na.x{M}x{K}", device="cuda")
    w_raw = synth.weights("q6k", N, K, 0, f"na.w{N}x{K}")
    w = mq.mq_prepack_q6k(w_raw.cuda(), N, K)
    p = mq.Plane.empty(M, K)
    mq.mq_quantize_q8(x, p)
    ref = torch.empty((M, N), device="cuda")
    assert _call("mq_gemm_q6k", p, w, N, ref) == mq.MQ_OK
    torch.cuda.synchronize()

    rng = np.random.default_rng(M + N + K)
    tail = np.arange(max(0, M - 400), M)
    rows = np.unique(np.r_[rng.choice(M, 12, replace=False), rng.choice(tail, min(12, len(tail)), replace=False), M - 1])
    _, bound = O.gemm_rows(p.qs.cpu().numpy(), p.d.cpu().numpy(), w_raw.numpy(), "q6k", N, K, rows=rows)
    want = ref.cpu().numpy().astype(np.float64)[rows]

    for call in range(2):   # two calls in a row share the scratch array
        out = torch.full((M, N), float("nan"), device="cuda")
        assert _call("mq_gemm_q6k_static", p, w, N, out) == mq.MQ_OK, f"call {call}"
        torch.cuda.synchronize()
        assert mq.mq_device_status() == mq.MQ_OK, f"call {call}: a bounded wait gave up"
        assert not torch.isnan(out).any(), f"call {call}: unwritten outputs"
        got = out.cpu().numpy().astype(np.float64)[rows]
        err = np.abs(got - want)
        assert np.all(err <= bound), f"call {call}: max diff/bound = {np.max(err / np.maximum(bound, 1e-30)):.3g}"
