"""The q6_K GEMV on prepacked rows (mq_gemv_q6k_packed) against the CPU oracle, which reads
the raw rows the packed ones were made from: every output within 1e-3 * sum_k |a||w| at
ragged and several-step shapes and 1..8 activation rows, each row of a multi-row call equal
to a one-row call, the bench's decode shapes at full size on sampled rows, and bit for bit
on integer-valued cases."""
import numpy as np
import pytest
import torch

from oracle import mq_oracle as O
from quant_int8_quantized_gb300 import mq, synth
from tests._gpu_util import Guarded, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _packed(w, N, K):
    return mq.mq_prepack_q6k(w.cuda(), N, K)


def _check(out, p, w, N, K, rows=None):
    ref, bound = O.gemm_rows(p.qs.cpu().numpy(), p.d.cpu().numpy(), w.cpu().numpy(), "q6k", N, K, rows=rows)
    got = out.cpu().numpy().astype(np.float64)
    if rows is not None:
        got = got[rows]
    err = np.abs(got - ref)
    assert np.all(err <= bound), f"max err/bound = {np.max(err / np.maximum(bound, 1e-30)):.3g}"


@pytest.mark.parametrize("N,K", [(256, 512), (1024, 5120), (100, 768), (1, 256), (7001, 3584), (3, 1280),
                                 (2049, 18944)])
def test_packed_gemv_parity(N, K):
    """One row: odd N (a lone last row), one super-block, a ragged last step (S not a multiple
    of 8), every element checked."""
    x = synth.with_outliers(synth.normal((1, K), 0, f"pg{N}x{K}"), 0, f"pgo{N}")
    w = synth.weights("q6k", N, K, 0, f"pgw{N}x{K}")
    p = mq.Plane.empty(1, K, op=False)
    mq.mq_quantize_q8(x.cuda(), p)
    g = Guarded((1, N), torch.float32)
    mq.mq_gemv_q6k_packed(p, _packed(w, N, K), N, g.t)
    torch.cuda.synchronize()
    g.check()
    assert g.untouched() == 0, "unwritten outputs"
    _check(g.t, p, w, N, K)


@pytest.mark.parametrize("M", [2, 3, 5, 8])
def test_packed_gemv_small_batch_every_element(M):
    """M activation rows: every element within the bound, and each row bit-identical to a
    one-row call on it."""
    N, K = 1001, 3584
    x = synth.with_outliers(synth.normal((M, K), 0, f"pbx{M}"), 0, f"pbo{M}")
    w = synth.weights("q6k", N, K, 0, "pbw")
    p = mq.Plane.empty(M, K, op=False)
    mq.mq_quantize_q8(x.cuda(), p)
    wp = _packed(w, N, K)
    g = Guarded((M, N), torch.float32)
    mq.mq_gemv_q6k_packed(p, wp, N, g.t)
    torch.cuda.synchronize()
    g.check()
    _check(g.t, p, w, N, K)
    for m in range(M):
        pm = mq.Plane(p.qs[m:m + 1], p.d[m:m + 1], p.s[m:m + 1])
        om = torch.empty(N, device="cuda")
        mq.mq_gemv_q6k_packed(pm, wp, N, om)
        assert torch.equal(om, g.t[m]), f"row {m}"


@pytest.mark.parametrize("N,K", [(5120, 13824), (2048, 5120), (152064, 3584)])
def test_packed_gemv_full_size_sampled_outputs(N, K):
    """The bench's decode shapes (down, k|v stacked) and the lm_head at full size; 512 sampled
    rows, always the first and the last."""
    x = synth.normal((1, K), 0, f"pf{K}", device="cuda")
    w = synth.weights("q6k", N, K, 0, f"pfw{N}", device="cuda")
    p = mq.Plane.empty(1, K, op=False)
    mq.mq_quantize_q8(x, p)
    g = Guarded((1, N), torch.float32)
    mq.mq_gemv_q6k_packed(p, mq.mq_prepack_q6k(w, N, K), N, g.t)
    torch.cuda.synchronize()
    g.check()
    assert g.untouched() == 0, "unwritten outputs"
    rows = np.unique(np.r_[np.random.default_rng(N).choice(N, 512, replace=False), 0, N - 1])
    rt = torch.as_tensor(rows, device="cuda")
    ref, bound = O.gemm_rows(p.qs.cpu().numpy(), p.d.cpu().numpy(), w[rt].cpu().numpy(), "q6k", len(rows), K)
    got = g.t[0, rt].cpu().numpy().astype(np.float64)[None, :]
    assert np.all(np.abs(got - ref) <= bound)
    assert mq.mq_device_status() == mq.MQ_OK


@pytest.mark.parametrize("N,K", [(33, 1280), (64, 2048), (9, 2304), (17, 8448)])
@pytest.mark.parametrize("M", [1, 3])
def test_packed_gemv_exact_integer_dots(N, K, M):
    """Unit super-block scales, sub-block scales of +-1 and integer activations whose every
    32-block holds a 127 (d_a = 1): every output is an exact integer below 2^24, so the GEMV
    on the packed rows must equal the f64 oracle on the raw rows bit for bit."""
    rng = np.random.default_rng(K + N + M)
    S = K // 256
    blk = rng.integers(0, 256, size=(N, S, 210), dtype=np.uint8)
    blk[:, :, 192:208] = rng.choice(np.array([-1, 1], np.int8), size=(N, S, 16)).view(np.uint8)
    blk[:, :, 208:210] = np.frombuffer(np.float16(1.0).tobytes(), np.uint8)
    w = torch.from_numpy(np.ascontiguousarray(blk.reshape(N, S * 210)))
    xi = rng.integers(-127, 128, size=(M, K)).astype(np.float32)
    for m in range(M):
        xi[m, rng.integers(0, 32) :: 32] = 127.0
    p = mq.Plane.empty(M, K, op=False)
    mq.mq_quantize_q8(torch.from_numpy(xi).cuda(), p)
    assert np.all(p.d.cpu().numpy() == 1.0)
    g = Guarded((M, N), torch.float32)
    mq.mq_gemv_q6k_packed(p, _packed(w, N, K), N, g.t)
    torch.cuda.synchronize()
    g.check()
    ref, _ = O.gemm_rows(p.qs.cpu().numpy(), p.d.cpu().numpy(), w.numpy(), "q6k", N, K)
    assert np.all(np.abs(ref) < 2 ** 24)
    assert np.array_equal(g.t.cpu().numpy().astype(np.float64), ref)
