"""Parity of the q5_K, q4_0 and q4_1 GEMVs (CUDA, through the C ABI) with the CPU
oracle: every output element within 1e-3 * sum_k |a||w| of the f64 reference on
seeded inputs (ragged N, several blocks per row, 1 to 8 activation rows), bit-exact
on integer-valued cases, and each row of a multi-row call bit-identical to a one-row
call on that row."""
import numpy as np
import pytest
import torch

from oracle import mq_oracle as O
from quant_int8_quantized_gb300 import mq, synth
from tests._gpu_util import Guarded, require_gpu

pytestmark = pytest.mark.gpu

KINDS = ["q5k", "q4_0", "q4_1"]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _plane(x):
    M, K = x.shape
    p = mq.Plane.empty(M, K, op=False)
    mq.mq_quantize_q8(x.cuda(), p)
    return p


def _check(out, p, w, kind, N, K):
    ref, bound = O.gemm_rows(p.qs.cpu().numpy(), p.d.cpu().numpy(), w.cpu().numpy(), kind, N, K)
    got = out.cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    assert np.all(err <= bound), f"{kind}: max err/bound = {np.max(err / np.maximum(bound, 1e-30)):.3g}"


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (1, 1000, 3584), (3, 7, 256), (8, 100, 768), (5, 333, 1280)])
def test_parity_every_element(kind, M, N, K):
    x = synth.with_outliers(synth.normal((M, K), 0, f"bt.x{M}x{K}"), 0, f"bt.o{M}x{K}")
    w = synth.weights(kind, N, K, 0, f"bt.{kind}.{N}x{K}")
    p = _plane(x)
    g = Guarded((M, N), torch.float32)
    mq.gemv(kind, p, w.cuda(), N, g.t)
    torch.cuda.synchronize()
    g.check()
    assert g.untouched() == 0, "unwritten outputs"
    _check(g.t, p, w, kind, N, K)


@pytest.mark.parametrize("kind", KINDS)
def test_rows_match_one_row_calls(kind):
    M, N, K = 6, 500, 2048
    x = synth.normal((M, K), 0, "bt.rows")
    w = synth.weights(kind, N, K, 0, f"bt.rows.{kind}").cuda()
    p = _plane(x)
    out = torch.empty((M, N), device="cuda")
    mq.gemv(kind, p, w, N, out)
    for m in range(M):
        om = torch.empty(N, device="cuda")
        mq.gemv(kind, mq.Plane(p.qs[m:m + 1], p.d[m:m + 1], p.s[m:m + 1]), w, N, om)
        assert torch.equal(om, out[m]), f"row {m}"


def _f16(v):
    return np.frombuffer(np.float16(v).tobytes(), np.uint8)


def _unit_activations(rng, M, K):
    """Integer activations with a 127 in every 32-block, so d_a = 1 and q_a = x."""
    x = rng.integers(-8, 9, size=(M, K)).astype(np.float32)
    for b in range(K // 32):
        x[np.arange(M), 32 * b + rng.integers(0, 32, size=M)] = 127.0
    return torch.from_numpy(x)


def _exact_weights(kind, rng, N, K):
    if kind == "q5k":
        S = K // 256
        blk = np.zeros((N, S, 176), np.uint8)
        blk[..., 0:2], blk[..., 2:4] = _f16(1.0), _f16(1.0)
        sc = rng.integers(0, 2, size=(N, S, 8))
        mn = rng.integers(0, 8, size=(N, S, 8))
        blk[..., 4:8] = sc[..., :4]
        blk[..., 8:12] = mn[..., :4]
        blk[..., 12:16] = sc[..., 4:] | (mn[..., 4:] << 4)
        blk[..., 16:176] = rng.integers(0, 256, size=(N, S, 160), dtype=np.uint8)
        return blk.reshape(N, -1)
    nb = K // 32
    if kind == "q4_0":
        blk = rng.integers(0, 256, size=(N, nb, 18), dtype=np.uint8)
        blk[..., 0:2] = _f16(1.0)
        return blk.reshape(N, -1)
    blk = rng.integers(0, 256, size=(N, nb, 20), dtype=np.uint8)
    blk[..., 0:2] = _f16(1.0)
    blk[..., 2:4] = _f16(-3.0)
    return blk.reshape(N, -1)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("M", [1, 4])
def test_exact_integer_dots(kind, M):
    """Unit weight scales (q5_K: d = dmin = 1, scales 0/1, mins 0..7; q4_0: d = 1; q4_1: d = 1,
    m = -3) and d_a = 1: every product and partial sum is an integer below 2^24, so the GEMV
    equals the f64 oracle bit for bit."""
    rng = np.random.default_rng(17 + M)
    N, K = 300, 1280
    w = torch.from_numpy(np.ascontiguousarray(_exact_weights(kind, rng, N, K))).cuda()
    p = _plane(_unit_activations(rng, M, K))
    assert np.all(p.d.cpu().numpy() == 1.0)
    out = torch.empty((M, N), device="cuda")
    mq.gemv(kind, p, w, N, out)
    ref, _ = O.gemm_rows(p.qs.cpu().numpy(), p.d.cpu().numpy(), w.cpu().numpy(), kind, N, K)
    assert np.all(np.abs(ref) < 2 ** 22)
    got = out.cpu().numpy().astype(np.float64)
    assert np.array_equal(got, ref), f"max diff {np.max(np.abs(got - ref))}"


@pytest.mark.parametrize("kind,N,K", [("q5k", 13824, 5120), ("q4_0", 5120, 5120), ("q4_1", 1024, 13824)])
def test_full_size_every_element(kind, N, K):
    """14B decode shapes at M = 1, every output checked."""
    x = synth.normal((1, K), 0, f"bt.full{K}", device="cuda")
    w = synth.weights(kind, N, K, 0, f"bt.full.{kind}", device="cuda")
    p = mq.Plane.empty(1, K, op=False)
    mq.mq_quantize_q8(x, p)
    g = Guarded((1, N), torch.float32)
    mq.gemv(kind, p, w, N, g.t)
    torch.cuda.synchronize()
    g.check()
    _check(g.t, p, w, kind, N, K)
    assert mq.mq_device_status() == mq.MQ_OK


# ----------------------------------------------------------------- q4_0 / q4_1 prefill GEMM

GEMM_KINDS = ["q4_0", "q4_1"]


def _op_plane(x):
    M, K = x.shape
    p = mq.Plane.empty(M, K)
    mq.mq_quantize_q8(x.cuda(), p)
    return p


@pytest.mark.parametrize("kind", GEMM_KINDS)
@pytest.mark.parametrize("M,N,K", [(16, 256, 512), (2, 1000, 3584), (130, 300, 768), (257, 129, 1280), (1, 8, 256)])
def test_gemm_parity_every_element(kind, M, N, K):
    x = synth.with_outliers(synth.normal((M, K), 0, f"bg.x{M}x{K}"), 0, f"bg.o{M}x{K}")
    w = synth.weights(kind, N, K, 0, f"bg.{kind}.{N}x{K}")
    p = _op_plane(x)
    g = Guarded((M, N), torch.float32)
    mq.gemm(kind, p, mq.gemm_weights(kind, w.cuda(), N, K), N, g.t)
    torch.cuda.synchronize()
    g.check()
    assert g.untouched() == 0, "unwritten outputs"
    _check(g.t, p, w, kind, N, K)
    assert mq.mq_device_status() == mq.MQ_OK


@pytest.mark.parametrize("kind", GEMM_KINDS)
@pytest.mark.parametrize("M", [16, 130])
def test_gemm_exact_integer_dots(kind, M):
    """d = 1 (q4_1: m = -3) and d_a = 1: every partial sum is an integer below 2^24, so the
    GEMM's two exact weight parts and the min term must give the f64 oracle bit for bit."""
    rng = np.random.default_rng(23 + M)
    N, K = 300, 1280
    w = torch.from_numpy(np.ascontiguousarray(_exact_weights(kind, rng, N, K))).cuda()
    p = _op_plane(_unit_activations(rng, M, K))
    assert np.all(p.d.cpu().numpy() == 1.0)
    out = torch.empty((M, N), device="cuda")
    mq.gemm(kind, p, w, N, out)
    ref, _ = O.gemm_rows(p.qs.cpu().numpy(), p.d.cpu().numpy(), w.cpu().numpy(), kind, N, K)
    assert np.all(np.abs(ref) < 2 ** 22)
    got = out.cpu().numpy().astype(np.float64)
    assert np.array_equal(got, ref), f"max diff {np.max(np.abs(got - ref))}"


@pytest.mark.parametrize("kind", GEMM_KINDS)
def test_gemm_full_size_sampled_rows(kind):
    """The 7B FFN up shape at M = 3314, every output written, 16 sampled rows against the oracle."""
    M, N, K = 3314, 18944, 3584
    x = synth.normal((M, K), 0, "bg.full.x", device="cuda")
    w = synth.weights(kind, N, K, 0, f"bg.full.{kind}", device="cuda")
    p = mq.Plane.empty(M, K)
    mq.mq_quantize_q8(x, p)
    g = Guarded((M, N), torch.float32)
    mq.gemm(kind, p, w, N, g.t)
    torch.cuda.synchronize()
    g.check()
    assert g.untouched() == 0, "unwritten outputs"
    rows = np.sort(np.random.default_rng(3).choice(M, 16, replace=False))
    rows[-1] = M - 1
    ref, bound = O.gemm_rows(p.qs.cpu().numpy(), p.d.cpu().numpy(), w.cpu().numpy(), kind, N, K, rows=rows)
    got = g.t.cpu().numpy().astype(np.float64)[rows]
    assert np.all(np.abs(got - ref) <= bound)
    assert mq.mq_device_status() == mq.MQ_OK
