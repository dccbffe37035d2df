"""The shape/token sweep and the one-layer FFN chain, at full size, on the GPU.

Sweep: M in {1, 16, 64, 512, 3314, 8192} x (N, K) in {1024x5120, 3584x3584,
18944x3584, 3584x18944, 13824x5120} x {q4_K, q6_K}; activations f32 N(0, 1)
with each entry scaled by 50 with probability 0.01 (outliers that stress the
per-block amax). M = 1 goes through the decode GEMV, M >= 16 through the GEMM.
Rows are independent, so the oracle checks a seeded sample of rows (always the
first and last) on a seeded sample of output columns (always the last), every
element within 1e-3 * sum_k |a||w|.

FFN chain (one 7B-shaped layer, M = 3314): RMSNorm->q8 plane (bit-exact on
sampled rows), gate and up q4_K GEMMs, SwiGLU->q8 of the GPU's gate and up
outputs (bit-exact), down q6_K GEMM on that plane — each stage checked
against the oracle applied to the GPU's own input of that stage.
"""
import numpy as np
import pytest
import torch

from oracle import mq_oracle as O
from quant_int8_quantized_gb300 import mq, synth
from tests._gpu_util import assert_operand_form, assert_plane_equal, require_gpu

pytestmark = pytest.mark.gpu

SWEEP_M = [1, 16, 64, 512, 3314, 8192]
SWEEP_NK = [(1024, 5120), (3584, 3584), (18944, 3584), (3584, 18944), (13824, 5120)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _sample(n, k, seed, always):
    rng = np.random.default_rng(seed)
    pick = rng.choice(n, min(k, n), replace=False)
    return np.unique(np.concatenate([pick, np.asarray(always, dtype=np.int64)]))


def _check_sampled(out, plane, w, kind, N, K, rows, cols):
    qs = plane.qs[torch.as_tensor(rows, device=plane.qs.device)].cpu().numpy()
    d = plane.d[torch.as_tensor(rows, device=plane.d.device)].cpu().numpy()
    wsub = w[torch.as_tensor(cols, device=w.device)].cpu().numpy()
    ref, bound = O.gemm_rows(qs, d, wsub, kind, len(cols), K)
    got = out[torch.as_tensor(rows, device=out.device)][:, torch.as_tensor(cols, device=out.device)]
    got = got.cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    worst = np.max(err / np.maximum(bound, 1e-30))
    assert np.all(err <= bound), f"{kind} M={plane.M} N={N} K={K}: max err/bound = {worst:.3g}"


@pytest.mark.parametrize("kind", ["q4k", "q6k"])
@pytest.mark.parametrize("N,K", SWEEP_NK)
def test_sweep(kind, N, K):
    dev = torch.device("cuda")
    w = synth.weights(kind, N, K, 0, f"sweep.{kind}.{N}x{K}", device=dev)
    wg = mq.gemm_weights(kind, w, N, K)
    cols = _sample(N, 384, N + K, [N - 1])
    for M in SWEEP_M:
        x = synth.with_outliers(synth.normal((M, K), 0, f"sweep.x.{M}x{K}", device=dev), 0, f"sweep.o.{M}x{K}")
        p = mq.Plane.empty(M, K, dev, op=M > 1)
        mq.mq_quantize_q8(x, p)
        out = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
        if M == 1:
            mq.gemv(kind, p, w, N, out.view(-1))
        else:
            mq.gemm(kind, p, wg, N, out)
        torch.cuda.synchronize()
        assert not torch.isnan(out).any(), f"unwritten outputs at M={M}"
        rows = _sample(M, 8, M * 7 + K, [0, M - 1])
        _check_sampled(out, p, w, kind, N, K, rows, cols)
        del x, p, out
    assert mq.mq_device_status() == mq.MQ_OK


def test_ffn_layer_chain():
    dev = torch.device("cuda")
    M, H, F = 3314, 3584, 18944
    x = synth.normal((M, H), 0, "ffn.x", device=dev)
    w_rms = synth.normal((H,), 0, "ffn.rms", 1.0, 0.1, device=dev)
    Wg = synth.weights("q4k", F, H, 0, "ffn.gate", device=dev)
    Wu = synth.weights("q4k", F, H, 0, "ffn.up", device=dev)
    Wd = synth.weights("q6k", H, F, 0, "ffn.down", device=dev)
    p_h = mq.Plane.empty(M, H, dev)
    mq.mq_rms_quant(x, w_rms, 1e-6, p_h)
    g = torch.empty((M, F), device=dev)
    u = torch.empty((M, F), device=dev)
    mq.mq_gemm_q4k(p_h, Wg, F, g)
    mq.mq_gemm_q4k(p_h, Wu, F, u)
    p_f = mq.Plane.empty(M, F, dev)
    mq.mq_swiglu_quant(g, u, p_f)
    y = torch.empty((M, H), device=dev)
    mq.mq_gemm_q6k(p_f, mq.mq_prepack_q6k(Wd, H, F), H, y)
    torch.cuda.synchronize()
    assert mq.mq_device_status() == mq.MQ_OK

    rows = _sample(M, 12, 99, [0, M - 1])
    rt = torch.as_tensor(rows, device=dev)
    # stage 1: the rms plane, bit-exact
    ref = O.rms_quant(x[rt].cpu().numpy(), w_rms.cpu().numpy(), 1e-6)
    got = (p_h.qs[rt].cpu().numpy(), p_h.d[rt].cpu().numpy(), p_h.s[rt].cpu().numpy())
    assert_plane_equal(got, ref, "ffn rms plane")
    assert_operand_form(p_h, got[0], got[1], rows=rows, what="ffn rms operand form")
    # stage 2: gate and up on the GPU's plane
    cols_f = _sample(F, 256, 5, [F - 1])
    _check_sampled(g, p_h, Wg, "q4k", F, H, rows, cols_f)
    _check_sampled(u, p_h, Wu, "q4k", F, H, rows, cols_f)
    # stage 3: SwiGLU of the GPU's gate and up outputs
    ref = O.swiglu_quant(g[rt].cpu().numpy(), u[rt].cpu().numpy())
    got = (p_f.qs[rt].cpu().numpy(), p_f.d[rt].cpu().numpy(), p_f.s[rt].cpu().numpy())
    assert_plane_equal(got, ref, "ffn swiglu plane")
    # stage 4: down on the GPU's SwiGLU plane
    cols_h = _sample(H, 256, 6, [H - 1])
    _check_sampled(y, p_f, Wd, "q6k", H, F, rows, cols_h)
