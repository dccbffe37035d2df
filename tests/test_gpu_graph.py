"""The entry points only enqueue work on the caller's stream, so a sequence of
them can be captured into a CUDA graph and replayed. A captured decode layer
(RMSNorm->q8, q4_K and q6_K GEMVs, SwiGLU->q8) and a captured prefill GEMM must
give bit-identical results to the same calls made eagerly, replay after replay,
and the GEMV outputs must stay within the oracle's bound."""
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


def _capture(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def test_decode_layer_graph_replay_matches_eager():
    dev = torch.device("cuda")
    H, F, KV = 1024, 2048, 256
    x = synth.normal((1, H), 5, "g.x", device=dev)
    w_rms = synth.normal((H,), 5, "g.rms", 1.0, 0.1, device=dev)
    g_in = synth.normal((1, F), 5, "g.g", device=dev)
    u_in = synth.normal((1, F), 5, "g.u", device=dev)
    Wq = synth.weights("q4k", H, H, 5, "g.wq", device=dev)
    Wv = synth.weights("q6k", KV, H, 5, "g.wv", device=dev)
    Wd = synth.weights("q6k", H, F, 5, "g.wd", device=dev)
    ph, pf = mq.Plane.empty(1, H, dev, op=False), mq.Plane.empty(1, F, dev, op=False)
    oq = torch.empty((H,), device=dev)
    ov = torch.empty((KV,), device=dev)
    od = torch.empty((H,), device=dev)

    def layer():
        mq.mq_rms_quant(x, w_rms, 1e-6, ph)
        mq.mq_gemv_q4k(ph, Wq, H, oq)
        mq.mq_gemv_q6k(ph, Wv, KV, ov)
        mq.mq_swiglu_quant(g_in, u_in, pf)
        mq.mq_gemv_q6k(pf, Wd, H, od)

    layer()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (oq, ov, od, ph.qs, ph.d, pf.qs, pf.d)]
    graph = _capture(layer)
    for t in (oq, ov, od):
        t.fill_(float("nan"))
    for _ in range(3):
        graph.replay()
        torch.cuda.synchronize()
        for a, b in zip(eager, (oq, ov, od, ph.qs, ph.d, pf.qs, pf.d)):
            assert torch.equal(a, b)
    assert mq.mq_device_status() == mq.MQ_OK
    # and the replayed outputs are right, not only repeatable
    qs, d = ph.qs.cpu().numpy(), ph.d.cpu().numpy()
    ref, bound = O.gemm_rows(qs, d, Wq.cpu().numpy(), "q4k", H, H)
    assert np.all(np.abs(oq.cpu().numpy()[None, :] - ref) <= bound)
    qs, d = pf.qs.cpu().numpy(), pf.d.cpu().numpy()
    ref, bound = O.gemm_rows(qs, d, Wd.cpu().numpy(), "q6k", H, F)
    assert np.all(np.abs(od.cpu().numpy()[None, :] - ref) <= bound)


def test_prefill_gemm_graph_replay_matches_eager():
    dev = torch.device("cuda")
    M, N, K = 200, 384, 1024
    x = synth.normal((M, K), 6, "g.px", device=dev)
    W4 = synth.weights("q4k", N, K, 6, "g.pw4", device=dev)
    W6 = mq.mq_prepack_q6k(synth.weights("q6k", N, K, 6, "g.pw6", device=dev), N, K)
    p = mq.Plane.empty(M, K, dev)
    o4 = torch.empty((M, N), device=dev)
    o6 = torch.empty((M, N), device=dev)

    def step():
        mq.mq_quantize_q8(x, p)
        mq.mq_gemm_q4k(p, W4, N, o4)
        mq.mq_gemm_q6k(p, W6, N, o6)

    step()
    torch.cuda.synchronize()
    e4, e6 = o4.clone(), o6.clone()
    graph = _capture(step)
    o4.zero_()
    o6.zero_()
    for _ in range(2):
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(o4, e4) and torch.equal(o6, e6)
    assert mq.mq_device_status() == mq.MQ_OK


@pytest.mark.parametrize("packed", [False, True])
def test_decode_layer_two_streams_matches_one_stream(packed):
    """The decode step's schedule: the k|v GEMV on a second stream beside attn_q, joined before
    the next producer, captured into a graph. Replays equal one-stream eager execution bit for
    bit, over two layers that reuse the planes; the q6_K k|v GEMV on raw or prepacked rows (the
    bench's decode uses the prepacked form)."""
    dev = torch.device("cuda")
    H, F, KV = 1024, 2048, 256
    x = synth.normal((1, H), 7, "s.x", device=dev)
    attn = synth.normal((1, H), 7, "s.attn", device=dev)
    w_rms = [synth.normal((H,), 7, f"s.rms{l}", 1.0, 0.1, device=dev) for l in range(2)]
    Wq = [synth.weights("q4k", H, H, 7, f"s.wq{l}", device=dev) for l in range(2)]
    Wkv = [synth.weights("q6k", 2 * KV, H, 7, f"s.wkv{l}", device=dev) for l in range(2)]
    if packed:
        Wkv = [mq.mq_prepack_q6k(w, 2 * KV, H) for w in Wkv]
    gemv6 = mq.mq_gemv_q6k_packed if packed else mq.mq_gemv_q6k
    Wo = [synth.weights("q4k", H, H, 7, f"s.wo{l}", device=dev) for l in range(2)]
    ph, pa = mq.Plane.empty(1, H, dev, op=False), mq.Plane.empty(1, H, dev, op=False)
    oq = [torch.empty((H,), device=dev) for _ in range(2)]
    okv = [torch.empty((2 * KV,), device=dev) for _ in range(2)]
    oo = [torch.empty((H,), device=dev) for _ in range(2)]
    side = torch.cuda.Stream()
    ev_h, ev_kv = torch.cuda.Event(), torch.cuda.Event()

    def layer_two_streams():
        main = torch.cuda.current_stream()
        for l in range(2):
            mq.mq_rms_quant(x, w_rms[l], 1e-6, ph)
            ev_h.record(main)
            side.wait_event(ev_h)
            gemv6(ph, Wkv[l], 2 * KV, okv[l], stream=side)
            ev_kv.record(side)
            mq.mq_gemv_q4k(ph, Wq[l], H, oq[l])
            main.wait_event(ev_kv)
            mq.mq_quantize_q8(attn, pa)
            mq.mq_gemv_q4k(pa, Wo[l], H, oo[l])

    def layer_one_stream():
        for l in range(2):
            mq.mq_rms_quant(x, w_rms[l], 1e-6, ph)
            mq.mq_gemv_q4k(ph, Wq[l], H, oq[l])
            gemv6(ph, Wkv[l], 2 * KV, okv[l])
            mq.mq_quantize_q8(attn, pa)
            mq.mq_gemv_q4k(pa, Wo[l], H, oo[l])

    layer_one_stream()
    torch.cuda.synchronize()
    ref = [t.clone() for t in oq + okv + oo]
    graph = _capture(layer_two_streams)
    for t in oq + okv + oo:
        t.fill_(float("nan"))
    for _ in range(3):
        graph.replay()
        torch.cuda.synchronize()
        for a, b in zip(ref, oq + okv + oo):
            assert torch.equal(a, b)
    assert mq.mq_device_status() == mq.MQ_OK
