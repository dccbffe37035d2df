"""Parity of the prefill GEMM and decode GEMV (CUDA, through the C ABI) with the
CPU oracle: every output element within 1e-3 * sum_k |a||w| of the f64
reference, on seeded inputs whose sizes span several tiles and a ragged tail,
plus full-size shapes checked on sampled rows."""
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


def _plane_from(x):
    M, K = x.shape
    p = mq.Plane.empty(M, K)
    mq.mq_quantize_q8(x.cuda(), p)
    return p


def _check(out, plane, w, kind, N, K, rows=None, slack=0.0):
    qs, d = plane.qs.cpu().numpy(), plane.d.cpu().numpy()
    ref, bound = O.gemm_rows(qs, d, w.cpu().numpy(), kind, N, K, rows=rows)
    got = out.cpu().numpy().astype(np.float64)
    if rows is not None:
        got = got[rows]
    err = np.abs(got - ref)
    worst = np.max(err / np.maximum(bound, 1e-30))
    assert np.all(err <= bound + slack), f"{kind}: max err/bound = {worst:.3g}"
    return worst


def _run(kind, x, N, K, fn, outliers_name=None):
    w = synth.weights(kind, N, K, 0, f"{kind}.{N}x{K}")
    p = _plane_from(x)
    g = Guarded((x.shape[0], N), torch.float32)
    wd = w.cuda()
    if fn is mq.gemm:
        wd = mq.gemm_weights(kind, wd, N, K)
    fn(kind, p, wd, N, g.t)
    torch.cuda.synchronize()
    g.check()
    return g.t, p, w


# ----------------------------------------------------------------- GEMM

GEMM_SHAPES = [
    (16, 256, 512),      # the tiny single matmul: 16 rows x 256 outputs x 512
    (1, 8, 256),
    (5, 100, 768),       # odd super-block count (q6_K rows only 2-byte aligned)
    (130, 300, 512),     # ragged in M and N, several tiles
    (257, 129, 1280),
]


@pytest.mark.parametrize("kind", ["q4k", "q6k"])
@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_gemm_parity(kind, M, N, K):
    x = synth.normal((M, K), 0, f"gx{M}x{K}")
    out, p, w = _run(kind, x, N, K, mq.gemm)
    _check(out, p, w, kind, N, K)


@pytest.mark.parametrize("kind", ["q4k", "q6k"])
def test_gemm_outlier_activations(kind):
    M, N, K = 64, 192, 1024
    x = synth.with_outliers(synth.normal((M, K), 0, "ox"), 0, "ox")
    out, p, w = _run(kind, x, N, K, mq.gemm)
    _check(out, p, w, kind, N, K)


@pytest.mark.parametrize("kind", ["q4k", "q6k"])
@pytest.mark.parametrize("M,N,K", [(1100, 2176, 2048), (300, 8320, 1280)])
def test_gemm_partial_last_wave_every_element(kind, M, N, K):
    """153 tiles (one full wave of 152 SMs + 1) and 195 tiles (+ 43): the q6_K kernel splits the
    last wave's tiles along K into the zeroed tile columns, q4_K runs them whole. Every output
    element is checked."""
    x = synth.normal((M, K), 0, f"lw{M}x{K}")
    out, p, w = _run(kind, x, N, K, mq.gemm)
    _check(out, p, w, kind, N, K)


@pytest.mark.parametrize("kind", ["q4k", "q6k"])
@pytest.mark.parametrize("M", [2, 3, 8, 15, 24, 40, 64, 65])
def test_gemm_small_batch_every_element(kind, M):
    """Small batches: one token tile of round_up(M, 16) (MMA N = 16 for M in [2, 16)), the weight
    rows split along K across the SMs; q4_K tiles of up to 64 tokens take the short-tile form
    (M = 65 is the first full-form tile). Every element of a ragged, several-tile product
    within the bound."""
    N, K = 1000, 3584
    x = synth.with_outliers(synth.normal((M, K), 0, f"sbx{M}"), 0, f"sbo{M}")
    out, p, w = _run(kind, x, N, K, mq.gemm)
    _check(out, p, w, kind, N, K)


@pytest.mark.parametrize("kind,N,K", [("q4k", 18944, 3584), ("q6k", 3584, 18944)])
def test_gemm_small_batch_full_size(kind, N, K):
    """M = 15 on the 7B FFN shapes, every element checked."""
    M = 15
    x = synth.normal((M, K), 0, f"sbf{K}", device="cuda")
    w = synth.weights(kind, N, K, 0, f"sbfw{kind}{N}", device="cuda")
    p = mq.Plane.empty(M, K)
    mq.mq_quantize_q8(x, p)
    g = Guarded((M, N), torch.float32)
    mq.gemm(kind, p, mq.gemm_weights(kind, w, N, K), N, g.t)
    torch.cuda.synchronize()
    g.check()
    assert g.untouched() == 0, "unwritten outputs"
    _check(g.t, p, w, kind, N, K)
    assert mq.mq_device_status() == mq.MQ_OK


@pytest.mark.parametrize("kind,N,K", [("q4k", 18944, 3584), ("q6k", 3584, 18944), ("q4k", 512, 3584)])
def test_gemm_full_size_sampled_rows(kind, N, K):
    """7B prefill shapes at M = 3314, oracle on 24 sampled rows (rows are independent); every
    output element checked as written (the q6_K shape splits its last round along K)."""
    M = 3314
    x = synth.normal((M, K), 0, f"fx{K}", device="cuda")
    w = synth.weights(kind, N, K, 0, f"fw{kind}{N}", device="cuda")
    p = mq.Plane.empty(M, K)
    mq.mq_quantize_q8(x, p)
    g = Guarded((M, N), torch.float32)
    mq.gemm(kind, p, mq.gemm_weights(kind, w, N, K), N, g.t)
    torch.cuda.synchronize()
    g.check()
    assert g.untouched() == 0, "unwritten outputs"
    rows = np.sort(np.random.default_rng(1).choice(M, 24, replace=False))
    rows[-1] = M - 1
    _check(g.t, p, w, kind, N, K, rows=rows)
    assert mq.mq_device_status() == mq.MQ_OK


@pytest.mark.parametrize("kind,M,N,K", [("q6k", 3314, 3584, 18944), ("q6k", 1000, 3456, 8192),
                                         ("q6k", 2000, 2560, 16384), ("q6k", 3314, 3584, 3584),
                                         ("q4k", 3314, 3584, 3584)])
def test_gemm_ordered_split_of_the_last_round(kind, M, N, K):
    """q6_K tile counts that leave the persistent grid's last round partly idle (504, 162 and
    220 tiles on 152 SMs) with enough super-blocks a row for a split to pay (74, 32, 64): those
    tiles run in a second launch as 2 to 4 K slices that add into the output in a fixed order
    (q6_K with 14 super-blocks a row, which does not split, and q4_K as controls). Sampled rows
    against the oracle, half of them in the last 400 tokens (where those tiles lie), every
    element written, the same bits on a second call and on three replays of a captured graph,
    and no bounded wait given up."""
    x = synth.normal((M, K), 0, f"ox{M}x{K}", device="cuda")
    w = synth.weights(kind, N, K, 0, f"ow{kind}{N}x{K}", device="cuda")
    wg = mq.gemm_weights(kind, w, N, K)
    p = mq.Plane.empty(M, K)
    mq.mq_quantize_q8(x, p)
    g = Guarded((M, N), torch.float32)
    mq.gemm(kind, p, wg, N, g.t)
    torch.cuda.synchronize()
    g.check()
    assert g.untouched() == 0, "unwritten outputs"
    first = g.t.clone()
    rng = np.random.default_rng(M + N)
    rows = np.unique(np.r_[rng.choice(M - 400, 12, replace=False), rng.choice(np.arange(M - 400, M), 12, replace=False),
                           M - 1])
    _check(g.t, p, w, kind, N, K, rows=rows)
    out = torch.empty((M, N), device="cuda")
    mq.gemm(kind, p, wg, N, out)
    torch.cuda.synchronize()
    assert torch.equal(out, first), "a second call gave other bits"
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        mq.gemm(kind, p, wg, N, out)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        mq.gemm(kind, p, wg, N, out)
    for _ in range(3):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, first), "a graph replay gave other bits"
    assert mq.mq_device_status() == mq.MQ_OK


@pytest.mark.parametrize("M,N0,N1,K", [(3314, 3584, 512, 3584), (3314, 18944, 18944, 3584), (1000, 2560, 1280, 1024),
                                        (400, 2560, 640, 1024)])
def test_gemm_q4k_pair(M, N0, N1, K):
    """Two q4_K GEMMs on one plane (attn_q | attn_k and ffn_gate | ffn_up at 3314 tokens, a small
    pair, and one too small to share a launch): each output within the oracle bound on sampled
    rows (half of them in the last 400 tokens) and bit-identical to mq_gemm_q4k's where that call
    does not split along K, every element written, the same bits on a second call."""
    x = synth.normal((M, K), 0, f"px{M}x{K}", device="cuda")
    w0 = synth.weights("q4k", N0, K, 0, f"pw0{N0}x{K}", device="cuda")
    w1 = synth.weights("q4k", N1, K, 0, f"pw1{N1}x{K}", device="cuda")
    p = mq.Plane.empty(M, K)
    mq.mq_quantize_q8(x, p)
    g0, g1 = Guarded((M, N0), torch.float32), Guarded((M, N1), torch.float32)
    mq.mq_gemm_q4k_pair(p, w0, N0, g0.t, w1, N1, g1.t)
    torch.cuda.synchronize()
    g0.check()
    g1.check()
    assert g0.untouched() == 0 and g1.untouched() == 0, "unwritten outputs"
    rng = np.random.default_rng(M + N0 + N1)
    tail = np.arange(max(0, M - 400), M)
    rows = np.unique(np.r_[rng.choice(M, 10, replace=False), rng.choice(tail, 10, replace=False), M - 1])
    for g, w, N in ((g0, w0, N0), (g1, w1, N1)):
        _check(g.t, p, w, "q4k", N, K, rows=rows)
        single = torch.empty((M, N), device="cuda")
        mq.mq_gemm_q4k(p, w, N, single)
        torch.cuda.synchronize()
        bt = 192 if M >= 192 else (M + 15) // 16 * 16
        tiles = -(-M // bt) * -(-N // 128)
        if tiles >= torch.cuda.get_device_properties(0).multi_processor_count:   # mq_gemm_q4k does not split
            assert torch.equal(single, g.t), f"N = {N}: other bits than mq_gemm_q4k"
    o0, o1 = torch.empty((M, N0), device="cuda"), torch.empty((M, N1), device="cuda")
    mq.mq_gemm_q4k_pair(p, w0, N0, o0, w1, N1, o1)
    torch.cuda.synchronize()
    assert torch.equal(o0, g0.t) and torch.equal(o1, g1.t), "a second call gave other bits"
    assert mq.mq_device_status() == mq.MQ_OK


# ----------------------------------------------------------------- GEMV

GEMV_SHAPES = [(256, 512), (1024, 5120), (100, 768), (5120, 13824), (1, 256), (7001, 3584), (3, 1280)]


@pytest.mark.parametrize("kind", ["q4k", "q6k"])
@pytest.mark.parametrize("M", [2, 3, 5, 8])
def test_gemv_small_batch_every_element(kind, M):
    """The GEMV with M activation rows (each weight super-block decoded once, dotted with every
    row): every element within the bound, and each row bit-identical to a one-row call on it
    (the per-row summation order does not depend on M)."""
    N, K = 1000, 3584
    x = synth.with_outliers(synth.normal((M, K), 0, f"vbx{M}"), 0, f"vbo{M}")
    out, p, w = _run(kind, x, N, K, mq.gemv)
    _check(out, p, w, kind, N, K)
    wd = w.cuda()
    for m in range(M):
        pm = mq.Plane(p.qs[m:m + 1], p.d[m:m + 1], p.s[m:m + 1])
        om = torch.empty(N, device="cuda")
        mq.gemv(kind, pm, wd, N, om)
        assert torch.equal(om, out[m]), f"row {m}"


@pytest.mark.parametrize("kind,N,K", [("q4k", 13824, 5120), ("q6k", 5120, 13824)])
def test_gemv_small_batch_full_size(kind, N, K):
    """M = 8 (the largest GEMV batch) on the 14B FFN shapes, every element checked."""
    M = 8
    x = synth.normal((M, K), 0, f"vbf{K}", device="cuda")
    w = synth.weights(kind, N, K, 0, f"vbfw{kind}{N}", device="cuda")
    p = mq.Plane.empty(M, K, op=False)
    mq.mq_quantize_q8(x, p)
    g = Guarded((M, N), torch.float32)
    mq.gemv(kind, p, w, N, g.t)
    torch.cuda.synchronize()
    g.check()
    assert g.untouched() == 0, "unwritten outputs"
    _check(g.t, p, w, kind, N, K)


@pytest.mark.parametrize("kind", ["q4k", "q6k"])
@pytest.mark.parametrize("N,K", GEMV_SHAPES)
def test_gemv_parity(kind, N, K):
    x = synth.normal((1, K), 0, f"vx{K}")
    out, p, w = _run(kind, x, N, K, mq.gemv)
    _check(out, p, w, kind, N, K)


@pytest.mark.parametrize("kind,N,K", [("q6k", 152064, 3584), ("q4k", 27648, 5120), ("q6k", 5120, 13824),
                                      ("q6k", 2048, 5120)])
def test_gemv_full_size_sampled_outputs(kind, N, K):
    """The bench's decode and lm_head GEMVs at full size (lm_head 152064 x 3584, gate|up and k|v
    stacked, down); outputs are independent rows, so the oracle checks 512 sampled ones, always
    the first and the last."""
    x = synth.normal((1, K), 0, f"fv{K}", device="cuda")
    w = synth.weights(kind, N, K, 0, f"fvw{kind}{N}", device="cuda")
    p = mq.Plane.empty(1, K, op=False)
    mq.mq_quantize_q8(x, p)
    g = Guarded((1, N), torch.float32)
    mq.gemv(kind, p, w, N, g.t)
    torch.cuda.synchronize()
    g.check()
    assert g.untouched() == 0, "unwritten outputs"
    rows = np.unique(np.r_[np.random.default_rng(N).choice(N, 512, replace=False), 0, N - 1])
    rt = torch.as_tensor(rows, device="cuda")
    ref, bound = O.gemm_rows(p.qs.cpu().numpy(), p.d.cpu().numpy(), w[rt].cpu().numpy(), kind, len(rows), K)
    got = g.t[0, rt].cpu().numpy().astype(np.float64)[None, :]
    assert np.all(np.abs(got - ref) <= bound)
    assert mq.mq_device_status() == mq.MQ_OK


@pytest.mark.parametrize("N,K", [(33, 1280), (64, 2048), (9, 2304), (17, 8448)])
def test_gemv_q6k_exact_integer_dots(N, K):
    """Unit super-block scales, sub-block scales of +-1 and integer activations whose every
    32-block holds a 127 (so d_a = 1 and q_a = x): every output is an exact integer below
    2^24, so the GPU must equal the f64 oracle bit for bit. Quants cover 0..63 uniformly."""
    rng = np.random.default_rng(K + N)
    S = K // 256
    blk = rng.integers(0, 256, size=(N, S, 210), dtype=np.uint8)
    blk[:, :, 192:208] = rng.choice(np.array([-1, 1], np.int8), size=(N, S, 16)).view(np.uint8)
    blk[:, :, 208:210] = np.frombuffer(np.float16(1.0).tobytes(), np.uint8)
    w = torch.from_numpy(np.ascontiguousarray(blk.reshape(N, S * 210))).cuda()
    xi = rng.integers(-127, 128, size=(1, K)).astype(np.float32)
    xi[0, rng.integers(0, 32) :: 32] = 127.0
    p = _plane_from(torch.from_numpy(xi))
    assert np.all(p.d.cpu().numpy() == 1.0)
    g = Guarded((1, N), torch.float32)
    mq.gemv("q6k", p, w, N, g.t)
    torch.cuda.synchronize()
    g.check()
    ref, _ = O.gemm_rows(p.qs.cpu().numpy(), p.d.cpu().numpy(), w.cpu().numpy(), "q6k", N, K)
    assert np.all(np.abs(ref) < 2 ** 24)
    assert np.array_equal(g.t.cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("kind", ["q4k", "q6k"])
def test_gemv_matches_gemm_at_one_row(kind):
    N, K = 384, 1536
    x = synth.normal((1, K), 0, "one")
    w = synth.weights(kind, N, K, 0, "one.w").cuda()
    p = _plane_from(x)
    a = torch.empty((1, N), device="cuda")
    b = torch.empty((1, N), device="cuda")
    mq.gemv(kind, p, w, N, a)
    mq.gemm(kind, p, mq.gemm_weights(kind, w, N, K), N, b)
    torch.cuda.synchronize()
    ref, bound = O.gemm_rows(p.qs.cpu().numpy(), p.d.cpu().numpy(), w.cpu().numpy(), kind, N, K)
    assert np.all(np.abs(a.cpu().numpy() - b.cpu().numpy()) <= 2 * bound)


def test_gemv_rejects_more_rows_than_it_takes():
    M = mq.MQ_GEMV_MAX_ROWS + 1
    p = mq.Plane.empty(M, 256)
    w = torch.zeros((8, 144), dtype=torch.uint8, device="cuda")
    out = torch.empty((M, 8), device="cuda")
    with pytest.raises(mq.MQError) as e:
        mq.mq_gemv_q4k(p, w, 8, out)
    assert e.value.status == mq.MQ_ERR_SHAPE


@pytest.mark.parametrize("N,K", [(1, 256), (7, 768), (300, 512), (64, 18944)])
def test_prepack_q6k_is_the_documented_layout(N, K):
    """Half h of each packed 224-byte block: raw ql[64h..], qh[32h..], scales[8h..], d, 6 zeros.
    The expected bytes are assembled here from the raw block, field by field."""
    S = K // 256
    raw = np.random.default_rng(N + K).integers(0, 256, size=(N, S, 210), dtype=np.uint8)
    want = np.zeros((N, S, 224), np.uint8)
    for h in range(2):
        o = 112 * h
        want[..., o:o + 64] = raw[..., 64 * h:64 * h + 64]
        want[..., o + 64:o + 96] = raw[..., 128 + 32 * h:128 + 32 * h + 32]
        want[..., o + 96:o + 104] = raw[..., 192 + 8 * h:192 + 8 * h + 8]
        want[..., o + 104:o + 106] = raw[..., 208:210]
    w = torch.from_numpy(np.ascontiguousarray(raw.reshape(N, S * 210))).cuda()
    g = Guarded((N, S * 224), torch.uint8)
    mq.mq_prepack_q6k(w, N, K, g.t)
    torch.cuda.synchronize()
    g.check()
    assert np.array_equal(g.t.cpu().numpy().reshape(N, S, 224), want)


def _unit_activations(rng, M, K, small_first_half=False):
    """Integer activations whose every 32-block holds a 127, so d_a = 1 and q_a = x. With
    small_first_half, elements 0..15 of each block lie in [-1, 1] and the 127 sits in 16..31."""
    x = rng.integers(-8, 9, size=(M, K)).astype(np.float32)
    for b in range(K // 32):
        if small_first_half:
            x[:, 32 * b:32 * b + 16] = rng.integers(-1, 2, size=(M, 16))
            x[np.arange(M), 32 * b + 16 + rng.integers(0, 16, size=M)] = 127.0
        else:
            x[np.arange(M), 32 * b + rng.integers(0, 32, size=M)] = 127.0
    return torch.from_numpy(x)


@pytest.mark.parametrize("d,dmin", [(1.0, 1.0), (1.0, 4.0), (1.0, 3.0), (0.5, 3.0), (2.0, 0.5)])
@pytest.mark.parametrize("M,N,K", [(16, 256, 512), (130, 200, 768), (300, 1100, 1280), (3, 300, 768), (8, 200, 1280),
                                   (48, 300, 768)])
def test_gemm_q4k_exact_integer_dots(M, N, K, d, dmin):
    """Super-block scales d, dmin chosen so that the kernel's power of two k (the least k >= 0
    with d 2^k >= dmin: 0, 2, 2, 3, 0 here) and its operands are exact: sub-block scales 0 or
    1, mins 0..7, d_a = 1, so ah = 4q, the weight operand sc q 2^-k and dmin / (d 2^k) are exact
    binary16 values and every partial sum is a multiple of 2^-3 far below 2^21. The GEMM (short
    tiles for M <= 64, full tiles above) must then equal the f64 oracle bit for bit."""
    rng = np.random.default_rng(M + N + K)
    S = K // 256
    blk = np.zeros((N, S, 144), np.uint8)
    blk[..., 0:2] = np.frombuffer(np.float16(d).tobytes(), np.uint8)
    blk[..., 2:4] = np.frombuffer(np.float16(dmin).tobytes(), np.uint8)
    sc = rng.integers(0, 2, size=(N, S, 8))
    mn = rng.integers(0, 8, size=(N, S, 8))
    # 6-bit fields < 16: bytes 0..3 scales 0..3, 4..7 mins 0..3, 8..11 scale | min << 4 of 4..7
    blk[..., 4:8] = sc[..., :4]
    blk[..., 8:12] = mn[..., :4]
    blk[..., 12:16] = sc[..., 4:] | (mn[..., 4:] << 4)
    blk[..., 16:144] = rng.integers(0, 256, size=(N, S, 128), dtype=np.uint8)
    w = torch.from_numpy(np.ascontiguousarray(blk.reshape(N, S * 144))).cuda()
    p = _plane_from(_unit_activations(rng, M, K))
    assert np.all(p.d.cpu().numpy() == 1.0)
    g = Guarded((M, N), torch.float32)
    mq.mq_gemm_q4k(p, w, N, g.t)
    torch.cuda.synchronize()
    g.check()
    ref, _ = O.gemm_rows(p.qs.cpu().numpy(), p.d.cpu().numpy(), w.cpu().numpy(), "q4k", N, K)
    assert np.all(np.abs(ref) < 2 ** 22)
    got = g.t.cpu().numpy().astype(np.float64)
    assert np.array_equal(got, ref), f"max diff {np.max(np.abs(got - ref))}"


@pytest.mark.parametrize("M,N,K", [(16, 256, 256), (130, 200, 768), (64, 300, 1280), (2, 300, 768), (15, 200, 1280)])
def test_gemm_q6k_exact_integer_dots(M, N, K):
    """d = 1, sub-block scales +-1, and in sub-blocks 2j (the first half of each 32-block, where
    the activations lie in [-1, 1]) also scale -128 with high bits 0, so the operand's two exact
    parts reach 2432 and 4096. With d_a = 1 every partial sum is an integer below 2^24 and the
    GEMM must equal the f64 oracle bit for bit."""
    rng = np.random.default_rng(M + N + K + 1)
    S = K // 256
    blk = rng.integers(0, 256, size=(N, S, 210), dtype=np.uint8)
    scales = rng.choice(np.array([-1, 1], np.int8), size=(N, S, 16))
    big = rng.random((N, S, 8)) < 0.5                      # sub-block 2j gets -128 with hi = 0
    scales[..., 0::2] = np.where(big, np.int8(-128), scales[..., 0::2])
    blk[..., 192:208] = scales.view(np.uint8)
    blk[..., 208:210] = np.frombuffer(np.float16(1.0).tobytes(), np.uint8)
    # hi = 0 for every element of a "big" sub-block: element e = 128h + 32t + l of sub-block
    # g = e // 16 takes its high bits from qh[32h + l] bits 2t, 2t + 1
    qh = blk[..., 128:192].copy()
    for e in range(256):
        g = e // 16
        if g % 2:
            continue
        h, r = divmod(e, 128)
        t, l = divmod(r, 32)
        mask = np.uint8(~(3 << (2 * t)) & 0xFF)
        qh[..., 32 * h + l] = np.where(big[..., g // 2], qh[..., 32 * h + l] & mask, qh[..., 32 * h + l])
    blk[..., 128:192] = qh
    w = torch.from_numpy(np.ascontiguousarray(blk.reshape(N, S * 210))).cuda()
    p = _plane_from(_unit_activations(rng, M, K, small_first_half=True))
    assert np.all(p.d.cpu().numpy() == 1.0)
    g = Guarded((M, N), torch.float32)
    mq.mq_gemm_q6k(p, mq.mq_prepack_q6k(w, N, K), N, g.t)
    torch.cuda.synchronize()
    g.check()
    ref, _ = O.gemm_rows(p.qs.cpu().numpy(), p.d.cpu().numpy(), w.cpu().numpy(), "q6k", N, K)
    wd = O.dequant_q6k(w.cpu().numpy(), N, K)
    assert np.max(np.abs(wd)) >= 2176               # the scale -128 with hi = 0 is exercised
    assert np.all(np.abs(ref) < 2 ** 22)
    got = g.t.cpu().numpy().astype(np.float64)
    assert np.array_equal(got, ref), f"max diff {np.max(np.abs(got - ref))}"
