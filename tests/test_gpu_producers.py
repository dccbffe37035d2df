"""Parity of the q8 plane producers (CUDA, through the C ABI) with the CPU oracle.

All three producers (quantize, fused RMSNorm, fused SwiGLU with its pinned exp)
must be bit-exact: the q8 arrays against the oracle's plane, and the GEMM
operand arrays (ah, ax, af) against the oracle's operand form of it.
Every output buffer starts poisoned (0xCD) inside guard bands, so an unwritten
slot or an out-of-bounds write fails the test.
"""
import numpy as np
import pytest
import torch

from oracle import mq_oracle as O
from quant_int8_quantized_gb300 import mq, synth
from tests._gpu_util import GuardedPlane, assert_operand_form, assert_plane_equal, require_gpu

pytestmark = pytest.mark.gpu

SHAPES = [(1, 256), (3, 512), (16, 512), (130, 768), (257, 3584), (5, 18944)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _x(M, K, name, outliers=False):
    x = synth.normal((M, K), 0, name)
    if outliers:
        x = synth.with_outliers(x, 0, name)
    return x


@pytest.mark.parametrize("M,K", SHAPES)
@pytest.mark.parametrize("outliers", [False, True])
def test_quantize_bit_exact(M, K, outliers):
    x = _x(M, K, f"q{M}x{K}", outliers)
    x[0, :32] = 0.0                     # an all-zero block
    if K >= 64:
        x[-1, 32:64] = 0.0
        x[-1, 40] = -3.0                # a single non-zero value
    gp = GuardedPlane(M, K)
    mq.mq_quantize_q8(x.cuda(), gp.plane)
    torch.cuda.synchronize()
    gp.check()
    assert_plane_equal(gp.numpy(), O.quantize_q8(x.numpy()), f"quantize {M}x{K}")


def _boundary_blocks(seed=7):
    """32-blocks whose element 0 is the block's amax and whose other elements sit on
    and a few ulps around (n + 1/2) * d, d = amax / 127 rounded to f32: the
    quotients v / d straddle the rounding boundaries of q = rint(v / d)."""
    rng = np.random.default_rng(seed)
    blocks = []
    for am in [127.0, 100.0, 3.0, 0.0123, 1e-3, 2.5e-36, 5e-39]:
        am = np.float32(am)
        d = np.float32(am / np.float32(127.0))
        vals = []
        for n in rng.integers(-126, 126, size=40):
            t = np.float32(np.float32(n + 0.5) * d)
            for k in (-3, -1, 0, 1, 3):
                v = t
                for _ in range(abs(k)):
                    v = np.nextafter(v, np.float32(np.inf if k > 0 else -np.inf), dtype=np.float32)
                vals.append(v)
        vals = np.array(vals, dtype=np.float32)
        vals = vals[np.abs(vals) < am]
        for i in range(0, len(vals) - 30, 31):
            blocks.append(np.concatenate([[am], vals[i:i + 31]]).astype(np.float32))
    blocks = np.stack(blocks)
    pad = (-len(blocks)) % 8
    if pad:
        blocks = np.concatenate([blocks, blocks[:pad]])
    return blocks.reshape(-1, 256)


def test_quantize_bit_exact_at_rounding_boundaries():
    x = torch.from_numpy(_boundary_blocks())
    M, K = x.shape
    gp = GuardedPlane(M, K)
    mq.mq_quantize_q8(x.cuda(), gp.plane)
    torch.cuda.synchronize()
    gp.check()
    assert_plane_equal(gp.numpy(), O.quantize_q8(x.numpy()), "quantize at rounding boundaries")


@pytest.mark.parametrize("M,K", SHAPES)
def test_rms_quant_bit_exact(M, K):
    x = _x(M, K, f"r{M}x{K}")
    w = synth.normal((K,), 0, f"rw{K}", mean=1.0, std=0.1)
    gp = GuardedPlane(M, K)
    mq.mq_rms_quant(x.cuda(), w.cuda(), 1e-6, gp.plane)
    torch.cuda.synchronize()
    gp.check()
    assert_plane_equal(gp.numpy(), O.rms_quant(x.numpy(), w.numpy(), 1e-6), f"rms {M}x{K}")


@pytest.mark.parametrize("M", [1, 7, 700])   # the 128-thread-per-row and the warp-per-row kernels
def test_rms_quant_both_launch_shapes(M):
    K = 5120
    x = _x(M, K, f"rr{M}")
    w = synth.normal((K,), 0, "rw5120", mean=1.0, std=0.1)
    gp = GuardedPlane(M, K)
    mq.mq_rms_quant(x.cuda(), w.cuda(), 1e-6, gp.plane)
    torch.cuda.synchronize()
    gp.check()
    assert_plane_equal(gp.numpy(), O.rms_quant(x.numpy(), w.numpy(), 1e-6), f"rms {M}x{K}")


@pytest.mark.parametrize("M,K", [(700, 1280), (640, 4096), (609, 256), (1000, 3584), (608, 10240), (610, 18944)])
def test_rms_quant_many_rows(M, K):
    """Enough rows to fill the machine: two rounds a warp, four for rows over 64 rounds, and
    the twice-reading kernel for rows over 128 rounds; ragged round counts."""
    x = _x(M, K, f"rw{M}x{K}")
    w = synth.normal((K,), 0, f"rww{K}", mean=1.0, std=0.1)
    gp = GuardedPlane(M, K)
    mq.mq_rms_quant(x.cuda(), w.cuda(), 1e-6, gp.plane)
    torch.cuda.synchronize()
    gp.check()
    assert_plane_equal(gp.numpy(), O.rms_quant(x.numpy(), w.numpy(), 1e-6), f"rms {M}x{K}")


def test_rms_quant_equals_quantize_of_oracle_rms_values():
    """Mode-2 identity: the fused plane equals the standalone quantize of the f32 RMSNorm output."""
    M, K = 64, 3584
    x = _x(M, K, "mode2")
    w = synth.normal((K,), 0, "mode2w", mean=1.0, std=0.1)
    fused = GuardedPlane(M, K)
    mq.mq_rms_quant(x.cuda(), w.cuda(), 1e-6, fused.plane)
    v = torch.from_numpy(O.rms_values(x.numpy(), w.numpy(), 1e-6)).cuda()
    sep = GuardedPlane(M, K)
    mq.mq_quantize_q8(v, sep.plane)
    torch.cuda.synchronize()
    assert_plane_equal(fused.numpy(), sep.numpy(), "fused vs separate")


@pytest.mark.parametrize("M,K", SHAPES)
def test_swiglu_quant_bit_exact(M, K):
    g = _x(M, K, f"g{M}x{K}") * 3
    u = _x(M, K, f"u{M}x{K}")
    g[0, :4] = torch.tensor([0.0, 40.0, -40.0, -100.0])
    gp = GuardedPlane(M, K)
    mq.mq_swiglu_quant(g.cuda(), u.cuda(), gp.plane)
    torch.cuda.synchronize()
    gp.check()
    assert_plane_equal(gp.numpy(), O.swiglu_quant(g.numpy(), u.numpy()), f"swiglu {M}x{K}")


def test_swiglu_quant_exp_range_edges():
    """SwiGLU at the edges of its exp's range (e^x is 0 below -86 and +inf above 88, so
    g / (1 + e^-g) is g or -0 there), one ulp either side of each edge, subnormal and huge
    gates (whose products with u stay finite), signed zeros: bit-exact. Each 32-block mixes edge
    values with ordinary ones."""
    f32 = np.float32
    edges = []
    for e in (86.0, 87.0, 88.0):
        for sgn in (1.0, -1.0):
            v = f32(sgn * e)
            edges += [np.nextafter(v, f32(-np.inf), dtype=f32), v, np.nextafter(v, f32(np.inf), dtype=f32)]
    edges += [f32(0.0), f32(-0.0), f32(1e-40), f32(-1e-40), f32(1e30), f32(-1e30), f32(1e37), f32(-1e37),
              f32(0.5), f32(-0.5), f32(20.0), f32(-20.0)]
    edges = np.array(edges, dtype=f32)
    K = 512
    g = np.resize(edges, (2, K)).astype(f32)
    g[1] = np.roll(g[1], 7)
    rng = np.random.default_rng(5)
    g[:, ::3] = rng.normal(0.0, 4.0, size=g[:, ::3].shape).astype(f32)
    u = rng.normal(0.0, 1.0, size=(2, K)).astype(f32)
    u[:, ::5] *= f32(1e-3)
    gp = GuardedPlane(2, K)
    mq.mq_swiglu_quant(torch.from_numpy(g).cuda(), torch.from_numpy(u).cuda(), gp.plane)
    torch.cuda.synchronize()
    gp.check()
    assert_plane_equal(gp.numpy(), O.swiglu_quant(g, u), "swiglu exp-range edges")


def test_producers_full_size_sampled_rows():
    """7B FFN shapes (M = 3314; hidden 3584, ffn 18944) with the oracle on 64 sampled rows."""
    M, K, KF = 3314, 3584, 18944
    rows = np.sort(np.random.default_rng(0).choice(M, 64, replace=False))
    rows[-1] = M - 1
    x = synth.normal((M, K), 0, "full.x", device="cuda")
    w = synth.normal((K,), 0, "full.w", mean=1.0, std=0.1, device="cuda")
    gp, gpf, gpq = GuardedPlane(M, K), GuardedPlane(M, KF), GuardedPlane(M, KF)
    p, pf, pq = gp.plane, gpf.plane, gpq.plane
    mq.mq_rms_quant(x, w, 1e-6, p)
    g = synth.normal((M, KF), 0, "full.g", device="cuda")
    u = synth.normal((M, KF), 0, "full.u", device="cuda")
    mq.mq_swiglu_quant(g, u, pf)
    mq.mq_quantize_q8(g, pq)
    torch.cuda.synchronize()
    for gx in (gp, gpf, gpq):   # every block's d and s written (their poison words are impossible values)
        gx.check()
        assert gx.g["d"].untouched() == 0 and gx.g["s"].untouched() == 0
        assert gx.g["ah"].untouched() == 0 and gx.g["ax"].untouched() == 0
    idx = torch.from_numpy(rows).cuda()
    sub = lambda pl: (pl.qs[idx].cpu().numpy(), pl.d[idx].cpu().numpy(), pl.s[idx].cpu().numpy())
    xs, ws = x[idx].cpu().numpy(), w.cpu().numpy()
    assert_plane_equal(sub(p), O.rms_quant(xs, ws, 1e-6), "rms full")
    assert_plane_equal(sub(pq), O.quantize_q8(g[idx].cpu().numpy()), "quantize full")
    assert_plane_equal(sub(pf), O.swiglu_quant(g[idx].cpu().numpy(), u[idx].cpu().numpy()), "swiglu full")
    for pl, what in ((p, "rms"), (pq, "quantize"), (pf, "swiglu")):
        qs_, d_, _ = sub(pl)
        assert_operand_form(pl, qs_, d_, rows=rows, what=f"{what} full operand form")
        assert not np.any(pl.af[:, :M].cpu().numpy().view(np.uint32) == 0xCDCDCDCD), f"{what}: af unwritten"
    assert mq.mq_device_status() == mq.MQ_OK


@pytest.mark.parametrize("kind", ["quantize", "rms", "swiglu"])
@pytest.mark.parametrize("M,K", [(1, 256), (5, 512), (130, 3584), (333, 18944), (3, 5120)])
def test_operand_only_plane(kind, M, K):
    """A GEMM-only plane (no q8 arrays): the producers write ah, ax, af equal to the oracle's
    operand form of the oracle's plane, and nothing else."""
    x = _x(M, K, f"op{kind}{M}x{K}", outliers=True)
    gp = GuardedPlane(M, K, q8=False)
    if kind == "quantize":
        mq.mq_quantize_q8(x.cuda(), gp.plane)
        ref = O.quantize_q8(x.numpy())
    elif kind == "rms":
        w = synth.normal((K,), 0, f"opw{K}", mean=1.0, std=0.1)
        mq.mq_rms_quant(x.cuda(), w.cuda(), 1e-6, gp.plane)
        ref = O.rms_quant(x.numpy(), w.numpy(), 1e-6)
    else:
        u = _x(M, K, f"opu{M}x{K}")
        mq.mq_swiglu_quant(x.cuda(), u.cuda(), gp.plane)
        ref = O.swiglu_quant(x.numpy(), u.numpy())
    torch.cuda.synchronize()
    gp.check(ref=(ref[0], ref[1]))


def test_misaligned_input_rejected():
    x = torch.zeros(2 * 256 + 1, dtype=torch.float32, device="cuda")[1:].view(2, 256)
    p = mq.Plane.empty(2, 256)
    with pytest.raises(mq.MQError) as e:
        mq.mq_quantize_q8(x, p)
    assert e.value.status == mq.MQ_ERR_ALIGN
