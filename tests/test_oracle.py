"""Pins for the CPU oracle: closed forms, hand-built blocks, invariants, brute force.

Each test checks the oracle against something other than itself, chosen so that
a plausible slip (a dropped term, a wrong sign, index or byte offset, the wrong
rounding mode) fails at least one of them.
"""
import json
import math
import os

from fractions import Fraction

import numpy as np
import pytest

from oracle import mq_oracle as O
from quant_int8_quantized_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------- f16

def test_f16_decode_matches_numpy_for_every_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32)
    ours = O.f16_bits_to_f64(bits)
    ref = bits.astype(np.uint16).view(np.float16).astype(np.float64)
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.all(both_nan | (ours == ref))


# ----------------------------------------------------------------------------- q4_K layout

def pack_q4k_scales(sc, mn):
    """Independent packer for the 12-byte q4_K scale field (inverse of the unpack).

    Bytes 0..3: scale of sub-block j in bits 0..5, bits 4..5 of scale j+4 in bits 6..7.
    Bytes 4..7: min of sub-block j in bits 0..5, bits 4..5 of min j+4 in bits 6..7.
    Bytes 8..11: low 4 bits of scale j+4 in bits 0..3, low 4 bits of min j+4 in bits 4..7.
    """
    out = [0] * 12
    for j in range(4):
        out[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        out[j + 4] = (mn[j] & 63) | ((mn[j + 4] >> 4) << 6)
        out[j + 8] = (sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4)
    return out


def test_q4k_scale_field_hand_example():
    # bytes chosen by hand; expected values worked out by hand from the field description
    packed = np.array([0xC1, 0x02, 0x43, 0x84, 0x05, 0xC6, 0x07, 0x48, 0x9A, 0x0B, 0xFC, 0x3D], np.uint8)
    sc, mn = O.q4k_scales_mins(packed)
    # sub-blocks 0..3: low 6 bits of bytes 0..3 / 4..7
    assert list(sc[:4]) == [0x01, 0x02, 0x03, 0x04]
    assert list(mn[:4]) == [0x05, 0x06, 0x07, 0x08]
    # sub-block 4: scale = (0x9A & 15) | (0xC1 >> 6) << 4 = 10 | 48 = 58; min = (0x9A >> 4) | (0x05 >> 6) << 4 = 9
    # sub-block 5: scale = 0xB | (0x02>>6)<<4 = 11; min = 0 | (0xC6>>6)<<4 = 48
    # sub-block 6: scale = 0xC | (0x43>>6)<<4 = 12 | 16 = 28; min = 0xF | (0x07>>6)<<4 = 15
    # sub-block 7: scale = 0xD | (0x84>>6)<<4 = 13 | 32 = 45; min = 0x3 | (0x48>>6)<<4 = 3 | 16 = 19
    assert list(sc[4:]) == [58, 11, 28, 45]
    assert list(mn[4:]) == [9, 48, 15, 19]


def test_q4k_scale_field_roundtrip_random():
    rng = np.random.default_rng(1)
    for _ in range(200):
        sc = rng.integers(0, 64, 8)
        mn = rng.integers(0, 64, 8)
        got_sc, got_mn = O.q4k_scales_mins(np.array(pack_q4k_scales(sc, mn), np.uint8))
        assert list(got_sc) == list(sc) and list(got_mn) == list(mn)


def _q4k_block(d=1.0, dmin=0.0, sc=None, mn=None, qs=None):
    b = np.zeros(144, np.uint8)
    b[0:2] = np.frombuffer(np.float16(d).tobytes(), np.uint8)
    b[2:4] = np.frombuffer(np.float16(dmin).tobytes(), np.uint8)
    sc = [1] * 8 if sc is None else sc
    mn = [0] * 8 if mn is None else mn
    b[4:16] = pack_q4k_scales(sc, mn)
    if qs is not None:
        b[16:144] = qs
    return b


@pytest.mark.parametrize("byte,high,element", [
    (0, 0, 0), (0, 1, 32), (1, 0, 1), (31, 1, 63), (32, 0, 64), (63, 1, 127),
    (64, 0, 128), (100, 0, 196), (100, 1, 228), (127, 1, 255)])
def test_q4k_nibble_positions_one_hot(byte, high, element):
    qs = np.zeros(128, np.uint8)
    qs[byte] = 0x70 if high else 0x07
    w = O.dequant_q4k(_q4k_block(qs=qs), 1, 256)[0]
    expect = np.zeros(256)
    expect[element] = 7.0
    assert np.array_equal(w, expect)


def test_q4k_scales_and_mins_per_sub_block():
    qs = np.full(128, 0x11, np.uint8)                 # every quant = 1
    w = O.dequant_q4k(_q4k_block(d=1.0, sc=[1, 2, 3, 4, 5, 6, 7, 63], qs=qs), 1, 256)[0]
    assert w[0] == 1 and w[31] == 1 and w[32] == 2 and w[100] == 4 and w[224] == 63 and w[255] == 63
    # d = 0: only the min term remains, -dmin * m[j]
    w = O.dequant_q4k(_q4k_block(d=0.0, dmin=0.5, sc=[0] * 8, mn=[0, 1, 2, 3, 4, 5, 6, 40], qs=qs), 1, 256)[0]
    assert w[0] == 0 and w[32] == -0.5 and w[64 + 5] == -1.0 and w[255] == -20.0


def test_q4k_superblocks_and_rows_are_independent():
    b0 = _q4k_block(d=2.0, qs=np.full(128, 0x11, np.uint8))
    b1 = _q4k_block(d=-1.0, dmin=1.0, mn=[1] * 8, qs=np.full(128, 0x22, np.uint8))
    w = O.dequant_q4k(np.concatenate([b0, b1, b1, b0]).reshape(2, 288), 2, 512)
    assert np.all(w[0, :256] == 2.0) and np.all(w[0, 256:] == -3.0)
    assert np.all(w[1, :256] == -3.0) and np.all(w[1, 256:] == 2.0)


# ----------------------------------------------------------------------------- q6_K layout

def _q6k_block(d=1.0, scales=None, ql=None, qh=None):
    b = np.zeros(210, np.uint8)
    if ql is not None:
        b[0:128] = ql
    if qh is not None:
        b[128:192] = qh
    sc = np.ones(16, np.int8) if scales is None else np.asarray(scales, np.int8)
    b[192:208] = sc.view(np.uint8)
    b[208:210] = np.frombuffer(np.float16(d).tobytes(), np.uint8)
    return b


@pytest.mark.parametrize("byte,high,element", [
    (0, 0, 0), (0, 1, 64), (5, 0, 5), (32, 0, 32), (32, 1, 96), (63, 1, 127),
    (64, 0, 128), (96, 0, 160), (100, 1, 228), (127, 1, 255)])
def test_q6k_low_nibble_positions_one_hot(byte, high, element):
    ql = np.zeros(128, np.uint8)
    ql[byte] = 0x50 if high else 0x05
    w = O.dequant_q6k(_q6k_block(ql=ql), 1, 256)[0]
    expect = np.full(256, -32.0)
    expect[element] = 5 - 32
    assert np.array_equal(w, expect)


@pytest.mark.parametrize("byte,shift,element", [
    (0, 0, 0), (0, 2, 32), (0, 4, 64), (0, 6, 96), (7, 4, 71), (31, 6, 127),
    (32, 0, 128), (40, 2, 168), (63, 6, 255)])
def test_q6k_high_pair_positions_one_hot(byte, shift, element):
    qh = np.zeros(64, np.uint8)
    qh[byte] = 3 << shift
    w = O.dequant_q6k(_q6k_block(qh=qh), 1, 256)[0]
    expect = np.full(256, -32.0)
    expect[element] = 48 - 32
    assert np.array_equal(w, expect)


def test_q6k_int8_scales_per_16():
    scales = np.arange(1, 17, dtype=np.int8)
    scales[5] = -3
    scales[15] = -128
    ql = np.full(128, 0x11, np.uint8)        # low 4 bits = 1
    qh = np.full(64, 0xAA, np.uint8)         # high 2 bits = 2 everywhere -> q = 33
    w = O.dequant_q6k(_q6k_block(d=0.5, scales=scales, ql=ql, qh=qh), 1, 256)[0]
    assert w[0] == 0.5 and w[15] == 0.5 and w[16] == 1.0 and w[80] == -1.5 and w[95] == -1.5
    assert w[240] == -64.0 and w[255] == -64.0
    # q = 32 gives zero whatever the scale
    w = O.dequant_q6k(_q6k_block(d=3.0, scales=scales, qh=np.full(64, 0xAA, np.uint8)), 1, 256)[0]
    assert np.all(w == 0.0)


def test_q6k_size_reproduces_pages_bandwidth():
    g = json.load(open(os.path.join(GOLDEN, "page_numbers.json")))["attn_v_q6k_decode"]
    nbytes = g["od"] * (g["id"] // O.QK_K) * O.Q6K_BYTES
    gbps = nbytes / (g["kernel_us"] * 1e-6) / 1e9
    assert abs(gbps - g["approx_GBps"]) < 1.0
    assert g["id"] // O.QK == json.load(open(os.path.join(GOLDEN, "page_numbers.json")))["decode_units"]["units_per_row"]


def test_swiglu_traffic_arithmetic():
    g = json.load(open(os.path.join(GOLDEN, "page_numbers.json")))["swiglu_traffic"]
    mb = g["ffn"] * g["tokens"] * 4 / 1e6
    assert abs(mb - g["f32_MB"]) < 0.1 and abs(2 * mb - g["saved_MB_per_layer"]) < 0.2


# ----------------------------------------------------------------------------- q8 quantization

def test_quantize_hand_block_ties_to_even():
    v = np.zeros(32, np.float32)
    v[:8] = [127.0, 2.5, 3.5, -2.5, 0.5, 1.5, -0.49, 126.6]
    qs, d, s = O.quantize_q8(v[None, :])
    assert d[0, 0] == np.float32(1.0)                   # amax 127 -> d = 1 exactly
    assert list(qs[0, :8]) == [127, 2, 4, -2, 0, 2, 0, 127]
    assert s[0, 0] == 127 + 2 + 4 - 2 + 0 + 2 + 0 + 127


def test_quantize_divides_rather_than_multiplies_by_the_reciprocal():
    """R4: q = rint(v / d) with the IEEE f32 quotient. The block holds 31 values next to
    rounding boundaries (n + 1/2) * d where v * f32(1/d) rounds to another integer; the
    expected quants come from the exact rational v / d, correctly rounded to f32 by exact
    comparison, then rounded half to even."""
    f32 = np.float32
    amax = f32(1.7)
    d = f32(amax / f32(127))
    inv = f32(f32(1) / d)

    def exact_quotient_f32(v):
        t = Fraction(float(v)) / Fraction(float(d))
        c = f32(float(t))
        cands = [np.nextafter(c, f32(-np.inf)), c, np.nextafter(c, f32(np.inf))]
        return min(cands, key=lambda z: (abs(Fraction(float(z)) - t), int(f32(z).view(np.uint32)) & 1))

    vals = []
    for n in range(126):
        c = f32((n + 0.5) * float(d))
        for k in range(-40, 41):
            v = c
            for _ in range(abs(k)):
                v = np.nextafter(v, f32(np.inf) if k > 0 else f32(-np.inf))
            if np.rint(exact_quotient_f32(v)) != np.rint(f32(v * inv)):
                vals.append(v)
                break
        if len(vals) == 31:
            break
    assert len(vals) == 31
    block = np.array([amax] + vals, np.float32)[None, :]
    qs, dd, ss = O.quantize_q8(block)
    assert dd[0, 0] == d
    expect = np.array([127] + [int(np.rint(exact_quotient_f32(v))) for v in vals])
    reciprocal = np.array([127] + [int(np.rint(f32(v * inv))) for v in vals])
    assert np.array_equal(qs[0].astype(int), expect)
    assert not np.any(expect[1:] == reciprocal[1:])   # every value tells the two rules apart
    assert ss[0, 0] == expect.sum()


def test_quantize_zero_and_single_value_blocks():
    v = np.zeros((1, 64), np.float32)
    v[0, 40] = -0.3
    qs, d, s = O.quantize_q8(v)
    assert d[0, 0] == 0 and np.all(qs[0, :32] == 0) and s[0, 0] == 0
    assert d[0, 1] == np.float32(np.float32(0.3) / np.float32(127))
    assert qs[0, 40] == -127 and s[0, 1] == -127 and np.count_nonzero(qs) == 1


def test_quantize_matches_brute_force_and_bounds():
    rng = np.random.default_rng(7)
    v = (rng.standard_normal((9, 256)) * np.exp(rng.uniform(-8, 8, (9, 1)))).astype(np.float32)
    v[3, 5] = 0.0
    qs, d, s = O.quantize_q8(v)
    for m in range(9):
        for b in range(8):
            blk = [float(t) for t in v[m, 32 * b:32 * b + 32]]
            amax = max(abs(t) for t in blk)
            db = float(np.float32(np.float64(amax) / 127.0))    # f64 divide then f32 round = IEEE f32 divide
            assert d[m, b] == np.float32(db)
            tot = 0
            for i, t in enumerate(blk):
                quot = float(np.float32(t / db))
                q = int(round(quot))                            # Python rounds ties to even
                q = max(-127, min(127, q))
                assert qs[m, 32 * b + i] == q
                tot += q
                assert abs(t - db * q) <= db * (0.5 + 2.0 ** -20) + 1e-45
            assert s[m, b] == tot
            am = int(np.argmax(np.abs(v[m, 32 * b:32 * b + 32])))
            assert abs(int(qs[m, 32 * b + am])) == 127


# ----------------------------------------------------------------------------- fused producers

def test_rms_scale_constant_rows_closed_form():
    K = 512
    x = np.full((2, K), 0.5, np.float32)
    x[1] = -4.0
    scale = O.rms_scale(x, 1e-6)
    assert scale[0] == np.float32(1.0) / np.sqrt(np.float32(0.25) + np.float32(1e-6))
    assert scale[1] == np.float32(1.0) / np.sqrt(np.float32(16.0) + np.float32(1e-6))
    qs, d, s = O.rms_quant(x, np.ones(K, np.float32), 1e-6)
    assert np.all(qs[0] == 127) and np.all(qs[1] == -127) and np.all(s[0] == 127 * 32)


def test_rms_sum_of_squares_within_summation_bound():
    rng = np.random.default_rng(3)
    K = 3584
    x = rng.standard_normal((5, K)).astype(np.float32)
    scale = O.rms_scale(x, 0.0).astype(np.float64)
    for m in range(5):
        exact = math.fsum(float(t) * float(t) for t in x[m])
        ss_from_scale = K / scale[m] ** 2
        assert abs(ss_from_scale - exact) <= exact * (K / 128 + 16) * 2.0 ** -23


def test_rms_values_close_to_f64_definition():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((4, 1024)).astype(np.float32)
    w = (1 + 0.1 * rng.standard_normal(1024)).astype(np.float32)
    v = O.rms_values(x, w, 1e-6).astype(np.float64)
    x64 = x.astype(np.float64)
    ref = x64 / np.sqrt((x64 ** 2).mean(1, keepdims=True) + 1e-6) * w
    assert np.max(np.abs(v - ref) / np.maximum(np.abs(ref), 1e-30)) < 2e-6


def test_rms_other_order_agrees_within_one_level():
    """A plain serial f64 order moves the scale by ulps: planes agree within +-1 level."""
    rng = np.random.default_rng(5)
    K = 3584
    x = rng.standard_normal((16, K)).astype(np.float32)
    w = (1 + 0.1 * rng.standard_normal(K)).astype(np.float32)
    qs, d, _ = O.rms_quant(x, w, 1e-6)
    x64 = x.astype(np.float64)
    scale = (1.0 / np.sqrt((x64 ** 2).sum(1) / K + 1e-6)).astype(np.float32)
    v = ((x * scale[:, None]) * w[None, :]).astype(np.float32)
    qs2, d2, _ = O.quantize_q8(v)
    assert np.max(np.abs(qs.astype(int) - qs2.astype(int))) <= 1
    assert np.max(np.abs(d - d2) / d) <= 2.0 ** -21


def test_exp_f32_within_1_ulp_of_f64_exp():
    """R10's exp against the f64 exp on a dense grid of its whole range: a dropped Taylor
    term, a wrong reduction constant or a wrong 2^n scaling each cost far more than 1 ulp."""
    x = np.linspace(-86.0, 88.0, 400_001).astype(np.float32)
    e = O.exp_f32(x).astype(np.float64)
    t = np.exp(x.astype(np.float64))
    ulp = np.spacing(t.astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(e - t) / ulp) <= 1.0


def _round_f32(t):
    """Correct (ties-to-even) rounding of an exact rational to f32, by comparing the
    three f32 values around float(t) exactly."""
    c = np.float32(float(t))
    cands = [np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))]
    return min(cands, key=lambda v: (abs(Fraction(float(v)) - t), int(np.float32(v).view(np.uint32)) & 1))


def test_fma_f32_is_correctly_rounded():
    rng = np.random.default_rng(11)
    n = 3000
    a = (rng.standard_normal(n) * np.exp2(rng.integers(-20, 20, n))).astype(np.float32)
    b = (rng.standard_normal(n) * np.exp2(rng.integers(-20, 20, n))).astype(np.float32)
    c = (rng.standard_normal(n) * np.exp2(rng.integers(-40, 40, n))).astype(np.float32)
    got = O.fma_f32(a, b, c)
    for i in range(n):
        exact = Fraction(float(a[i])) * Fraction(float(b[i])) + Fraction(float(c[i]))
        assert got[i] == _round_f32(exact), (a[i], b[i], c[i])
    # a*b = 1 + 2^-11 + 2^-24 sits on an f32 midpoint: alone it rounds to even; a tiny c
    # that f64 loses must still push it up (a plain f64 sum then f32 rounding would not)
    a1 = np.float32(1 + 2.0 ** -12)
    assert O.fma_f32(a1, a1, np.float32(0.0)) == np.float32(1 + 2.0 ** -11)
    assert O.fma_f32(a1, a1, np.float32(2.0 ** -60)) == np.float32(1 + 2.0 ** -11 + 2.0 ** -23)
    assert np.float32(float(a1) * float(a1) + 2.0 ** -60) == np.float32(1 + 2.0 ** -11)


def test_exp_f32_special_cases():
    assert O.exp_f32(np.float32(0.0)) == np.float32(1.0)
    # at x = f32(k ln 2) the reduction gives n = k and r ~ 0: e^x is 2^k times e^r
    k = np.arange(-120, 127)
    xf = (k * np.log(2.0)).astype(np.float32)
    e = O.exp_f32(xf).astype(np.float64)
    r = xf.astype(np.float64) - k * np.log(2.0)
    assert np.all(np.abs(e / (np.exp2(k.astype(np.float64)) * np.exp(r)) - 1.0) < 2.0 ** -22)
    assert np.all(O.exp_f32(np.array([-86.5, -1e30], np.float32)) == 0.0)
    assert np.all(np.isinf(O.exp_f32(np.array([88.5, 1e30], np.float32))))
    # the Taylor coefficients are 1/k! correctly rounded to f32: e^r on tiny r is 1 + r
    r = np.float32(2.0 ** -20)
    assert O.exp_f32(r) == np.float32(1.0) + r


def test_swiglu_values_close_to_f64_definition():
    rng = np.random.default_rng(6)
    g = (rng.standard_normal((3, 512)) * 4).astype(np.float32)
    g[0, :4] = [0.0, 30.0, -30.0, -100.0]
    u = rng.standard_normal((3, 512)).astype(np.float32)
    v = O.swiglu_values(g, u).astype(np.float64)
    g64, u64 = g.astype(np.float64), u.astype(np.float64)
    ref = g64 / (1 + np.exp(-g64)) * u64
    assert v[0, 0] == 0.0 and abs(v[0, 1] - 30.0 * u64[0, 1]) <= abs(u64[0, 1]) * 30 * 1e-6
    assert np.all(np.abs(v - ref) <= 1e-6 * np.abs(ref) + 1e-37)


# ----------------------------------------------------------------------------- matmul

def test_gemm_closed_form_all_ones():
    K = 512
    w = np.concatenate([_q4k_block(d=1.0, qs=np.full(128, 0x11, np.uint8))] * 2)[None, :]
    w = np.repeat(w, 3, axis=0)
    wdeq = O.dequant_q4k(w, 3, K)
    assert np.all(wdeq == 1.0)
    qs, d, s = O.quantize_q8(np.ones((2, K), np.float32))
    out = O.gemm(qs, d, wdeq)
    expect = K * 127 * float(np.float32(1.0) / np.float32(127.0))
    assert np.all(out == expect)


def _integer_factorized_q4k(qs, d, s, w, N, K):
    dd, dmin, sc, mn, q = O.q4k_fields(w, N, K)
    M = qs.shape[0]
    S = K // 256
    out = np.zeros((M, N))
    qa = qs.astype(np.int64).reshape(M, S, 8, 32)
    qw = q.reshape(N, S, 8, 32)
    for m in range(M):
        for n in range(N):
            tot = 0.0
            for sb in range(S):
                for j in range(8):
                    I = int(np.dot(qa[m, sb, j], qw[n, sb, j]))
                    da = float(d[m, sb * 8 + j])
                    tot += da * (dd[n, sb] * sc[n, sb, j] * I - dmin[n, sb] * mn[n, sb, j] * int(s[m, sb * 8 + j]))
            out[m, n] = tot
    return out


def _integer_factorized_q6k(qs, d, w, N, K):
    dd, sc, q = O.q6k_fields(w, N, K)
    M = qs.shape[0]
    S = K // 256
    out = np.zeros((M, N))
    qa = qs.astype(np.int64).reshape(M, S, 8, 2, 16)
    qw = (q - 32).reshape(N, S, 8, 2, 16)
    for m in range(M):
        for n in range(N):
            tot = 0.0
            for sb in range(S):
                for j in range(8):
                    lo = int(np.dot(qa[m, sb, j, 0], qw[n, sb, j, 0]))
                    hi = int(np.dot(qa[m, sb, j, 1], qw[n, sb, j, 1]))
                    tot += float(d[m, sb * 8 + j]) * dd[n, sb] * (sc[n, sb, 2 * j] * lo + sc[n, sb, 2 * j + 1] * hi)
            out[m, n] = tot
    return out


def test_gemm_integer_identity_q4k():
    rng = np.random.default_rng(11)
    M, N, K = 3, 4, 512
    w = rng.integers(0, 256, (N, K // 256 * 144), dtype=np.uint8)
    for n in range(N):
        for sb in range(K // 256):
            w[n, sb * 144:sb * 144 + 4] = np.frombuffer(np.abs(rng.standard_normal(2) * 0.01).astype(np.float16).tobytes(), np.uint8)
    qs, d, s = O.quantize_q8(rng.standard_normal((M, K)).astype(np.float32))
    ref = _integer_factorized_q4k(qs, d, s, w, N, K)
    out = O.gemm(qs, d, O.dequant_q4k(w, N, K))
    assert np.max(np.abs(out - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_gemm_integer_identity_q6k():
    rng = np.random.default_rng(12)
    M, N, K = 3, 4, 512
    w = rng.integers(0, 256, (N, K // 256 * 210), dtype=np.uint8)
    for n in range(N):
        for sb in range(K // 256):
            w[n, sb * 210 + 208:sb * 210 + 210] = np.frombuffer(np.float16(abs(rng.standard_normal()) * 0.01).tobytes(), np.uint8)
    qs, d, s = O.quantize_q8(rng.standard_normal((M, K)).astype(np.float32))
    ref = _integer_factorized_q6k(qs, d, w, N, K)
    out = O.gemm(qs, d, O.dequant_q6k(w, N, K))
    assert np.max(np.abs(out - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_gemm_within_quantization_bound_of_f32_product():
    rng = np.random.default_rng(13)
    M, N, K = 4, 6, 768
    x = rng.standard_normal((M, K)).astype(np.float32)
    w = synth.q4k_weights(N, K, 0, "bound").numpy()
    wdeq = O.dequant_q4k(w, N, K)
    qs, d, s = O.quantize_q8(x)
    out = O.gemm(qs, d, wdeq)
    exact = x.astype(np.float64) @ wdeq.T
    half_step = np.repeat(d.astype(np.float64), 32, axis=1) / 2 * (1 + 2.0 ** -20)
    bound = half_step @ np.abs(wdeq).T
    assert np.all(np.abs(out - exact) <= bound)


def test_gemm_rows_subset_matches_full():
    rng = np.random.default_rng(14)
    M, N, K = 5, 7, 512
    w = synth.q6k_weights(N, K, 0, "subset").numpy()
    qs, d, s = O.quantize_q8(rng.standard_normal((M, K)).astype(np.float32))
    full = O.gemm(qs, d, O.dequant_q6k(w, N, K))
    sub, bound = O.gemm_rows(qs, d, w, "q6k", N, K, rows=[1, 4], cols=[0, 6, 3])
    ref = full[[1, 4]][:, [0, 6, 3]]
    assert np.allclose(sub, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    assert np.all(bound >= 0)
