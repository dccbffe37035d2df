"""Pins of the oracle's evaluation orders and of its tolerance formula.

Three oracle functions decide results bit for bit, or decide what every matmul
parity test accepts, in ways that a bound or a comparison with the f64
definition cannot catch:

  * rms_sumsq: the R8 summation order of RMSNorm's sum of squares;
  * exp_f32: the R10 exp, evaluated step by step with fused multiply-adds;
  * gemm_bound: the R11 tolerance 1e-3 * sum_k |a||w| per output element.

Each is pinned here by values worked out by hand (or in exact rational
arithmetic, rounded to f32 at every step the definition rounds), chosen so that
the plausible slips fail: another summation order, an unfused Horner step, a
wrong tolerance factor or a dropped absolute value.
"""
import math
from fractions import Fraction

import numpy as np

from oracle import mq_oracle as O

U = 2.0 ** -24          # half an ulp of 1.0 in f32


# ----------------------------------------------------------------------------- R8 order

def _crafted_rms_row():
    """K = 384 (three float4 rounds of 32 lanes). Squares, in units of U:
    lane 0, round 0: float4 (3*2^-12, 1, 3*2^-12, 3*2^-12) -> (9U, 1, 9U, 9U);
    lane 0, rounds 1 and 2: 2^-12 -> U each; lane 1, round 0: 9U; lane 17, round 0: U."""
    x = np.zeros((1, 384), np.float32)
    t = 3 * 2.0 ** -12
    x[0, 0:4] = [t, 1.0, t, t]
    x[0, 4 * 32] = 2.0 ** -12
    x[0, 4 * 64] = 2.0 ** -12
    x[0, 4 * 1] = t
    x[0, 4 * 17] = 2.0 ** -12
    return x


def test_rms_sumsq_r8_order_hand_worked():
    """Worked by hand (ulp of numbers in [1, 2) is 2U; every tie goes to the even mantissa):
    lane 0 term ((9U + 1) + 9U) + 9U: 1 + 9U -> 1 + 8U (tie), + 9U -> 1 + 16U (tie),
    + 9U -> 1 + 24U (tie). Lane chain: + U -> 1 + 24U (tie), + U -> 1 + 24U.
    Butterfly at 16: lane 1 becomes 9U + U = 10U; at 8, 4, 2 only zeros join; at 1 lane 0
    takes 1 + 24U + 10U = 1 + 34U (exact). So ss = 1 + 34U.
    Other orders give other sums on this row: a serial pass over the elements in index
    order loses every small square after the 1 (1 + 32U); a pairwise float4 term
    (x0x0 + x1x1) + (x2x2 + x3x3) gives 1 + 26U for lane 0's term and 1 + 38U in the end;
    walking each lane's rounds backwards gives 1 + 36U."""
    ss = O.rms_sumsq(_crafted_rms_row())
    assert ss.dtype == np.float32
    assert float(ss[0]) == 1.0 + 34 * U


def test_rms_sumsq_crafted_row_separates_the_orders():
    """The alternative orders named above really do land elsewhere on the crafted row
    (each written out with scalar f32 adds), so the pin above discriminates them."""
    x = _crafted_rms_row()[0]
    f = np.float32
    sq = [f(v) * f(v) for v in x]
    serial = f(0)
    for s in sq:
        serial = f(serial + s)
    assert float(serial) == 1.0 + 32 * U
    lanes = [f(0)] * 32
    for j in range(3):
        for l in range(32):
            a, b, c, d = sq[4 * (32 * j + l):4 * (32 * j + l) + 4]
            lanes[l] = f(lanes[l] + f(f(a + b) + f(c + d)))
    for off in (16, 8, 4, 2, 1):
        lanes = [f(lanes[l] + lanes[l ^ off]) for l in range(32)]
    assert float(lanes[0]) == 1.0 + 38 * U
    lanes = [f(0)] * 32
    for j in (2, 1, 0):
        for l in range(32):
            a, b, c, d = sq[4 * (32 * j + l):4 * (32 * j + l) + 4]
            lanes[l] = f(lanes[l] + f(f(f(a + b) + c) + d))
    for off in (16, 8, 4, 2, 1):
        lanes = [f(lanes[l] + lanes[l ^ off]) for l in range(32)]
    assert float(lanes[0]) == 1.0 + 36 * U


def test_rms_scale_uses_the_pinned_sum():
    x = _crafted_rms_row()
    ss = np.float32(1.0 + 34 * U)
    expect = np.float32(1.0) / np.sqrt(ss / np.float32(384) + np.float32(1e-6))
    assert O.rms_scale(x, 1e-6)[0] == expect


# ----------------------------------------------------------------------------- R10 exp bits

def _rn32(t: Fraction) -> Fraction:
    """Round an exact rational to the nearest f32 (ties to even), as an exact rational.
    Normal range only (every intermediate of the exp below stays normal)."""
    if t == 0:
        return Fraction(0)
    sign = -1 if t < 0 else 1
    a = abs(t)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = a / Fraction(2) ** (e - 23)          # in [2^23, 2^24)
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * Fraction(n) * Fraction(2) ** (e - 23)


def _exp_exact_steps(x: float, fused: bool = True) -> float:
    """R10 evaluated in exact rational arithmetic, rounding to f32 exactly where the
    definition rounds: n = rint(rn(x * log2e)); r = rn(rn(x - n*ln2_hi) - n*ln2_lo) with
    each line one fused multiply-add; p = 1/7!; p = rn(p*r + 1/k!) for k = 6..0; p * 2^n.
    With fused=False every product is rounded before its add (a plain Horner step)."""
    X = Fraction(float(np.float32(x)))
    log2e = Fraction(float(np.float32(1.0 / math.log(2.0))))
    hi = Fraction(0.693145751953125)
    lo = Fraction(float(np.float32(math.log(2.0) - 0.693145751953125)))
    c = [Fraction(float(np.float32(1.0 / math.factorial(k)))) for k in range(8)]
    t = _rn32(X * log2e)
    n = round(t)                                  # Python rounds ties to even
    step = (lambda a, b, z: _rn32(a * b + z)) if fused else (lambda a, b, z: _rn32(_rn32(a * b) + z))
    r = step(Fraction(-n), hi, X)
    r = step(Fraction(-n), lo, r)
    p = c[7]
    for k in range(6, -1, -1):
        p = step(p, r, c[k])
    return float(p * Fraction(2) ** n)


def test_exp_f32_bits_equal_exact_step_evaluation():
    rng = np.random.default_rng(21)
    xs = np.concatenate([rng.uniform(-86, 88, 300), rng.uniform(-1, 1, 100), [0.5, -0.5, 1.0, 10.0, -20.0]])
    xs = xs.astype(np.float32)
    got = O.exp_f32(xs)
    for x, g in zip(xs, got):
        assert float(g) == _exp_exact_steps(float(x)), x


def test_exp_f32_pin_rejects_an_unfused_horner():
    """On these arguments an evaluation that rounds each product before its add lands on
    other bits at least once, so the bit pin above tells fused and unfused steps apart."""
    rng = np.random.default_rng(22)
    xs = rng.uniform(-20, 20, 300).astype(np.float32)
    differ = sum(_exp_exact_steps(float(x)) != _exp_exact_steps(float(x), fused=False) for x in xs)
    assert differ > 0


# ----------------------------------------------------------------------------- R11 bound

def _q4k_block_bytes(d, dmin, qs):
    """One q4_K super-block with every sub-block scale and min equal to 1."""
    b = np.zeros(144, np.uint8)
    b[0:2] = np.frombuffer(np.float16(d).tobytes(), np.uint8)
    b[2:4] = np.frombuffer(np.float16(dmin).tobytes(), np.uint8)
    b[4:8] = 1          # scales 0..3 = 1 (top bits 0)
    b[8:12] = 1         # mins 0..3 = 1
    b[12:16] = 0x11     # scales and mins 4..7 = 1
    b[16:144] = qs
    return b


def test_gemm_bound_hand_worked_1x1x256():
    """d = 1, dmin = 1/2, every scale and min 1, so w = q - 1/2. The 128 quant bytes are
    0, 17, 34, ..., i.e. byte i holds i mod 16 in both nibbles: each value 0..15 appears 16
    times. a = +1, -1, +1, ... (plane d = 1, q = +-1).
    sum |a||w| = 16 * sum_q |q - 1/2| = 16 * (1/2 + sum_{q=1..15} (q - 1/2)) = 16 * 113 = 1808,
    so the bound is 1e-3 * 1808 = 1.808. A tolerance factor of 1e-2 gives 18.08; w in place
    of |w| gives 16 * 112 * 1e-3 = 1.792; a in place of |a| gives 0."""
    qs_bytes = np.array([(i % 16) * 17 for i in range(128)], np.uint8)
    w = _q4k_block_bytes(1.0, 0.5, qs_bytes)[None, :]
    wdeq = O.dequant_q4k(w, 1, 256)
    assert sorted(set(wdeq[0].tolist())) == [q - 0.5 for q in range(16)]
    qa = np.array([[1 if k % 2 == 0 else -1 for k in range(256)]], np.int8)
    da = np.ones((1, 8), np.float32)
    bound = O.gemm_bound(qa, da, wdeq)
    assert bound.shape == (1, 1)
    assert abs(bound[0, 0] - 1.808) <= 1e-12
    _, b2 = O.gemm_rows(qa, da, w, "q4k", 1, 256)
    assert abs(b2[0, 0] - 1.808) <= 1e-12


def test_gemm_bound_scales_with_activation_scale():
    """The bound follows the dequantized activation d_a * q_a: d_a = 0.25 gives 0.452."""
    qs_bytes = np.array([(i % 16) * 17 for i in range(128)], np.uint8)
    wdeq = O.dequant_q4k(_q4k_block_bytes(1.0, 0.5, qs_bytes)[None, :], 1, 256)
    qa = np.ones((1, 256), np.int8)
    bound = O.gemm_bound(qa, np.full((1, 8), 0.25, np.float32), wdeq)
    assert abs(bound[0, 0] - 0.452) <= 1e-12
