"""Pins of the oracle's GEMM activation operand form (operand_form, reading R20).

The form is checked against values worked out by hand (the power-of-two choice,
a tie in the binary16 rounding, the hi/lo split of a block sum) and against the
properties that make it a faithful operand: the scaled values are the
dequantized activations to within 2^-11, the block sums are exact.
"""
import numpy as np
import pytest

from oracle import mq_oracle as O


def _plane(d_blocks, q):
    """A one-row plane of K = 256 from 8 block scales and 256 quants."""
    return np.asarray(q, np.int8).reshape(1, 256), np.asarray(d_blocks, np.float32).reshape(1, 8)


@pytest.mark.parametrize("D,e", [
    (1.0, 2),            # 1 = 0.5 * 2^1 -> e = 3 - 1; 1 * 2^2 = 4
    (4.0, 0),            # 4 = 0.5 * 2^3 -> e = 0
    (7.99, 0),           # 7.99 = 0.99875 * 2^3 -> e = 0
    (8.0, -1),           # 8 = 0.5 * 2^4 -> e = -1; 8 / 2 = 4
    (0.001, 12),         # 0.001 = 0.512 * 2^-9 -> e = 12; 0.001 * 4096 = 4.096
    (1e-40, 126),        # subnormal f32: E = -132, e = 135 clamped to 126
    (2e36, -118),        # 2e36 = 0.752 * 2^121 -> e = -118
])
def test_exponent_hand_values(D, e):
    d = [D] + [D / 2] * 7
    qs, dd = _plane(d, np.ones(256))
    _, _, af = O.operand_form(qs, dd)
    assert af[0, 0] == np.float32(2.0 ** -e)


def test_unit_scales_give_exact_quadrupled_quants():
    """d = 1 everywhere: e = 2, so ah = 4q exactly and af = 1/4. Block 0 holds 31 quants
    of 127 and one of 126 (sum 4063): sigma = 16252, whose binary16 neighbours are 16248
    and 16256 (ulp 8 in [8192, 16384)); 16252 is the midpoint, and the tie goes to the
    even significand 16256 / 8 = 2032, so hi = 16256 and lo = -4."""
    q = np.zeros(256, np.int64)
    q[:32] = 127
    q[31] = 126
    q[32:64] = -5
    q[64:96] = np.arange(-16, 16)
    qs, d = _plane([1.0] * 8, q)
    ah, ax, af = O.operand_form(qs, d)
    assert np.array_equal(ah[0].astype(np.float64), 4.0 * q)
    assert af[0, 0] == np.float32(0.25)
    assert float(ax[0, 0, 0]) == 16256.0 and float(ax[0, 0, 8]) == -4.0
    assert float(ax[0, 0, 1]) == -640.0 and float(ax[0, 0, 9]) == 0.0
    assert float(ax[0, 0, 2]) == -64.0 and float(ax[0, 0, 10]) == 0.0
    assert np.all(ax[0, 0, 3:8] == 0) and np.all(ax[0, 0, 11:] == 0)


def test_binary16_rounding_ties_to_even():
    """d = 1 + 2^-11 (exact in f32), e = 2. q = 1: 4 + 2^-9 lies halfway between 4 and
    4 + 2^-8 (binary16 ulp at 4 is 2^-8): ties to even give 4. q = 3: f32(3 d) = 3 + 3*2^-11
    exactly, times 4 is 12 + 3*2^-9, 0.75 ulp (2^-7 at 12) above 12: rounds up to 12 + 2^-7."""
    d = np.float32(1.0 + 2.0 ** -11)
    q = np.zeros(256, np.int64)
    q[0], q[1], q[2] = 1, 3, -1
    qs, dd = _plane([d] * 8, q)
    ah, _, _ = O.operand_form(qs, dd)
    assert float(ah[0, 0]) == 4.0
    assert float(ah[0, 1]) == 12.0 + 2.0 ** -7
    assert float(ah[0, 2]) == -4.0


def test_zero_super_block():
    qs = np.zeros((2, 512), np.int8)
    d = np.zeros((2, 16), np.float32)
    d[1, 8:] = 0.5
    qs[1, 256:] = 3
    ah, ax, af = O.operand_form(qs, d)
    assert np.all(ah[0] == 0) and np.all(ax[0] == 0) and np.all(af[:, 0] == 1.0)
    assert np.all(ah[1, :256] == 0) and af[0, 1] == 1.0
    # second super-block of row 1: D = 0.5 = 0.5 * 2^0 -> e = 3, ah = 8 * 0.5 * 3 = 12
    assert np.all(ah[1, 256:].astype(np.float32) == 12.0) and af[1, 1] == np.float32(1 / 8)


def test_scaled_values_within_binary16_rounding_of_the_dequantized_plane():
    rng = np.random.default_rng(31)
    x = (rng.standard_normal((6, 1024)) * np.exp(rng.uniform(-20, 20, (6, 1)))).astype(np.float32)
    x[2] *= np.where(rng.random(1024) < 0.01, 50.0, 1.0).astype(np.float32)
    qs, d, s = O.quantize_q8(x)
    ah, ax, af = O.operand_form(qs, d)
    a = O.dequant_plane(qs, d).reshape(6, 4, 256)
    got = ah.astype(np.float64).reshape(6, 4, 256) * af.T.astype(np.float64)[..., None]
    big = np.abs(a) * af.T[..., None] ** -1 >= 2.0 ** -14        # binary16 normal range after scaling
    err = np.abs(got - a)
    assert np.all(err[big] <= 2.0 ** -11 * np.abs(a[big]))
    assert np.max(np.abs(ah.astype(np.float32))) < 1016.0
    sig = ah.astype(np.float64).reshape(6, 4, 8, 32).sum(-1)
    hl = ax[..., :8].astype(np.float64) + ax[..., 8:].astype(np.float64)
    assert np.all(np.abs(hl - sig) <= 2.0 ** -22 * np.abs(sig) + 2.0 ** -25)
    # the block sums are those of the scaled activations: d * s up to the rounding of ah
    ds = (d.astype(np.float64) * s).reshape(6, 4, 8) / af.T[..., None]
    assert np.all(np.abs(sig - ds) <= 2.0 ** -11 * np.abs(a).reshape(6, 4, 8, 32).sum(-1) / af.T[..., None] + 1e-30)
