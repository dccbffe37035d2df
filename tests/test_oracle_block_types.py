"""Pins of the oracle's q5_K, q4_0 and q4_1 dequantization (readings R21-R23 of the
oracle header) against hand-built blocks whose values are worked out here from the
stated byte order, and against the already-pinned q4_K: a plausible slip (a
transposed qh index, a swapped nibble half, a dropped min or offset) fails one of
them."""
import numpy as np
import pytest

from oracle import mq_oracle as O

pytestmark = pytest.mark.filterwarnings("ignore")


def f16(x):
    return np.frombuffer(np.float16(x).tobytes(), np.uint8)


def unit_scale_field():
    """12-byte q4_K-style field with every 6-bit scale = 1 and every min = 0."""
    f = np.zeros(12, np.uint8)
    f[0:4] = 1          # scales of sub-blocks 0..3 (low 6 bits of bytes 0..3)
    f[8:12] = 1         # scales of sub-blocks 4..7 (low nibbles of bytes 8..11), mins 0
    return f


# ----------------------------------------------------------------- q5_K

def q5k_block(d, dmin, field, qh, qs):
    b = np.zeros(176, np.uint8)
    b[0:2], b[2:4], b[4:16], b[16:48], b[48:176] = f16(d), f16(dmin), field, qh, qs
    return b


def test_q5k_fifth_bits_land_where_the_reading_puts_them():
    # d = 1, unit scales, no mins, all nibbles 0: an element is 16 exactly when its fifth
    # bit is set. qh[5] bit 2 -> group j = 1, low half: element 64 + 5 = 69.
    # qh[7] bit 3 -> group 1, high half: element 64 + 32 + 7 = 103.
    # qh[0] bit 7 -> group 3, high half: element 192 + 32 + 0 = 224.
    # qh[31] bit 0 -> group 0, low half: element 31.
    qh = np.zeros(32, np.uint8)
    qh[5], qh[7], qh[0], qh[31] = 0b100, 0b1000, 0b10000000, 0b1
    w = O.dequant_q5k(q5k_block(1.0, 0.0, unit_scale_field(), qh, np.zeros(128, np.uint8))[None], 1, 256)[0]
    expect = np.zeros(256)
    expect[[69, 103, 224, 31]] = 16.0
    assert np.array_equal(w, expect)


def test_q5k_nibbles_scales_and_mins_by_hand():
    # d = 0.5, dmin = 0.25; sub-block 0 scale 3, min 2; sub-block 1 (high nibbles of the
    # first 32 bytes) scale 1, min 4; others scale 1, min 0.
    field = np.zeros(12, np.uint8)
    field[0:4] = [3, 1, 1, 1]
    field[4:8] = [2, 4, 0, 0]
    field[8:12] = 1
    qs = np.zeros(128, np.uint8)
    qs[0] = 0x9 | (0x2 << 4)       # element 0: 9, element 32: 2
    qh = np.zeros(32, np.uint8)
    qh[0] = 0b11                    # fifth bits of elements 0 and 32
    w = O.dequant_q5k(q5k_block(0.5, 0.25, field, qh, qs)[None], 1, 256)[0]
    assert w[0] == 0.5 * 3 * (9 + 16) - 0.25 * 2            # 36.0
    assert w[32] == 0.5 * 1 * (2 + 16) - 0.25 * 4           # 8.0
    assert w[1] == -0.25 * 2 and w[33] == -0.25 * 4          # q = 0: the min alone
    assert w[64] == 0.0


def test_q5k_without_fifth_bits_is_q4k_of_the_same_fields():
    rng = np.random.default_rng(5)
    N, S = 3, 2
    q4 = rng.integers(0, 256, size=(N, S, 144), dtype=np.uint8)
    q4[..., 0:2] = f16(0.01)
    q4[..., 2:4] = f16(0.003)
    q5 = np.zeros((N, S, 176), np.uint8)
    q5[..., 0:16] = q4[..., 0:16]
    q5[..., 48:176] = q4[..., 16:144]
    a = O.dequant_q5k(q5.reshape(N, -1), N, 256 * S)
    b = O.dequant_q4k(q4.reshape(N, -1), N, 256 * S)
    assert np.array_equal(a, b)
    # all fifth bits set: each element gains exactly 16 * d * sc of its sub-block
    q5[..., 16:48] = 0xFF
    c = O.dequant_q5k(q5.reshape(N, -1), N, 256 * S)
    d, _, sc, _, _ = O.q4k_fields(q4.reshape(N, -1), N, 256 * S)
    gain = (16.0 * d[..., None] * sc[..., np.arange(256) // 32]).reshape(N, -1)
    assert np.array_equal(c - b, gain)


# ----------------------------------------------------------------- q4_0 / q4_1

def test_q4_0_by_hand():
    blk = np.zeros(18, np.uint8)
    blk[0:2] = f16(0.5)
    blk[2:18] = 0x88                 # every element 8 -> 0
    blk[2] = 0x3A                    # element 0: 0xA = 10 -> 0.5 * 2 = 1.0; element 16: 3 -> -2.5
    blk[17] = 0xF0                   # element 15: 0 -> -4.0; element 31: 15 -> 3.5
    w = O.dequant_q4_0(blk[None], 1, 32)[0]
    expect = np.zeros(32)
    expect[0], expect[16], expect[15], expect[31] = 1.0, -2.5, -4.0, 3.5
    assert np.array_equal(w, expect)


def test_q4_1_by_hand():
    blk = np.zeros(20, np.uint8)
    blk[0:2], blk[2:4] = f16(0.25), f16(-1.0)
    blk[5] = 0xF0                    # element 1: 0 -> -1.0; element 17: 15 -> 2.75
    w = O.dequant_q4_1(blk[None], 1, 32)[0]
    expect = np.full(32, -1.0)
    expect[17] = 2.75
    assert np.array_equal(w, expect)


def test_q4_1_with_m_minus_8d_is_q4_0():
    rng = np.random.default_rng(7)
    N, nb = 4, 16
    qs = rng.integers(0, 256, size=(N, nb, 16), dtype=np.uint8)
    d = (2.0 ** -rng.integers(3, 9, size=(N, nb))).astype(np.float16)   # powers of two: -8d exact
    b0 = np.zeros((N, nb, 18), np.uint8)
    b1 = np.zeros((N, nb, 20), np.uint8)
    b0[..., 0:2] = d.view(np.uint8).reshape(N, nb, 2)
    b0[..., 2:18] = qs
    b1[..., 0:2] = d.view(np.uint8).reshape(N, nb, 2)
    b1[..., 2:4] = (-8 * d).astype(np.float16).view(np.uint8).reshape(N, nb, 2)
    b1[..., 4:20] = qs
    K = 32 * nb
    assert np.array_equal(O.dequant_q4_0(b0.reshape(N, -1), N, K), O.dequant_q4_1(b1.reshape(N, -1), N, K))


@pytest.mark.parametrize("kind,bpb,elems", [("q5k", 176, 256), ("q4_0", 18, 32), ("q4_1", 20, 32)])
def test_gemm_rows_is_the_brute_force_dot(kind, bpb, elems):
    """gemm_rows for the new kinds equals the hand loop over k of d_a q_a w on a tiny case."""
    rng = np.random.default_rng(11)
    M, N, K = 2, 3, 256
    w = rng.integers(0, 256, size=(N, K // elems * bpb), dtype=np.uint8)
    for b in range(K // elems):   # finite scales
        w[:, b * bpb:b * bpb + 2] = f16(0.02).reshape(1, 2)
        if kind != "q4_0":
            w[:, b * bpb + 2:b * bpb + 4] = f16(0.01).reshape(1, 2)
    qs = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    d = rng.random((M, K // 32)).astype(np.float32)
    ref, bound = O.gemm_rows(qs, d, w, kind, N, K)
    wd = O.dequant(kind, w, N, K)
    for m in range(M):
        for n in range(N):
            s = 0.0
            for k in range(K):
                s += float(d[m, k // 32]) * int(qs[m, k]) * wd[n, k]
            assert abs(ref[m, n] - s) <= 1e-9 * max(1.0, abs(s))
            assert bound[m, n] >= 0
