"""CPU oracle for the block-quantized matmul hot path.

TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and the
cpu_baseline / reference leg of bench.py may import this module. The product
path (the CUDA library and its Python binding) never calls it, and this module
shares no code, table or constant generator with the CUDA path.

Plain, slow, obviously correct numpy. Floating-point steps that decide an
integer (the q8 quantization) run in f32, the precision the pages' kernels use;
dot products run in f64 on dequantized values.

Sources (engineering write-ups of the "minfer" inference engine):
  [r60]  "64 · r60 — the coronation: flipping the verified gate set to default-on"
  [r52]  "55 · r52 — skip-write mode 2: skipping the f32 intermediate write-out"
  [D3-7] "72 · D3-7 — attn_v-q6K MMVQ routing (2b) + rms wide-block / positions memo (2c)"

Readings taken where the pages are silent:
  R1  q4_K super-block byte order (the pages only name the type).
  R2  q6_K super-block byte order.
  R3  an all-zero activation block has d = 0, q = 0, s = 0.
  R4  q = rint(v / d) with an IEEE f32 division (not v * (1/d)).
  R5  rint rounds ties to even.
  R6  q is clamped to [-127, 127].
  R7  d is stored as f32 and s as int32.
  R8  RMSNorm sum-of-squares order: 32 lane partials, lane l serially adding
      float4 number l, l+32, ...; each float4 contributes
      ((x0*x0 + x1*x1) + x2*x2) + x3*x3 with separately rounded f32 ops; the 32
      partials are combined by an xor butterfly at offsets 16, 8, 4, 2, 1.
  R9  scale = 1 / sqrt(ss / K + eps) with correctly rounded f32 sqrt and divide
      (the pages use rsqrtf, an approximation with no exact CPU counterpart).
  R10 SwiGLU's exp is pinned, since an f32 exp has no single correct result:
      e^x by Cody-Waite range reduction (n = rint(x log2 e), r = (x - n ln2_hi)
      - n ln2_lo with a 16-bit ln2_hi, two fused multiply-adds) and the degree-7
      Taylor series in Horner form (one fused multiply-add a step, emulated
      exactly by fma_f32), then the exact scaling by 2^n; 0 below x = -86 and
      +inf above x = 88. With it the SwiGLU
      plane is bit-exact like the others; v = (g / (1 + e^-g)) * u with an IEEE
      f32 division, as the pages write it.
  R11 the GEMM/GEMV error bound is per output element:
      |gpu - oracle| <= 1e-3 * sum_k |a[m,k]| * |w[n,k]|, a the dequantized q8
      activation.
  R21 q5_K super-block byte order (the pages name the type only, in the decode
      dispatch): the GGUF block of that name, 176 bytes: d (f16), dmin (f16),
      the 12-byte scale/min field packed as in q4_K, 32 bytes qh of fifth bits,
      128 bytes of nibbles. Element e = 64j + l (l < 32) takes the low nibble of
      byte 32j + l and bit 2j of qh[l]; element 64j + 32 + l the high nibble and
      bit 2j + 1. w = d * sc[e/32] * q - dmin * m[e/32], q in 0..31.
  R22 q4_0 block byte order (the pages name the type only, in the prefill
      dispatch list): 18 bytes per 32 elements, d (f16) then 16 bytes; element l
      (l < 16) is the low nibble of byte l, element 16 + l the high nibble;
      w = d * (q - 8).
  R23 q4_1 block byte order: 20 bytes per 32 elements, d (f16), m (f16), then
      16 bytes of nibbles placed as in q4_0; w = d * q + m.
  R20 the prefill GEMM reads the activations in an operand form derived from
      the plane (operand_form): each row's super-block of dequantized values
      d * q, scaled by a power of two and rounded to binary16, with its exact
      per-block sums and the power of two. The pages' GEMM consumes the int8
      plane directly; this form is what the f16 tensor pipe multiplies.

Parity pins live in tests/test_oracle.py, tests/test_oracle_order_pins.py,
tests/test_oracle_operand_form.py and tests/test_oracle_block_types.py (closed
forms, hand-built blocks, invariants, brute force). Parity unpinned: whether
R1/R2/R21-R23 match the byte order of real GGUF files (no such file is
available).
"""
from __future__ import annotations

import math

import numpy as np

QK = 32            # activation block length (q8)
QK_K = 256         # weight super-block length
Q4K_BYTES = 144    # d (f16), dmin (f16), 12 bytes of packed 6-bit scales/mins, 128 bytes of nibbles
Q6K_BYTES = 210    # 128 bytes low nibbles, 64 bytes high 2-bit pairs, 16 int8 scales, d (f16)
Q5K_BYTES = 176    # d, dmin (f16), 12 bytes of packed 6-bit scales/mins, 32 bytes of fifth bits, 128 of nibbles
Q4_0_BYTES = 18    # per 32 elements: d (f16), 16 bytes of nibbles
Q4_1_BYTES = 20    # per 32 elements: d (f16), m (f16), 16 bytes of nibbles


# --------------------------------------------------------------------------- f16

def f16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Decode IEEE binary16 bit patterns to float64 (exact, subnormals included)."""
    b = np.asarray(bits).astype(np.int64)
    sign = np.where((b >> 15) & 1, -1.0, 1.0)
    e = (b >> 10) & 0x1F
    m = (b & 0x3FF).astype(np.float64)
    normal = (1.0 + m / 1024.0) * np.exp2(e.astype(np.float64) - 15.0)
    sub = m * 2.0 ** -24
    val = np.where(e == 0, sub, normal)
    val = np.where(e == 31, np.where(m == 0, np.inf, np.nan), val)
    return sign * val


def _u16_le(lo: np.ndarray, hi: np.ndarray) -> np.ndarray:
    return lo.astype(np.int64) | (hi.astype(np.int64) << 8)


# --------------------------------------------------------------------------- q4_K (R1)

def q4k_scales_mins(packed: np.ndarray):
    """Unpack the 12-byte scale field of q4_K into 8 six-bit scales and 8 six-bit mins.

    Sub-blocks 0..3 take the low 6 bits of bytes j (scale) and j+4 (min).
    Sub-blocks 4..7 take a nibble of byte j+4 (low: scale, high: min) and the
    top two bits of byte j-4 (scale) or byte j (min) as bits 4..5.
    """
    q = packed.astype(np.int64)
    sc = np.zeros(q.shape[:-1] + (8,), np.int64)
    mn = np.zeros(q.shape[:-1] + (8,), np.int64)
    for j in range(4):
        sc[..., j] = q[..., j] & 63
        mn[..., j] = q[..., j + 4] & 63
    for j in range(4, 8):
        sc[..., j] = (q[..., j + 4] & 15) | ((q[..., j - 4] >> 6) << 4)
        mn[..., j] = (q[..., j + 4] >> 4) | ((q[..., j] >> 6) << 4)
    return sc, mn


def q4k_fields(w: np.ndarray, N: int, K: int):
    """Split raw q4_K bytes [N, K/256*144] into d, dmin [N,S], sc, mn [N,S,8], q [N,S,256]."""
    S = K // QK_K
    blk = np.asarray(w, np.uint8).reshape(N, S, Q4K_BYTES)
    d = f16_bits_to_f64(_u16_le(blk[..., 0], blk[..., 1]))
    dmin = f16_bits_to_f64(_u16_le(blk[..., 2], blk[..., 3]))
    sc, mn = q4k_scales_mins(blk[..., 4:16])
    qs = blk[..., 16:144].astype(np.int64)
    q = np.zeros((N, S, QK_K), np.int64)
    for p in range(4):                       # 32 bytes hold sub-blocks 2p (low) and 2p+1 (high)
        chunk = qs[..., 32 * p:32 * p + 32]
        q[..., 64 * p:64 * p + 32] = chunk & 15
        q[..., 64 * p + 32:64 * p + 64] = chunk >> 4
    return d, dmin, sc, mn, q


def dequant_q4k(w: np.ndarray, N: int, K: int) -> np.ndarray:
    """w[n,k] = d * sc[j] * q - dmin * m[j], j = (k mod 256) / 32. Returns f64 [N, K]."""
    d, dmin, sc, mn, q = q4k_fields(w, N, K)
    j = np.arange(QK_K) // QK
    out = d[..., None] * sc[..., j] * q - dmin[..., None] * mn[..., j]
    return out.reshape(N, K)


# --------------------------------------------------------------------------- q6_K (R2)

def q6k_fields(w: np.ndarray, N: int, K: int):
    """Split raw q6_K bytes into d [N,S], int8 scales [N,S,16], 6-bit q [N,S,256]."""
    S = K // QK_K
    blk = np.asarray(w, np.uint8).reshape(N, S, Q6K_BYTES)
    ql = blk[..., 0:128].astype(np.int64)
    qh = blk[..., 128:192].astype(np.int64)
    sc = blk[..., 192:208].view(np.int8).astype(np.int64)
    d = f16_bits_to_f64(_u16_le(blk[..., 208], blk[..., 209]))
    e = np.arange(QK_K)
    h, r = e // 128, e % 128          # half of the super-block
    t, l = r // 32, r % 32            # quarter within the half, position in the quarter
    low_byte = ql[..., 64 * h + l + 32 * (t & 1)]
    low = np.where(t < 2, low_byte & 15, low_byte >> 4)
    high = (qh[..., 32 * h + l] >> (2 * t)) & 3
    q = low | (high << 4)
    return d, sc, q


def dequant_q6k(w: np.ndarray, N: int, K: int) -> np.ndarray:
    """w[n,k] = d * sc[g] * (q - 32), g = (k mod 256) / 16. Returns f64 [N, K]."""
    d, sc, q = q6k_fields(w, N, K)
    g = np.arange(QK_K) // 16
    out = d[..., None] * sc[..., g] * (q - 32)
    return out.reshape(N, K)


# --------------------------------------------------------------------------- q5_K (R21)

def q5k_fields(w: np.ndarray, N: int, K: int):
    """Split raw q5_K bytes [N, K/256*176] into d, dmin [N,S], sc, mn [N,S,8], q [N,S,256]."""
    S = K // QK_K
    blk = np.asarray(w, np.uint8).reshape(N, S, Q5K_BYTES)
    d = f16_bits_to_f64(_u16_le(blk[..., 0], blk[..., 1]))
    dmin = f16_bits_to_f64(_u16_le(blk[..., 2], blk[..., 3]))
    sc, mn = q4k_scales_mins(blk[..., 4:16])
    qh = blk[..., 16:48].astype(np.int64)
    qs = blk[..., 48:176].astype(np.int64)
    q = np.zeros((N, S, QK_K), np.int64)
    for j in range(4):
        nib = qs[..., 32 * j:32 * j + 32]
        q[..., 64 * j:64 * j + 32] = (nib & 15) | (((qh >> (2 * j)) & 1) << 4)
        q[..., 64 * j + 32:64 * j + 64] = (nib >> 4) | (((qh >> (2 * j + 1)) & 1) << 4)
    return d, dmin, sc, mn, q


def dequant_q5k(w: np.ndarray, N: int, K: int) -> np.ndarray:
    """w[n,k] = d * sc[j] * q - dmin * m[j], j = (k mod 256) / 32, q in 0..31. f64 [N, K]."""
    d, dmin, sc, mn, q = q5k_fields(w, N, K)
    j = np.arange(QK_K) // QK
    out = d[..., None] * sc[..., j] * q - dmin[..., None] * mn[..., j]
    return out.reshape(N, K)


# --------------------------------------------------------------------------- q4_0, q4_1 (R22, R23)

def _nibbles32(qs: np.ndarray) -> np.ndarray:
    """16 bytes -> 32 four-bit values: low nibbles first (elements 0..15), then high."""
    q = qs.astype(np.int64)
    return np.concatenate([q & 15, q >> 4], axis=-1)


def dequant_q4_0(w: np.ndarray, N: int, K: int) -> np.ndarray:
    """w[n,k] = d * (q - 8) per block of 32. f64 [N, K]."""
    blk = np.asarray(w, np.uint8).reshape(N, K // QK, Q4_0_BYTES)
    d = f16_bits_to_f64(_u16_le(blk[..., 0], blk[..., 1]))
    q = _nibbles32(blk[..., 2:18])
    return (d[..., None] * (q - 8)).reshape(N, K)


def dequant_q4_1(w: np.ndarray, N: int, K: int) -> np.ndarray:
    """w[n,k] = d * q + m per block of 32. f64 [N, K]."""
    blk = np.asarray(w, np.uint8).reshape(N, K // QK, Q4_1_BYTES)
    d = f16_bits_to_f64(_u16_le(blk[..., 0], blk[..., 1]))
    m = f16_bits_to_f64(_u16_le(blk[..., 2], blk[..., 3]))
    q = _nibbles32(blk[..., 4:20])
    return (d[..., None] * q + m[..., None]).reshape(N, K)


def dequant(kind: str, w: np.ndarray, N: int, K: int) -> np.ndarray:
    return {"q4k": dequant_q4k, "q6k": dequant_q6k, "q5k": dequant_q5k, "q4_0": dequant_q4_0,
            "q4_1": dequant_q4_1}[kind](w, N, K)


# --------------------------------------------------------------------------- q8 activations

def quantize_q8(v: np.ndarray):
    """Quantize f32 rows to blocks of 32 ([r52] §2.2; [D3-7] Excerpt C's per-block epilogue).

    Per block: amax = max |v| (exact), d = amax / 127 (f32), q = rint(v / d)
    clamped to [-127, 127] (R4-R6), s = sum q (int32). d == 0 gives q = 0 (R3).
    Returns qs int8 [M, K], d f32 [M, K/32], s int32 [M, K/32].
    """
    v = np.asarray(v, np.float32)
    M, K = v.shape
    blocks = v.reshape(M, K // QK, QK)
    amax = np.max(np.abs(blocks), axis=-1)
    d = (amax / np.float32(127.0)).astype(np.float32)
    nz = d != 0
    safe = np.where(nz, d, np.float32(1.0)).astype(np.float32)
    q = np.rint(blocks / safe[..., None])
    q = np.clip(q, -127, 127)
    q = np.where(nz[..., None], q, 0).astype(np.int8)
    s = q.astype(np.int32).sum(axis=-1, dtype=np.int32)
    return q.reshape(M, K), d, s


def operand_form(qs: np.ndarray, d: np.ndarray):
    """The prefill GEMM's activation operand, derived from a q8 plane (R20).

    For every row m and super-block t (8 blocks of 32):
      D = max_j d[m, 8t + j];  e = 3 - E where D = f * 2^E, f in [1/2, 1) (so that
      D * 2^e lies in [4, 8)), clamped to [-126, 126]; e = 0 when D == 0;
      ah[m, k] = f16(f32(d * q) * 2^e)           (the f32 product rounded, then
                                                  scaled exactly, then rounded to
                                                  binary16, ties to even);
      sigma_j = sum of the 32 ah values of block j (exact in f32: they are
                multiples of the smallest one's ulp and stay below 2^15);
      ax[m, t, j] = f16(sigma_j), ax[m, t, 8 + j] = f16(sigma_j - ax[m, t, j]);
      af[t, m] = 2^-e (f32).
    Then 2^-e * ah is the dequantized activation d * q to within 2^-11 relative
    (binary16 normal range), and 2^-e * (ax_hi + ax_lo) the block sums of those
    values to within 2^-22 relative.
    Returns ah f16 [M, K], ax f16 [M, K/256, 16], af f32 [K/256, M].
    """
    qs = np.asarray(qs)
    d = np.asarray(d, np.float32)
    M, K = qs.shape
    S = K // QK_K
    D = d.reshape(M, S, 8).max(axis=-1)
    _, E = np.frexp(D)
    e = np.clip(3 - E, -126, 126)
    e = np.where(D == 0, 0, e).astype(np.int64)
    scale = np.ldexp(np.float32(1.0), e.astype(np.int32)).astype(np.float32)          # [M, S]
    dq = (np.repeat(d, QK, axis=1) * qs.astype(np.float32)).astype(np.float32)       # f32(d * q)
    t = (dq.reshape(M, S, QK_K) * scale[..., None]).astype(np.float32)              # exact scaling
    ah = t.astype(np.float16).reshape(M, K)
    sig = ah.astype(np.float32).reshape(M, S, 8, QK).astype(np.float64).sum(axis=-1)
    sig32 = sig.astype(np.float32)
    assert np.all(sig32.astype(np.float64) == sig), "block sum of ah not exact in f32"
    hi = sig32.astype(np.float16)
    lo = (sig32 - hi.astype(np.float32)).astype(np.float32).astype(np.float16)
    ax = np.concatenate([hi, lo], axis=-1)
    af = np.ldexp(np.float32(1.0), (-e).astype(np.int32)).astype(np.float32).T.copy()
    return ah, ax, af


def dequant_plane(qs: np.ndarray, d: np.ndarray) -> np.ndarray:
    """a[m,k] = d[m, k/32] * q[m,k] in f64."""
    M, K = qs.shape
    return (qs.astype(np.float64).reshape(M, K // QK, QK) * d.astype(np.float64)[..., None]).reshape(M, K)


# --------------------------------------------------------------------------- fused producers

def rms_sumsq(x: np.ndarray) -> np.ndarray:
    """Per-row sum of squares in f32, in the R8 order ([r52] §3.2; [D3-7] §2c(i), Excerpt C).

    Lane l (0..31) keeps a running f32 sum over float4 number l, l+32, l+64, ... of the
    row, each float4 adding ((x0*x0 + x1*x1) + x2*x2) + x3*x3 with every product and sum
    rounded separately; the 32 lane sums are then combined by an xor butterfly at
    offsets 16, 8, 4, 2, 1 (every lane ends with the same value).
    """
    x = np.asarray(x, np.float32)
    M, K = x.shape
    f4 = x.reshape(M, K // 128, 32, 4)          # float4 number 32*j + lane
    lane = np.zeros((M, 32), np.float32)
    for j in range(K // 128):                   # each lane's serial chain
        v = f4[:, j]
        term = ((v[..., 0] * v[..., 0] + v[..., 1] * v[..., 1]) + v[..., 2] * v[..., 2]) + v[..., 3] * v[..., 3]
        lane = lane + term
    idx = np.arange(32)
    for off in (16, 8, 4, 2, 1):                # xor butterfly
        lane = lane + lane[:, idx ^ off]
    return lane[:, 0]


def rms_scale(x: np.ndarray, eps: float) -> np.ndarray:
    """Per-row 1/sqrt(mean(x^2) + eps) in f32 with the R8 sum and correctly rounded ops (R9)."""
    x = np.asarray(x, np.float32)
    ss = rms_sumsq(x)
    K = x.shape[1]
    return (np.float32(1.0) / np.sqrt(ss / np.float32(K) + np.float32(eps))).astype(np.float32)


def rms_values(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """The f32 RMSNorm output v = (x * scale) * w that the fused producer quantizes."""
    x = np.asarray(x, np.float32)
    scale = rms_scale(x, eps)
    return ((x * scale[:, None]) * np.asarray(w, np.float32)[None, :]).astype(np.float32)


def rms_quant(x: np.ndarray, w: np.ndarray, eps: float):
    """Fused RMSNorm -> q8 plane ([r52] §3.2 mode-2 rms kernel): quantize_q8(rms_values)."""
    return quantize_q8(rms_values(x, w, eps))


def fma_f32(a, b, c) -> np.ndarray:
    """a*b + c rounded once to f32 (IEEE fused multiply-add) for f32 a, b, c.

    a*b is exact in f64 (two 24-bit significands). s = a*b + c is rounded to f64
    and its error e = (a*b + c) - s recovered exactly (Knuth's TwoSum). Rounding s
    to f32 is then the correct rounding of a*b + c, unless s lies exactly halfway
    between two f32 values while e != 0 (a midpoint has at most 25 significant
    bits, so no other midpoint can separate s from the exact value); there the
    exact value lies on e's side of the midpoint. Results stay normal here.
    """
    f64 = np.float64
    a64, b64, c64 = (np.asarray(v, np.float32).astype(f64) for v in (a, b, c))
    p = a64 * b64
    s = p + c64
    bv = s - p
    e = (p - (s - bv)) + (c64 - bv)
    r = s.astype(np.float32)
    other = np.nextafter(r, np.where(s > r.astype(f64), np.float32(np.inf), np.float32(-np.inf)))
    mid = (r.astype(f64) + other.astype(f64)) * 0.5
    tie = (s != r.astype(f64)) & (s == mid) & (e != 0)
    fixed = np.where(e > 0, np.maximum(r, other), np.minimum(r, other))
    return np.where(tie, fixed, r).astype(np.float32)


def exp_f32(x: np.ndarray) -> np.ndarray:
    """e^x in f32 (R10): Cody-Waite range reduction and the Taylor series.

    n = rint(x * log2(e)) (product rounded to f32, then ties-to-even),
    r = fma(-n, ln2_lo, fma(-n, ln2_hi, x)) with ln2_hi = 0.693145751953125 (16
    significant bits) and ln2_lo = ln 2 - ln2_hi in f32,
    p = 1 + r(1 + r(1/2! + r(1/3! + ... + r/7!))) in Horner form, one fused
    multiply-add per step, each coefficient 1/k! rounded to f32, and
    e^x = p * 2^n (exact: n is in [-124, 127] on [-86, 88], so the product stays
    normal). Below -86, e^x < 2^-124 and 1 + e^x rounds to 1, so 0 is returned;
    above 88, +inf.
    """
    f32 = np.float32
    x = np.asarray(x, f32)
    log2e = f32(1.0 / math.log(2.0))
    ln2_hi = f32(0.693145751953125)
    ln2_lo = f32(math.log(2.0) - 0.693145751953125)
    coef = [f32(1.0 / math.factorial(k)) for k in range(8)]
    xc = np.clip(x, f32(-86.0), f32(88.0))
    n = np.rint(xc * log2e)
    r = fma_f32(-n, ln2_lo, fma_f32(-n, ln2_hi, xc))
    p = np.full_like(xc, coef[7])
    for k in range(6, -1, -1):
        p = fma_f32(p, r, coef[k])
    e = (p * np.ldexp(f32(1.0), n.astype(np.int32))).astype(f32)
    e = np.where(x < f32(-86.0), f32(0.0), e)
    return np.where(x > f32(88.0), f32(np.inf), e).astype(f32)


def swiglu_values(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """v = (g / (1 + exp(-g))) * u in f32 ([r52] §3.2 mode-2 swiglu kernel; R10)."""
    g = np.asarray(g, np.float32)
    u = np.asarray(u, np.float32)
    e = exp_f32(-g)
    return ((g / (np.float32(1.0) + e)) * u).astype(np.float32)


def swiglu_quant(g: np.ndarray, u: np.ndarray):
    """Fused SwiGLU -> q8 plane: quantize_q8(swiglu_values)."""
    return quantize_q8(swiglu_values(g, u))


# --------------------------------------------------------------------------- matmul

def gemm(qs: np.ndarray, d: np.ndarray, w_deq: np.ndarray) -> np.ndarray:
    """out[m,n] = sum_k (d_a[m,k/32] q_a[m,k]) * w[n,k] in f64 ([r60] §3.2 MMQ dispatch)."""
    return dequant_plane(qs, d) @ np.asarray(w_deq, np.float64).T


def gemm_bound(qs: np.ndarray, d: np.ndarray, w_deq: np.ndarray, rel: float = 1e-3) -> np.ndarray:
    """Per-element tolerance rel * sum_k |a[m,k]| |w[n,k]| (R11)."""
    return rel * (np.abs(dequant_plane(qs, d)) @ np.abs(np.asarray(w_deq, np.float64)).T)


def gemm_rows(qs, d, w_raw, kind: str, N: int, K: int, rows=None, cols=None):
    """Oracle GEMM on a subset of output rows / columns (dequantizes only what it needs)."""
    rows = np.arange(qs.shape[0]) if rows is None else np.asarray(rows)
    cols = np.arange(N) if cols is None else np.asarray(cols)
    row_bytes = w_raw.shape[1]
    wsub = np.asarray(w_raw, np.uint8).reshape(N, row_bytes)[cols]
    wdeq = dequant(kind, wsub, len(cols), K)
    a_q, a_d = np.asarray(qs)[rows], np.asarray(d)[rows]
    return gemm(a_q, a_d, wdeq), gemm_bound(a_q, a_d, wdeq)
