// Decode / small-batch matrix products of a q8 plane by q5_K, q4_0 and q4_1
// weights: the other block types of the pages' decode and prefill dispatch
// ("72 · D3-7 — attn_v-q6K MMVQ routing (2b) + rms wide-block", Excerpt B, the
// q5_K decode arm; "64 · r60 — the coronation", §3.2, Q4_0 / Q4_1 in the matmul
// dispatch). The pages name these types but print no layout; the block formats
// read here are the GGUF blocks of those names:
//   q5_K  176 B per 256: d, dmin (f16), the q4_K 12-byte scale/min field, 32 bytes
//         qh of fifth bits, 128 bytes of nibbles; element 64j + l (l < 32) is the
//         low nibble of byte 32j + l plus 16 * bit 2j of qh[l], element 64j + 32 + l
//         the high nibble plus 16 * bit 2j + 1; w = d * sc * q - dmin * m.
//   q4_0  18 B per 32: d (f16), 16 bytes; element l < 16 the low nibble of byte l,
//         element 16 + l the high nibble; w = d * (q - 8).
//   q4_1  20 B per 32: d, m (f16), 16 bytes as q4_0; w = d * q + m.
//
// Integer dp4a block dots with the int8 activation blocks, then the scales, as the
// q4_K / q6_K GEMVs; up to MQ_GEMV_MAX_ROWS activation rows per call, each weight
// load decoded once and dotted with every row. HBM roofline: the weight stream,
// 0.6875 (q5_K), 0.5625 (q4_0) or 0.625 (q4_1) B per weight, plus 4 B per output.

#include "gemv_common.cuh"

namespace {

using gemv::dp4a_us;
using gemv::kThreads;
using gemv::warp_sum;
constexpr int kQ5KBytes = 176;
constexpr int kQ40Bytes = 18;
constexpr int kQ41Bytes = 20;

// q5_K: a warp takes two consecutive rows at a time; lane = 4*g + p, super-block g
// of an 8-super-block step, 64-element group p (sub-blocks 2p and 2p+1). The lane
// holds the group's 32 nibble bytes and all 32 qh bytes of the super-block.
//   sum q a over sub-block 2p   = sum lo a + 16 * sum (qh >> 2p & 1) a
//   sum q a over sub-block 2p+1 = (sum (16 hi) a) / 16 + 16 * sum (qh >> (2p+1) & 1) a
// with dp4a on bytes masked in place; every sum is an exact integer.
struct Q5Loads {
    uint4 hv[2], q0[2], q1[2], h0[2], h1[2];
};

template <int MR>
__global__ void __launch_bounds__(kThreads) gemv_q5k_kernel(const uint8_t* __restrict__ W,
                                                            const int8_t* __restrict__ aq,
                                                            const float* __restrict__ ad,
                                                            const int32_t* __restrict__ as,
                                                            float* __restrict__ out, int N, int K, int M) {
    const int lane = threadIdx.x & 31;
    const int S = K / mq::QK_K, nst = (S + 7) / 8, nb = K / mq::QK;
    const int g = lane >> 2, p = lane & 3;
    const bool hi = p >= 2;
    const uint32_t sh0 = 16u * (uint32_t)(p & 1), sh1 = sh0 + 8u;
    const size_t row_bytes = (size_t)S * kQ5KBytes;
    const uint32_t m4 = 0x0F0F0F0Fu, m4h = 0xF0F0F0F0u, one = 0x01010101u;
    const int npairs = (N + 1) / 2;
    const int G = gridDim.x * gemv::kWarpsPerBlock;
    for (int pr = blockIdx.x * gemv::kWarpsPerBlock + (threadIdx.x >> 5); pr < npairs; pr += G) {
        const int row = 2 * pr;
        const bool two = row + 1 < N;
        const uint8_t* wr = W + (size_t)row * row_bytes;
        float acc[2][MR];
#pragma unroll
        for (int m = 0; m < MR; ++m) acc[0][m] = acc[1][m] = 0.0f;
        for (int st = 0; st < nst; ++st) {
            const int sb = 8 * st + g;
            if (sb >= S) continue;
            Q5Loads L;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                if (r == 1 && !two) break;
                const uint8_t* b = wr + (size_t)r * row_bytes + (size_t)sb * kQ5KBytes;
                L.hv[r] = __ldg(reinterpret_cast<const uint4*>(b));
                L.h0[r] = __ldg(reinterpret_cast<const uint4*>(b + 16));
                L.h1[r] = __ldg(reinterpret_cast<const uint4*>(b + 32));
                L.q0[r] = __ldcs(reinterpret_cast<const uint4*>(b + 48 + 32 * p));
                L.q1[r] = __ldcs(reinterpret_cast<const uint4*>(b + 64 + 32 * p));
            }
            const int b0 = sb * 8 + 2 * p;
            int sc0[2], sc1[2], mn0[2], mn1[2];
            float d[2], dmin[2];
#pragma unroll
            for (int m = 0; m < MR; ++m) {
                if (m >= M) break;   // uniform
                const int4* a = reinterpret_cast<const int4*>(aq + (size_t)m * K + b0 * 32);
                const int4 a0 = __ldg(a), a1 = __ldg(a + 1), a2 = __ldg(a + 2), a3 = __ldg(a + 3);
                const float2 da = __ldg(reinterpret_cast<const float2*>(ad + (size_t)m * nb + b0));
                const int2 sv = __ldg(reinterpret_cast<const int2*>(as + (size_t)m * nb + b0));
                if (m == 0) {   // per weight row, decoded once the first row's loads are in flight
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const uint4 hv = L.hv[r];
                        const uint32_t x0 = hv.y >> sh0, y0 = hv.z >> sh0, z0 = hv.w >> sh0;
                        const uint32_t x1 = hv.y >> sh1, y1 = hv.z >> sh1, z1 = hv.w >> sh1;
                        sc0[r] = (int)(hi ? ((z0 & 15u) | ((x0 >> 2) & 48u)) : (x0 & 63u));
                        sc1[r] = (int)(hi ? ((z1 & 15u) | ((x1 >> 2) & 48u)) : (x1 & 63u));
                        mn0[r] = (int)(hi ? (((z0 >> 4) & 15u) | ((y0 >> 2) & 48u)) : (y0 & 63u));
                        mn1[r] = (int)(hi ? (((z1 >> 4) & 15u) | ((y1 >> 2) & 48u)) : (y1 & 63u));
                        d[r] = mq_f16_to_f32((uint16_t)(hv.x & 0xffffu));
                        dmin[r] = mq_f16_to_f32((uint16_t)(hv.x >> 16));
                    }
                }
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    if (r == 1 && !two) break;
                    const uint4 q0 = L.q0[r], q1 = L.q1[r], h0 = L.h0[r], h1 = L.h1[r];
                    const int s0 = 2 * p, s1 = 2 * p + 1;
                    int I0 = __dp4a((int)(q0.x & m4), a0.x, 0);
                    I0 = __dp4a((int)(q0.y & m4), a0.y, I0);
                    I0 = __dp4a((int)(q0.z & m4), a0.z, I0);
                    I0 = __dp4a((int)(q0.w & m4), a0.w, I0);
                    I0 = __dp4a((int)(q1.x & m4), a1.x, I0);
                    I0 = __dp4a((int)(q1.y & m4), a1.y, I0);
                    I0 = __dp4a((int)(q1.z & m4), a1.z, I0);
                    I0 = __dp4a((int)(q1.w & m4), a1.w, I0);
                    int F0 = dp4a_us((h0.x >> s0) & one, a0.x, 0);
                    F0 = dp4a_us((h0.y >> s0) & one, a0.y, F0);
                    F0 = dp4a_us((h0.z >> s0) & one, a0.z, F0);
                    F0 = dp4a_us((h0.w >> s0) & one, a0.w, F0);
                    F0 = dp4a_us((h1.x >> s0) & one, a1.x, F0);
                    F0 = dp4a_us((h1.y >> s0) & one, a1.y, F0);
                    F0 = dp4a_us((h1.z >> s0) & one, a1.z, F0);
                    F0 = dp4a_us((h1.w >> s0) & one, a1.w, F0);
                    int H = dp4a_us(q0.x & m4h, a2.x, 0);
                    H = dp4a_us(q0.y & m4h, a2.y, H);
                    H = dp4a_us(q0.z & m4h, a2.z, H);
                    H = dp4a_us(q0.w & m4h, a2.w, H);
                    H = dp4a_us(q1.x & m4h, a3.x, H);
                    H = dp4a_us(q1.y & m4h, a3.y, H);
                    H = dp4a_us(q1.z & m4h, a3.z, H);
                    H = dp4a_us(q1.w & m4h, a3.w, H);
                    int F1 = dp4a_us((h0.x >> s1) & one, a2.x, 0);
                    F1 = dp4a_us((h0.y >> s1) & one, a2.y, F1);
                    F1 = dp4a_us((h0.z >> s1) & one, a2.z, F1);
                    F1 = dp4a_us((h0.w >> s1) & one, a2.w, F1);
                    F1 = dp4a_us((h1.x >> s1) & one, a3.x, F1);
                    F1 = dp4a_us((h1.y >> s1) & one, a3.y, F1);
                    F1 = dp4a_us((h1.z >> s1) & one, a3.z, F1);
                    F1 = dp4a_us((h1.w >> s1) & one, a3.w, F1);
                    const int T0 = I0 + 16 * F0, T1 = (H >> 4) + 16 * F1;   // exact integer dots
                    acc[r][m] += d[r] * (da.x * (float)(sc0[r] * T0) + da.y * (float)(sc1[r] * T1)) -
                                 dmin[r] * (da.x * (float)(mn0[r] * sv.x) + da.y * (float)(mn1[r] * sv.y));
                }
            }
        }
#pragma unroll
        for (int m = 0; m < MR; ++m) {
            if (m >= M) break;
            const float v0 = warp_sum(acc[0][m]), v1 = warp_sum(acc[1][m]);
            if (lane == 0) {
                out[(size_t)m * N + row] = v0;
                if (two) out[(size_t)m * N + row + 1] = v1;
            }
        }
    }
}

// q4_0 / q4_1: one row per warp; lane l takes the 32-element blocks l, l + 32, ...
// A q4_0 block is only 2-byte aligned (18 B), so it is read as nine 16-bit words; a
// q4_1 block (20 B) is 4-byte aligned, five 32-bit words. Nibble bytes w: the low
// nibbles (w & 0x0F0F0F0F) pair with activation bytes 0..15, the high nibbles with
// bytes 16..31; I = sum q a, exact. q4_0: d_w d_a (I - 8 s); q4_1: d_a (d_w I + m s),
// s the activation block's quant sum.
template <bool Q41, int MR>
__global__ void __launch_bounds__(kThreads) gemv_q4x_kernel(const uint8_t* __restrict__ W,
                                                            const int8_t* __restrict__ aq,
                                                            const float* __restrict__ ad,
                                                            const int32_t* __restrict__ as,
                                                            float* __restrict__ out, int N, int K, int M) {
    constexpr int kB = Q41 ? kQ41Bytes : kQ40Bytes;
    const int lane = threadIdx.x & 31;
    const int nb = K / mq::QK;
    const size_t row_bytes = (size_t)nb * kB;
    const uint32_t m4 = 0x0F0F0F0Fu;
    const int G = gridDim.x * gemv::kWarpsPerBlock;
    for (int row = blockIdx.x * gemv::kWarpsPerBlock + (threadIdx.x >> 5); row < N; row += G) {
        const uint8_t* wr = W + (size_t)row * row_bytes;
        float acc[MR];
#pragma unroll
        for (int m = 0; m < MR; ++m) acc[m] = 0.0f;
        for (int b = lane; b < nb; b += 32) {
            const uint8_t* blk = wr + (size_t)b * kB;
            uint32_t q[4];
            float dw, mw = 0.0f;
            if constexpr (Q41) {
                const uint32_t* w32 = reinterpret_cast<const uint32_t*>(blk);
                const uint32_t h = __ldg(w32);
                dw = mq_f16_to_f32((uint16_t)(h & 0xffffu));
                mw = mq_f16_to_f32((uint16_t)(h >> 16));
#pragma unroll
                for (int i = 0; i < 4; ++i) q[i] = __ldcs(w32 + 1 + i);
            } else {
                const unsigned short* w16 = reinterpret_cast<const unsigned short*>(blk);
                dw = mq_f16_to_f32((uint16_t)__ldg(w16));
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    q[i] = (uint32_t)__ldcs(w16 + 1 + 2 * i) | ((uint32_t)__ldcs(w16 + 2 + 2 * i) << 16);
            }
#pragma unroll
            for (int m = 0; m < MR; ++m) {
                if (m >= M) break;   // uniform
                const int4* a = reinterpret_cast<const int4*>(aq + (size_t)m * K + b * 32);
                const int4 a0 = __ldg(a), a1 = __ldg(a + 1);
                const float da = __ldg(ad + (size_t)m * nb + b);
                const int sa = __ldg(as + (size_t)m * nb + b);
                int I = dp4a_us(q[0] & m4, a0.x, 0);
                I = dp4a_us(q[1] & m4, a0.y, I);
                I = dp4a_us(q[2] & m4, a0.z, I);
                I = dp4a_us(q[3] & m4, a0.w, I);
                I = dp4a_us((q[0] >> 4) & m4, a1.x, I);
                I = dp4a_us((q[1] >> 4) & m4, a1.y, I);
                I = dp4a_us((q[2] >> 4) & m4, a1.z, I);
                I = dp4a_us((q[3] >> 4) & m4, a1.w, I);
                if constexpr (Q41) acc[m] += da * (dw * (float)I + mw * (float)sa);
                else acc[m] += dw * da * (float)(I - 8 * sa);
            }
        }
#pragma unroll
        for (int m = 0; m < MR; ++m) {
            if (m >= M) break;
            const float v = warp_sum(acc[m]);
            if (lane == 0) out[(size_t)m * N + row] = v;
        }
    }
}

template <typename K1, typename K2, typename K4, typename K8, typename... Args>
int launch_rows(int M, long long units, K1 k1, K2 k2, K4 k4, K8 k8, cudaStream_t stream, Args... args) {
    auto go = [&](auto kern) {
        return mq::launch_plain(kern, dim3(gemv::grid_for(units, kern)), dim3(kThreads), 0, stream, args...);
    };
    return M == 1 ? go(k1) : M == 2 ? go(k2) : M <= 4 ? go(k4) : go(k8);
}

}  // namespace

extern "C" size_t mq_q5k_row_bytes(int K) { return K > 0 ? (size_t)(K / mq::QK_K) * kQ5KBytes : 0; }
extern "C" size_t mq_q4_0_row_bytes(int K) { return K > 0 ? (size_t)(K / mq::QK) * kQ40Bytes : 0; }
extern "C" size_t mq_q4_1_row_bytes(int K) { return K > 0 ? (size_t)(K / mq::QK) * kQ41Bytes : 0; }

extern "C" int mq_gemv_q5k(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream) {
    int rc = gemv::check(a, w, N, out);
    if (rc != MQ_OK || N == 0) return rc;
    return launch_rows(a->M, (N + 1) / 2, gemv_q5k_kernel<1>, gemv_q5k_kernel<2>, gemv_q5k_kernel<4>,
                       gemv_q5k_kernel<8>, stream, static_cast<const uint8_t*>(w), (const int8_t*)a->qs,
                       (const float*)a->d, (const int32_t*)a->s, out, N, a->K, a->M);
}

extern "C" int mq_gemv_q4_0(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream) {
    int rc = gemv::check(a, w, N, out);
    if (rc != MQ_OK || N == 0) return rc;
    return launch_rows(a->M, N, gemv_q4x_kernel<false, 1>, gemv_q4x_kernel<false, 2>, gemv_q4x_kernel<false, 4>,
                       gemv_q4x_kernel<false, 8>, stream, static_cast<const uint8_t*>(w), (const int8_t*)a->qs,
                       (const float*)a->d, (const int32_t*)a->s, out, N, a->K, a->M);
}

extern "C" int mq_gemv_q4_1(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream) {
    int rc = gemv::check(a, w, N, out);
    if (rc != MQ_OK || N == 0) return rc;
    return launch_rows(a->M, N, gemv_q4x_kernel<true, 1>, gemv_q4x_kernel<true, 2>, gemv_q4x_kernel<true, 4>,
                       gemv_q4x_kernel<true, 8>, stream, static_cast<const uint8_t*>(w), (const int8_t*)a->qs,
                       (const float*)a->d, (const int32_t*)a->s, out, N, a->K, a->M);
}
