// Decode (M == 1) matrix-vector products of a q8 plane by q4_K / q6_K weights.
//
// "72 · D3-7 — attn_v-q6K MMVQ routing (2b) + rms wide-block", §2 (2b) and
// Excerpt A2: the decode matmul streams each weight row once and takes integer
// dot products of 4-bit / 6-bit quants with the int8 activation blocks, then
// applies the block scales. Here one warp owns one output row. Each lane task
// is 32 weights (16 consecutive positions of two sub-blocks), so 8 lanes cover
// one 256-weight super-block and a warp covers 4 super-blocks per step; the
// weight loads of a step are contiguous across the warp. The activation plane
// (a few KB) stays in L1/L2 and is shared by every warp.
//
// HBM roofline: the weight stream, 0.5625 B/weight (q4_K) or 0.8203 B/weight
// (q6_K), plus 4 B per output.

#include "mq_internal.cuh"

namespace {

constexpr int kThreads = 256;        // 8 rows per block
constexpr int kRowsPerBlock = kThreads / 32;
constexpr int kSteps = 4;            // steps (4 super-blocks each) with loads in flight

__device__ __forceinline__ uint32_t byte_of(uint32_t w0, uint32_t w1, uint32_t w2, int i) {
    const uint32_t w = (i < 4) ? w0 : (i < 8 ? w1 : w2);
    return (w >> (8 * (i & 3))) & 0xffu;
}

// 6-bit scale and min of sub-block j from the 12-byte q4_K scale field.
__device__ __forceinline__ void q4k_scale_min(uint32_t w0, uint32_t w1, uint32_t w2, int j, int& sc, int& mn) {
    if (j < 4) {
        sc = (int)(byte_of(w0, w1, w2, j) & 63u);
        mn = (int)(byte_of(w0, w1, w2, j + 4) & 63u);
    } else {
        const uint32_t b = byte_of(w0, w1, w2, j + 4);
        sc = (int)((b & 15u) | ((byte_of(w0, w1, w2, j - 4) >> 6) << 4));
        mn = (int)((b >> 4) | ((byte_of(w0, w1, w2, j) >> 6) << 4));
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__global__ void __launch_bounds__(kThreads) gemv_q4k_kernel(const uint8_t* __restrict__ W,
                                                            const int8_t* __restrict__ aq,
                                                            const float* __restrict__ ad,
                                                            const int32_t* __restrict__ as,
                                                            float* __restrict__ out, int N, int K) {
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
    if (row >= N) return;   // warp-uniform
    const int S = K / mq::QK_K;
    const uint8_t* wr = W + (size_t)row * S * mq::Q4K_BYTES;
    const int t = lane & 7;
    const int p = t >> 1;        // 32-byte group of qs: sub-blocks 2p (low nibbles), 2p+1 (high)
    const int h = t & 1;         // which 16 of the 32 positions
    const int j0 = 2 * p, j1 = 2 * p + 1;
    float acc = 0.0f;
    for (int base = 0; base < S; base += 4 * kSteps) {
        uint4 hv[kSteps], qv[kSteps];
#pragma unroll
        for (int u = 0; u < kSteps; ++u) {
            const int sb = base + 4 * u + (lane >> 3);
            if (sb < S) {
                const uint8_t* blk = wr + (size_t)sb * mq::Q4K_BYTES;
                hv[u] = __ldg(reinterpret_cast<const uint4*>(blk));
                qv[u] = __ldcs(reinterpret_cast<const uint4*>(blk + 16 + 32 * p + 16 * h));
            }
        }
#pragma unroll
        for (int u = 0; u < kSteps; ++u) {
            const int sb = base + 4 * u + (lane >> 3);
            if (sb < S) {
                const int b0 = sb * 8 + j0, b1 = sb * 8 + j1;
                const int4 a0 = __ldg(reinterpret_cast<const int4*>(aq + b0 * 32 + 16 * h));
                const int4 a1 = __ldg(reinterpret_cast<const int4*>(aq + b1 * 32 + 16 * h));
                const uint32_t m4 = 0x0F0F0F0Fu;
                int I0 = 0, I1 = 0;
                I0 = __dp4a((int)(qv[u].x & m4), a0.x, I0);
                I0 = __dp4a((int)(qv[u].y & m4), a0.y, I0);
                I0 = __dp4a((int)(qv[u].z & m4), a0.z, I0);
                I0 = __dp4a((int)(qv[u].w & m4), a0.w, I0);
                I1 = __dp4a((int)((qv[u].x >> 4) & m4), a1.x, I1);
                I1 = __dp4a((int)((qv[u].y >> 4) & m4), a1.y, I1);
                I1 = __dp4a((int)((qv[u].z >> 4) & m4), a1.z, I1);
                I1 = __dp4a((int)((qv[u].w >> 4) & m4), a1.w, I1);
                const float d = mq_f16_to_f32((uint16_t)(hv[u].x & 0xffffu));
                const float dmin = mq_f16_to_f32((uint16_t)(hv[u].x >> 16));
                int sc0, mn0, sc1, mn1;
                q4k_scale_min(hv[u].y, hv[u].z, hv[u].w, j0, sc0, mn0);
                q4k_scale_min(hv[u].y, hv[u].z, hv[u].w, j1, sc1, mn1);
                const float da0 = __ldg(ad + b0), da1 = __ldg(ad + b1);
                acc += da0 * (d * (float)(sc0 * I0)) + da1 * (d * (float)(sc1 * I1));
                if (h == 0) {   // the block-sum (min) term is counted once per 32-block
                    acc -= dmin * (da0 * (float)(mn0 * __ldg(as + b0)) + da1 * (float)(mn1 * __ldg(as + b1)));
                }
            }
        }
    }
    acc = warp_sum(acc);
    if (lane == 0) out[row] = acc;
}

// q6_K rows are only 2-byte aligned (210 B super-blocks), so a lane fetches the
// 16 bytes it needs as five aligned words and realigns them with funnel shifts.
// The words never leave the super-block.
__device__ __forceinline__ void load16_realign(const uint8_t* p, uint32_t out[4]) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~(uintptr_t)3);
    const uint32_t sh = (uint32_t)(a & 3) * 8;
    uint32_t v[5];
#pragma unroll
    for (int i = 0; i < 5; ++i) v[i] = __ldcs(w + i);
#pragma unroll
    for (int i = 0; i < 4; ++i) out[i] = __funnelshift_r(v[i], v[i + 1], sh);
}

// Bytes of 6-bit quants q (0..63) -> bytes of q - 32 as int8: q + 96 never
// carries out of a byte, and flipping bit 7 then subtracts 128.
__device__ __forceinline__ int q6_minus32(uint32_t lo4, uint32_t hi2) {
    return (int)(((lo4 | (hi2 << 4)) + 0x60606060u) ^ 0x80808080u);
}

__global__ void __launch_bounds__(kThreads) gemv_q6k_kernel(const uint8_t* __restrict__ W,
                                                            const int8_t* __restrict__ aq,
                                                            const float* __restrict__ ad,
                                                            float* __restrict__ out, int N, int K) {
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
    if (row >= N) return;   // warp-uniform
    const int S = K / mq::QK_K;
    const uint8_t* wr = W + (size_t)row * S * mq::Q6K_BYTES;
    const int t = lane & 7;
    const int hh = t >> 2;          // half of the super-block (128 elements)
    const int qq = (t >> 1) & 1;    // quarter pair: quarters qq (low nibbles) and qq+2 (high nibbles)
    const int h = t & 1;            // which 16 of the 32 positions
    const int g0 = 8 * hh + 2 * qq + h, g1 = g0 + 4;       // 16-element sub-blocks (scale index)
    const int blk0 = 4 * hh + qq, blk1 = blk0 + 2;          // 32-element activation blocks in the super-block
    float acc = 0.0f;
    for (int base = 0; base < S; base += 4 * kSteps) {
#pragma unroll
        for (int u = 0; u < kSteps; ++u) {
            const int sb = base + 4 * u + (lane >> 3);
            if (sb < S) {
                const uint8_t* blk = wr + (size_t)sb * mq::Q6K_BYTES;
                uint32_t ql[4], qh[4];
                load16_realign(blk + 64 * hh + 32 * qq + 16 * h, ql);
                load16_realign(blk + 128 + 32 * hh + 16 * h, qh);
                const int sc0 = (int)(int8_t)__ldg(blk + 192 + g0);
                const int sc1 = (int)(int8_t)__ldg(blk + 192 + g1);
                const float d = mq_f16_to_f32(__ldg(reinterpret_cast<const unsigned short*>(blk + 208)));
                const int b0 = sb * 8 + blk0, b1 = sb * 8 + blk1;
                const int4 a0 = __ldg(reinterpret_cast<const int4*>(aq + b0 * 32 + 16 * h));
                const int4 a1 = __ldg(reinterpret_cast<const int4*>(aq + b1 * 32 + 16 * h));
                const int a0w[4] = {a0.x, a0.y, a0.z, a0.w};
                const int a1w[4] = {a1.x, a1.y, a1.z, a1.w};
                const uint32_t m4 = 0x0F0F0F0Fu, m2 = 0x03030303u;
                const int s0 = 2 * qq, s1 = 2 * qq + 4;   // qh bit position of quarters qq and qq+2
                int I0 = 0, I1 = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    I0 = __dp4a(q6_minus32(ql[i] & m4, (qh[i] >> s0) & m2), a0w[i], I0);
                    I1 = __dp4a(q6_minus32((ql[i] >> 4) & m4, (qh[i] >> s1) & m2), a1w[i], I1);
                }
                acc += d * (__ldg(ad + b0) * (float)(sc0 * I0) + __ldg(ad + b1) * (float)(sc1 * I1));
            }
        }
    }
    acc = warp_sum(acc);
    if (lane == 0) out[row] = acc;
}

int check_gemv(const mq_q8_plane* a, const void* w, int N, const float* out) {
    if (!a) return MQ_ERR_NULL;
    if (N < 0 || a->M != 1 || !mq::valid_k(a->K)) return MQ_ERR_SHAPE;
    int rc = mq::check_plane(a, a->M, a->K);
    if (rc != MQ_OK || N == 0) return rc;
    if (!w || !out) return MQ_ERR_NULL;
    if (!mq::aligned16(w) || !mq::aligned16(out)) return MQ_ERR_ALIGN;
    return mq::check_arch();
}

}  // namespace

extern "C" int mq_gemv_q4k(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream) {
    int rc = check_gemv(a, w, N, out);
    if (rc != MQ_OK || N == 0) return rc;
    gemv_q4k_kernel<<<(N + kRowsPerBlock - 1) / kRowsPerBlock, kThreads, 0, stream>>>(
        static_cast<const uint8_t*>(w), a->qs, a->d, a->s, out, N, a->K);
    return mq::launch_status();
}

extern "C" int mq_gemv_q6k(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream) {
    int rc = check_gemv(a, w, N, out);
    if (rc != MQ_OK || N == 0) return rc;
    gemv_q6k_kernel<<<(N + kRowsPerBlock - 1) / kRowsPerBlock, kThreads, 0, stream>>>(
        static_cast<const uint8_t*>(w), a->qs, a->d, out, N, a->K);
    return mq::launch_status();
}
