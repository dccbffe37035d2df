// Decode (M == 1) and small-batch matrix-vector products of a q8 plane by q4_K / q6_K weights.
//
// "72 · D3-7 — attn_v-q6K MMVQ routing (2b) + rms wide-block", §2 (2b) and
// Excerpt A2: the decode matmul streams each weight row once and takes integer
// dot products of 4-bit / 6-bit quants with the int8 activation blocks, then
// applies the block scales.
//
// q4_K: a warp owns two consecutive rows at a time (grid-stride over row pairs),
// which share the activation loads. A lane task is 64 weights — two whole
// 32-blocks of one super-block — so the per-block scale work (the 6-bit scale
// decode, the f32 scaling) is spread over as many weights as possible; 4 lanes
// cover a super-block and a warp covers 8 super-blocks per step. (Loads are not
// software-pipelined across steps: the registers that would take cost more in
// occupancy than they gain.) Lane roles are fixed, so the byte positions of a
// lane's scales are known once.
//
// q6_K, prepacked rows (mq_prepack_q6k): the q4_K form (see gemv_q6kp_kernel below).
//
// q6_K, raw rows: one warp per row; a lane task is 32 weights (16 positions of two
// quarters), 8 lanes per super-block, 4 super-blocks per step. The row is staged
// through shared memory by cp.async copies of its 16-byte-aligned window, two
// 8-super-block chunks in flight (three for rows of at most three chunks), so
// that the global loads are few, wide and coalesced although the rows are only
// 2-byte aligned. Two rows (warps) a block.
//
// The activation plane (a few KB) stays in L1/L2 and is shared by every warp.
//
// Both are ordinary launches: they start once the kernel that produced the
// activation plane has completed, so the plane is read-only for their whole
// lifetime and may be read through the non-coherent path (__ldg). (Launched
// early with programmatic serialization, such loads returned a stale plane under
// graph replay, and the coherent loads that fix that made these kernels slower
// than the overlap gained.) A block lets the next kernel on the stream be
// scheduled as soon as it starts, which the producers use.
//
// HBM roofline: the weight stream, 0.5625 B/weight (q4_K) or 0.8203 B/weight
// (q6_K; the prepacked rows read 0.875), plus 4 B per output.

#include "mq_internal.cuh"
#include "gemv_common.cuh"
#include "tc.cuh"

namespace {

using gemv::dp4a_us;
using gemv::kThreads;   // q4_K: 4 warps (row pairs) per block; measured faster than 256 and 512
using gemv::warp_sum;
constexpr int kRowsPerBlock = gemv::kWarpsPerBlock;   // q4_K: warps (row pairs) per block

// Lane = 4*g + p: in each 8-super-block step, super-block g of the step and its
// 32-byte quant group p, i.e. sub-blocks 2p (low nibbles) and 2p+1 (high
// nibbles), all 32 positions. A warp takes two consecutive rows at a time, which
// share the activation loads. The high nibbles are dotted in place (bytes
// 16*hi) and the sum divided by 16, exactly.
struct Q4Loads {
    uint4 hv[2], q0[2], q1[2];   // per row: scale header, quant bytes 0-15 and 16-31 of group p
};

__device__ __forceinline__ void load_q4k(Q4Loads& L, const uint8_t* blk, size_t row_bytes, bool two, int p) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        if (r == 1 && !two) break;
        const uint8_t* b = blk + r * row_bytes;
        L.hv[r] = __ldg(reinterpret_cast<const uint4*>(b));
        L.q0[r] = __ldcs(reinterpret_cast<const uint4*>(b + 16 + 32 * p));
        L.q1[r] = __ldcs(reinterpret_cast<const uint4*>(b + 32 + 32 * p));
    }
}

// MR: activation rows handled per launch (M <= MR); each weight load is decoded
// once and dotted with every row. One-row decode is capped at 64 registers, so that 8
// blocks (32 warps) fit an SM: more row pairs in flight (the token 2% faster than at 80
// registers and 6 blocks; issuing three steps' loads at once at 4 blocks was 7% slower).
template <int MR>
__global__ void __launch_bounds__(kThreads, MR == 1 ? 8 : (MR == 8 ? 4 : 5)) gemv_q4k_kernel(const uint8_t* __restrict__ W,
                                                            const int8_t* __restrict__ aq,
                                                            const float* __restrict__ ad,
                                                            const int32_t* __restrict__ as,
                                                            float* __restrict__ out, int N, int K, int M) {
    mq_grid_release();
    const int lane = threadIdx.x & 31;
    const int S = K / mq::QK_K, nst = (S + 7) / 8, nb = K / mq::QK;
    const int g = lane >> 2, p = lane & 3;
    const bool hi = p >= 2;
    const uint32_t sh0 = 16u * (uint32_t)(p & 1), sh1 = sh0 + 8u;   // byte (2p mod 4), (2p+1 mod 4) of a word
    const size_t row_bytes = (size_t)S * mq::Q4K_BYTES;
    const uint32_t m4 = 0x0F0F0F0Fu, m4h = 0xF0F0F0F0u;
    const int npairs = (N + 1) / 2;
    const int G = gridDim.x * kRowsPerBlock;
    for (int pr = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5); pr < npairs; pr += G) {   // warp-uniform
        const int row = 2 * pr;
        const bool two = row + 1 < N;
        const uint8_t* wr = W + (size_t)row * row_bytes;
        float acc[2][MR];
#pragma unroll
        for (int m = 0; m < MR; ++m) acc[0][m] = acc[1][m] = 0.0f;
        Q4Loads cur;
        for (int st = 0; st < nst; ++st) {
            const int sb = 8 * st + g;
            if (sb < S) {
                load_q4k(cur, wr + (size_t)sb * mq::Q4K_BYTES, row_bytes, two, p);
                const int b0 = sb * 8 + 2 * p;
                int sc0[2], sc1[2], mn0[2], mn1[2];
                float d[2], dmin[2];
#pragma unroll
                for (int m = 0; m < MR; ++m) {
                    if (m >= M) break;   // uniform
                    const int4* a = reinterpret_cast<const int4*>(aq + (size_t)m * K + b0 * 32);   // blocks b0, b0 + 1
                    const int4 a0 = __ldg(a), a1 = __ldg(a + 1), a2 = __ldg(a + 2), a3 = __ldg(a + 3);
                    const float2 da = __ldg(reinterpret_cast<const float2*>(ad + (size_t)m * nb + b0));
                    const int2 sv = __ldg(reinterpret_cast<const int2*>(as + (size_t)m * nb + b0));
                    if (m == 0) {
                        // per weight row, decoded once (after the first row's activation loads
                        // are in flight): the 6-bit scales and mins of sub-blocks 2p, 2p+1, d, dmin
#pragma unroll
                        for (int r = 0; r < 2; ++r) {
                            const uint4 hv = cur.hv[r];
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
                        const uint4 q0 = cur.q0[r], q1 = cur.q1[r];
                        int I0 = __dp4a((int)(q0.x & m4), a0.x, 0);
                        I0 = __dp4a((int)(q0.y & m4), a0.y, I0);
                        I0 = __dp4a((int)(q0.z & m4), a0.z, I0);
                        I0 = __dp4a((int)(q0.w & m4), a0.w, I0);
                        I0 = __dp4a((int)(q1.x & m4), a1.x, I0);
                        I0 = __dp4a((int)(q1.y & m4), a1.y, I0);
                        I0 = __dp4a((int)(q1.z & m4), a1.z, I0);
                        I0 = __dp4a((int)(q1.w & m4), a1.w, I0);
                        int H = dp4a_us(q0.x & m4h, a2.x, 0);
                        H = dp4a_us(q0.y & m4h, a2.y, H);
                        H = dp4a_us(q0.z & m4h, a2.z, H);
                        H = dp4a_us(q0.w & m4h, a2.w, H);
                        H = dp4a_us(q1.x & m4h, a3.x, H);
                        H = dp4a_us(q1.y & m4h, a3.y, H);
                        H = dp4a_us(q1.z & m4h, a3.z, H);
                        H = dp4a_us(q1.w & m4h, a3.w, H);
                        const int I1 = H >> 4;   // exact: every term is a multiple of 16
                        acc[r][m] += d[r] * (da.x * (float)(sc0[r] * I0) + da.y * (float)(sc1[r] * I1)) -
                                     dmin[r] * (da.x * (float)(mn0[r] * sv.x) + da.y * (float)(mn1[r] * sv.y));
                    }
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

// q6_K rows are only 2-byte aligned (210 B super-blocks). Each warp streams its
// row through a ring of kQ6Stages shared-memory buffers, kQ6Chunk super-blocks a
// buffer (rows of up to three chunks get four buffers, so that all of a row is
// requested at once; longer rows get three, which leaves room for more warps): the 16-byte-aligned window around a chunk arrives by 16-byte cp.async
// copies (coalesced, no registers held while in flight). W is 16-byte aligned and
// a chunk is 1680 = 105 * 16 bytes, so every chunk of a row starts at the same
// offset mis (mod 16) inside its window.
constexpr int kQ6Rows = 2;                        // rows (warps) per block: small blocks spread evenly over the SMs
constexpr int kQ6Chunk = 8;                       // super-blocks per buffer
constexpr int kQ6ChunkBytes = 1696;               // 16-aligned window of 8 x 210 B at an even offset
constexpr int kQ6PieceIters = (kQ6ChunkBytes / 16 + 31) / 32;
static_assert(kQ6ChunkBytes % 16 == 0 && kQ6ChunkBytes >= ((14 + kQ6Chunk * mq::Q6K_BYTES + 15) / 16) * 16,
              "q6_K chunk buffer");
static_assert((kQ6Chunk * mq::Q6K_BYTES) % 16 == 0, "chunks keep the row's offset mod 16");

// 16 bytes at a shared address a = 2 (mod 4): five aligned words, halves recombined.
__device__ __forceinline__ void lds16_off2(uint32_t a, uint32_t out[4]) {
    uint32_t v[5];
#pragma unroll
    for (int i = 0; i < 5; ++i) v[i] = tc::lds_u32(a - 2 + 4 * i);
#pragma unroll
    for (int i = 0; i < 4; ++i) out[i] = __byte_perm(v[i], v[i + 1], 0x5432);
}

// Requests `pieces` 16-byte pieces from lo into the buffer at dst. Only the
// matrix's last chunk can end inside a piece; there the piece is read only up to
// the matrix end and zero-filled.
__device__ __forceinline__ void q6_issue_chunk(uint32_t dst, const uint8_t* lo, int pieces, bool last,
                                               const uint8_t* wend, int lane) {
#pragma unroll
    for (int k = 0; k < kQ6PieceIters; ++k) {
        const int i = lane + 32 * k;
        if (i < pieces) {
            const uint8_t* src = lo + 16 * i;
            uint32_t bytes = 16;
            if (last) {
                const ptrdiff_t left = wend - src;
                bytes = left < 16 ? (uint32_t)left : 16u;
            }
            tc::cp_async16_zfill(dst + 16 * i, src, bytes);
        }
    }
}

// Lane = 8*g + t. Step k of a chunk takes super-blocks j = 2g + k (k = 0, 1): the
// four super-blocks of a step start at word offsets that differ mod 4 (their
// shared-memory words fall in distinct banks) and share one alignment mod 4,
// which alternates between the two steps. Within a super-block, t = 4*hh + 2*qq
// + h: half hh, quarters qq (low nibbles of ql) and qq + 2 (high nibbles),
// positions 16h .. 16h + 15 — two 16-element sub-blocks.
//
// Integer dot of sub-block quants q = lo + 16*hi (q - 32 is the weight) with
// activation bytes a, from unsigned-by-signed dp4a on bytes masked in place:
//   L = sum (lo << 4e) a  (e = 0 for low nibbles, 1 for high nibbles),
//   H = sum (hi << 2p) a  (p = the quarter: its qh bit pair),
//   S = sum a,
//   sum (q - 32) a = (L >> 4e) + 16 * (H >> 2p) - 32 * S,
// every shift exact because each sum is a multiple of the power of two.
template <int kQ6Stages, int MR>
__global__ void __launch_bounds__(32 * kQ6Rows) gemv_q6k_kernel(const uint8_t* __restrict__ W,
                                                                const int8_t* __restrict__ aq,
                                                                const float* __restrict__ ad,
                                                                float* __restrict__ out, int N, int K, int M) {
    __shared__ __align__(16) uint8_t stage[kQ6Rows][kQ6Stages][kQ6ChunkBytes];
    mq_grid_release();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int row = blockIdx.x * kQ6Rows + wid;
    if (row >= N) return;   // warp-uniform
    const int S = K / mq::QK_K;
    const int nc = (S + kQ6Chunk - 1) / kQ6Chunk;
    const size_t row_off = (size_t)row * S * mq::Q6K_BYTES;
    const uint32_t mis = (uint32_t)(row_off & 15);
    const uint8_t* wlo = W + (row_off - mis);   // aligned window start of chunk 0
    const uint8_t* wend = W + (size_t)N * S * mq::Q6K_BYTES;
    const bool last_row = row == N - 1;
    const uint32_t buf0 = tc::smem_u32(&stage[wid][0][0]);
    auto pieces_of = [&](int c) {
        const int n = min(kQ6Chunk, S - c * kQ6Chunk);
        return (int)((mis + (uint32_t)n * mq::Q6K_BYTES + 15) >> 4);
    };
#pragma unroll
    for (int c = 0; c < kQ6Stages - 1; ++c) {
        if (c < nc)
            q6_issue_chunk(buf0 + c * kQ6ChunkBytes, wlo + (size_t)c * kQ6Chunk * mq::Q6K_BYTES, pieces_of(c),
                           last_row && c == nc - 1, wend, lane);
        tc::cp_async_commit();
    }
    const int g = lane >> 3, t = lane & 7;
    const int hh = t >> 2, qq = (t >> 1) & 1, h = t & 1;
    const int g0 = 8 * hh + 2 * qq + h, g1 = g0 + 4;       // 16-element sub-blocks (scale index)
    const int blk0 = 4 * hh + qq;                           // 32-element activation block of quarter qq
    const uint32_t off_ql = 64 * hh + 32 * qq + 16 * h, off_qh = 128 + 32 * hh + 16 * h;
    const uint32_t mh0 = 0x03030303u << (2 * qq), mh1 = 0x03030303u << (2 * qq + 4);
    const int shl0 = 4 - 2 * qq, shr1 = 2 * qq;
    const int8_t* aql = aq + blk0 * 32 + 16 * h;            // + 256 per super-block; quarter qq+2 at +64
    const float* adl = ad + blk0;                           // + 8 per super-block; quarter qq+2 at +2
    const int nb = K / mq::QK;
    float acc[MR];
#pragma unroll
    for (int m = 0; m < MR; ++m) acc[m] = 0.0f;
    int stg = 0;
    for (int c = 0; c < nc; ++c) {
        const int cn = c + kQ6Stages - 1;
        if (cn < nc) {
            const int sn = stg == 0 ? kQ6Stages - 1 : stg - 1;   // (c + kQ6Stages - 1) mod kQ6Stages
            q6_issue_chunk(buf0 + sn * kQ6ChunkBytes, wlo + (size_t)cn * kQ6Chunk * mq::Q6K_BYTES, pieces_of(cn),
                           last_row && cn == nc - 1, wend, lane);
        }
        tc::cp_async_commit();
        tc::cp_async_wait<kQ6Stages - 1>();   // this lane's copies of chunk c have landed
        __syncwarp();                          // and every other lane's
        const uint32_t base = buf0 + stg * kQ6ChunkBytes + mis;
        const int n = min(kQ6Chunk, S - c * kQ6Chunk);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int j = 2 * g + k;
            if (j < n) {
                const uint32_t blk = base + j * mq::Q6K_BYTES;
                uint32_t ql[4], qh[4];
                if (((mis + 2 * k) & 3u) == 0) {   // warp-uniform
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        ql[i] = tc::lds_u32(blk + off_ql + 4 * i);
                        qh[i] = tc::lds_u32(blk + off_qh + 4 * i);
                    }
                } else {
                    lds16_off2(blk + off_ql, ql);
                    lds16_off2(blk + off_qh, qh);
                }
                const int sc0 = tc::lds_s8(blk + 192 + g0);
                const int sc1 = tc::lds_s8(blk + 192 + g1);
                const float d = mq_f16_to_f32((uint16_t)tc::lds_u16(blk + 208));
                const int sb = c * kQ6Chunk + j;
#pragma unroll
                for (int m = 0; m < MR; ++m) {
                    if (m >= M) break;   // uniform
                    const int8_t* am = aql + (size_t)m * K + sb * 256;
                    const int4 a0 = __ldg(reinterpret_cast<const int4*>(am));
                    const int4 a1 = __ldg(reinterpret_cast<const int4*>(am + 64));
                    const int a0w[4] = {a0.x, a0.y, a0.z, a0.w};
                    const int a1w[4] = {a1.x, a1.y, a1.z, a1.w};
                    int L0 = 0, L1 = 0, H0 = 0, H1 = 0, S0 = 0, S1 = 0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        L0 = dp4a_us(ql[i] & 0x0F0F0F0Fu, a0w[i], L0);
                        L1 = dp4a_us(ql[i] & 0xF0F0F0F0u, a1w[i], L1);
                        H0 = dp4a_us(qh[i] & mh0, a0w[i], H0);
                        H1 = dp4a_us(qh[i] & mh1, a1w[i], H1);
                        S0 = __dp4a(0x01010101, a0w[i], S0);
                        S1 = __dp4a(0x01010101, a1w[i], S1);
                    }
                    const int I0 = L0 + (H0 << shl0) - (S0 << 5);
                    const int I1 = (L1 >> 4) + (H1 >> shr1) - (S1 << 5);
                    const float* adm = adl + (size_t)m * nb + sb * 8;
                    acc[m] += d * (__ldg(adm) * (float)(sc0 * I0) + __ldg(adm + 2) * (float)(sc1 * I1));
                }
            }
        }
        __syncwarp();   // buffer stg is read by every lane before it is refilled
        stg = stg == kQ6Stages - 1 ? 0 : stg + 1;
    }
#pragma unroll
    for (int m = 0; m < MR; ++m) {
        if (m >= M) break;
        const float v = warp_sum(acc[m]);
        if (lane == 0) out[(size_t)m * N + row] = v;
    }
}

// q6_K in the prepacked layout (mq_prepack_q6k: 224-byte super-blocks, 16-byte aligned,
// each half contiguous: ql 64 B, qh 32 B, 8 int8 scales, f16 d). With every super-block
// aligned the rows need no shared-memory staging: the kernel takes the q4_K GEMV's form, a
// warp on two consecutive rows (sharing the activation loads), 8 super-blocks a step.
// Lane = 4*g + 2*hh + c: super-block g of the step, its half hh and the positions 16c ..
// 16c + 15 of each of the half's four 32-blocks t (elements 128 hh + 32 t + l): four 16-byte
// loads a row (ql bytes 16c.., ql bytes 32 + 16c.., qh bytes 16c.., and the half's scales and
// d), 64 weights. Quarter t takes the low (t < 2) or high nibble of ql[l + 32 (t & 1)], the
// bit pair 2t of qh[l] and scale byte 2t + c; the integer dot is the raw kernel's
// (L >> 4e) + 16 (H >> 2t) - 32 S.
template <int MR>
__global__ void __launch_bounds__(kThreads, MR == 1 ? 6 : 4) gemv_q6kp_kernel(const uint8_t* __restrict__ W,
                                                                          const int8_t* __restrict__ aq,
                                                                          const float* __restrict__ ad,
                                                                          float* __restrict__ out, int N, int K,
                                                                          int M) {
    mq_grid_release();
    const int lane = threadIdx.x & 31;
    const int S = K / mq::QK_K, nst = (S + 7) / 8, nb = K / mq::QK;
    const int g = lane >> 2, hh = (lane >> 1) & 1, c = lane & 1;
    const size_t row_bytes = (size_t)S * mq::Q6K_PACKED_BYTES;
    const int npairs = (N + 1) / 2;
    const int G = gridDim.x * kRowsPerBlock;
    for (int pr = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5); pr < npairs; pr += G) {   // warp-uniform
        const int row = 2 * pr;
        const bool two = row + 1 < N;
        const uint8_t* wr = W + (size_t)row * row_bytes;
        float acc[2][MR];
#pragma unroll
        for (int m = 0; m < MR; ++m) acc[0][m] = acc[1][m] = 0.0f;
        for (int st = 0; st < nst; ++st) {
            const int sb = 8 * st + g;
            if (sb >= S) continue;
            uint4 qa[2], qb[2], qh[2], hd[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                if (r == 1 && !two) break;
                const uint8_t* half = wr + r * row_bytes + (size_t)sb * mq::Q6K_PACKED_BYTES + 112 * hh;
                qa[r] = __ldcs(reinterpret_cast<const uint4*>(half + 16 * c));
                qb[r] = __ldcs(reinterpret_cast<const uint4*>(half + 32 + 16 * c));
                qh[r] = __ldcs(reinterpret_cast<const uint4*>(half + 64 + 16 * c));
                hd[r] = __ldg(reinterpret_cast<const uint4*>(half + 96));
            }
            const int b0 = sb * 8 + 4 * hh;   // the half's first 32-block
#pragma unroll
            for (int m = 0; m < MR; ++m) {
                if (m >= M) break;   // uniform
                const int8_t* am = aq + (size_t)m * K + (size_t)b0 * 32 + 16 * c;
                const float4 da = __ldg(reinterpret_cast<const float4*>(ad + (size_t)m * nb + b0));
                const float dav[4] = {da.x, da.y, da.z, da.w};
                int4 av[4];
                int Sa[4];
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    av[t] = __ldg(reinterpret_cast<const int4*>(am + 32 * t));
                    int s4 = __dp4a(0x01010101, av[t].x, 0);
                    s4 = __dp4a(0x01010101, av[t].y, s4);
                    s4 = __dp4a(0x01010101, av[t].z, s4);
                    Sa[t] = __dp4a(0x01010101, av[t].w, s4);
                }
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    if (r == 1 && !two) break;
                    const uint32_t qaw[4] = {qa[r].x, qa[r].y, qa[r].z, qa[r].w};
                    const uint32_t qbw[4] = {qb[r].x, qb[r].y, qb[r].z, qb[r].w};
                    const uint32_t qhw[4] = {qh[r].x, qh[r].y, qh[r].z, qh[r].w};
                    const uint32_t scw = (c ? (hd[r].x >> 8) : hd[r].x);   // scale bytes 2t + c at bits 16t
                    const uint32_t scw2 = (c ? (hd[r].y >> 8) : hd[r].y);
                    float part = 0.0f;
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int4 a4 = av[t];
                        const int aw[4] = {a4.x, a4.y, a4.z, a4.w};
                        const uint32_t lm = t < 2 ? 0x0F0F0F0Fu : 0xF0F0F0F0u;
                        const uint32_t hm = 0x03030303u << (2 * t);
                        int L = 0, H = 0;
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            L = gemv::dp4a_us(((t & 1) ? qbw[w] : qaw[w]) & lm, aw[w], L);
                            H = gemv::dp4a_us(qhw[w] & hm, aw[w], H);
                        }
                        const int I = (L >> (t < 2 ? 0 : 4)) + 16 * (H >> (2 * t)) - 32 * Sa[t];
                        const int sc = (int)(int8_t)(((t < 2 ? scw : scw2) >> (16 * (t & 1))) & 0xffu);
                        part += dav[t] * (float)(sc * I);
                    }
                    acc[r][m] += mq_f16_to_f32((uint16_t)(hd[r].z & 0xffffu)) * part;
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

}  // namespace

namespace mq {
// The decode kernels have no bounded waits; nothing to report.
int take_gemv_device_error(cudaStream_t, unsigned* code) {
    *code = 0;
    return MQ_OK;
}
}  // namespace mq

extern "C" int mq_gemv_q4k(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream) {
    int rc = gemv::check(a, w, N, out);
    if (rc != MQ_OK || N == 0) return rc;
    auto go = [&](auto kern) {
        return mq::launch_plain(kern, dim3(gemv::grid_for((N + 1) / 2, kern)), dim3(kThreads), 0,
                                stream, static_cast<const uint8_t*>(w), a->qs, a->d, a->s, out, N, a->K, a->M);
    };
    const int M = a->M;
    return M == 1 ? go(gemv_q4k_kernel<1>) : M == 2 ? go(gemv_q4k_kernel<2>) : M <= 4 ? go(gemv_q4k_kernel<4>)
                                                                                  : go(gemv_q4k_kernel<8>);
}

extern "C" int mq_gemv_q6k(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream) {
    int rc = gemv::check(a, w, N, out);
    if (rc != MQ_OK || N == 0) return rc;
    const int chunks = (a->K / mq::QK_K + kQ6Chunk - 1) / kQ6Chunk;
    auto go = [&](auto k4, auto k3) {
        return mq::launch_plain(chunks <= 3 ? k4 : k3, dim3((N + kQ6Rows - 1) / kQ6Rows), dim3(32 * kQ6Rows), 0,
                                stream, static_cast<const uint8_t*>(w), a->qs, a->d, out, N, a->K, a->M);
    };
    const int M = a->M;
    return M == 1   ? go(gemv_q6k_kernel<4, 1>, gemv_q6k_kernel<3, 1>)
           : M == 2 ? go(gemv_q6k_kernel<4, 2>, gemv_q6k_kernel<3, 2>)
           : M <= 4 ? go(gemv_q6k_kernel<4, 4>, gemv_q6k_kernel<3, 4>)
                    : go(gemv_q6k_kernel<4, 8>, gemv_q6k_kernel<3, 8>);
}

extern "C" int mq_gemv_q6k_packed(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream) {
    int rc = gemv::check(a, w, N, out);
    if (rc != MQ_OK || N == 0) return rc;
    auto go = [&](auto kern) {
        return mq::launch_plain(kern, dim3(gemv::grid_for((N + 1) / 2, kern)), dim3(kThreads), 0, stream,
                                static_cast<const uint8_t*>(w), a->qs, a->d, out, N, a->K, a->M);
    };
    const int M = a->M;
    return M == 1 ? go(gemv_q6kp_kernel<1>) : M == 2 ? go(gemv_q6kp_kernel<2>) : M <= 4 ? go(gemv_q6kp_kernel<4>)
                                                                                   : go(gemv_q6kp_kernel<8>);
}
