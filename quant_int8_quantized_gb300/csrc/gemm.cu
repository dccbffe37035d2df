// Prefill GEMM: q8 activation plane x q4_K / q6_K super-block weights -> f32.
//
// "64 · r60 — the coronation", §3.1-§3.2: for nt >= 16 tokens the matmul runs
// as integer dot products of int8 activation blocks (32 wide, scale d_a) with
// the weight quants, rescaled per block; q6_K runs as k32 chunks whose two
// 16-element halves carry their own int8 scales.
//
// sm_103a has no int8 tcgen05 MMA, so the integer products run on the f16
// tensor pipe with f32 accumulation, on operands that are small integers and
// therefore exact in f16:
//   A (activations): q_a in [-127, 127].
//   B (q4_K):        sc * q with sc in 0..63, q in 0..15, at most 945.
//   B (q6_K):        sc * (q - 32) = sc*lo + 16*sc*(hi - 2) with q = lo + 16*hi,
//                    split into two exact operands (|.| <= 2048 and a multiple
//                    of 16 with |.| <= 4096), accumulated into the same block sum.
// One MMA group per 32-wide activation block yields the exact integer block
// dot I in TMEM (all partial sums are integers below 2^24). The epilogue then
// applies the scales: per block acc += d_a * I (one FMA per element), per
// super-block out += d * acc (and for q4_K out -= dmin * sum_j m_j d_a,j s_j).

#include <cuda_fp16.h>

#include "mq_internal.cuh"
#include "tc.cuh"

namespace {

__device__ unsigned int g_gemm_error;   // bit 0: a bounded wait gave up

constexpr int BM = 128;                 // activation rows per tile (MMA M)
constexpr int BN = 128;                 // weight rows per tile (MMA N)
constexpr int kThreads = 256;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kLBO = 128;          // K-adjacent core matrices
constexpr uint32_t kSBO = 512;          // 8-row groups (32 K = 4 core matrices per row group)
constexpr uint32_t kTileBytes = 128 * 32 * 2;
constexpr uint32_t kTmemCols = 128;

struct __align__(1024) Smem {
    uint8_t a[kTileBytes];
    uint8_t b[2][kTileBytes];
    float wd[BN];
    float wdmin[BN];
    int8_t wsc[BN][16];
    uint8_t wmn[BN][8];
    uint64_t bar;
    uint32_t tmem;
    int abort;
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;   // + alignment slack
constexpr size_t kSmemRequest = 72 * 1024;           // keeps at most 3 CTAs (3 x 128 TMEM columns) per SM

// byte offset of the 8-element group kg (0..3) of row r inside an operand tile
__device__ __forceinline__ uint32_t tile_off(int r, int kg) {
    return (uint32_t)((r >> 3) * kSBO + kg * kLBO + (r & 7) * 16);
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void store_row16(uint8_t* tile, int r, int h, const float (&v)[16]) {
    uint4 p0, p1;
    p0.x = pack_h2(v[0], v[1]);
    p0.y = pack_h2(v[2], v[3]);
    p0.z = pack_h2(v[4], v[5]);
    p0.w = pack_h2(v[6], v[7]);
    p1.x = pack_h2(v[8], v[9]);
    p1.y = pack_h2(v[10], v[11]);
    p1.z = pack_h2(v[12], v[13]);
    p1.w = pack_h2(v[14], v[15]);
    *reinterpret_cast<uint4*>(tile + tile_off(r, 2 * h)) = p0;
    *reinterpret_cast<uint4*>(tile + tile_off(r, 2 * h + 1)) = p1;
}

template <bool Q6>
__global__ void __launch_bounds__(kThreads, 1) gemm_sync_kernel(const int8_t* __restrict__ aq,
                                                                const float* __restrict__ ad,
                                                                const int32_t* __restrict__ as,
                                                                const uint8_t* __restrict__ W,
                                                                float* __restrict__ out, int M, int N, int K) {
    extern __shared__ uint8_t smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int S = K / mq::QK_K, KB = K / mq::QK;
    const size_t row_bytes = (size_t)S * (Q6 ? mq::Q6K_BYTES : mq::Q4K_BYTES);

    if (warp == 0) tc::tmem_alloc(&sm.tmem, kTmemCols);
    if (tid == 0) {
        tc::mbar_init(&sm.bar, 1);
        tc::fence_mbar_init();
        sm.abort = 0;
    }
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = sm.tmem;

    // epilogue ownership: TMEM lane (= tile row) r, 64 columns starting at c0
    const int r = 32 * (warp & 3) + lane;
    const int c0 = 64 * (warp >> 2);
    const int m = m0 + r;
    float outv[64];
#pragma unroll
    for (int c = 0; c < 64; ++c) outv[c] = 0.0f;

    // conversion ownership: tile row cr, 16 K positions starting at 16*ch
    const int cr = tid >> 1, ch = tid & 1;
    const uint32_t idesc = tc::instr_desc(BM, BN, 0);
    uint32_t phase = 0;

    for (int sb = 0; sb < S && !sm.abort; ++sb) {
        // per-super-block weight scales of row n0 + tid
        if (tid < BN) {
            const int n = n0 + tid;
            if (n < N) {
                const uint8_t* blk = W + (size_t)n * row_bytes + (size_t)sb * (Q6 ? mq::Q6K_BYTES : mq::Q4K_BYTES);
                if (Q6) {
                    sm.wd[tid] = __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(blk + 208)));
                    for (int g = 0; g < 16; ++g) sm.wsc[tid][g] = (int8_t)blk[192 + g];
                } else {
                    sm.wd[tid] = __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(blk)));
                    sm.wdmin[tid] = __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(blk + 2)));
                    const uint8_t* q = blk + 4;
                    for (int j = 0; j < 8; ++j) {
                        int sc, mn;
                        if (j < 4) {
                            sc = q[j] & 63;
                            mn = q[j + 4] & 63;
                        } else {
                            sc = (q[j + 4] & 15) | ((q[j - 4] >> 6) << 4);
                            mn = (q[j + 4] >> 4) | ((q[j] >> 6) << 4);
                        }
                        sm.wsc[tid][j] = (int8_t)sc;
                        sm.wmn[tid][j] = (uint8_t)mn;
                    }
                }
            } else {
                sm.wd[tid] = 0.0f;
                sm.wdmin[tid] = 0.0f;
                for (int g = 0; g < 16; ++g) sm.wsc[tid][g] = 0;
                for (int j = 0; j < 8; ++j) sm.wmn[tid][j] = 0;
            }
        }
        __syncthreads();

        float acc[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) acc[c] = 0.0f;
        float beta[8];

        for (int j = 0; j < 8; ++j) {
            const int kb = sb * 8 + j;
            // ---- A: activation quants -> f16
            {
                float v[16];
                const int mm = m0 + cr;
                if (mm < M) {
                    const int4 raw = *reinterpret_cast<const int4*>(aq + (size_t)mm * K + kb * 32 + 16 * ch);
                    const int w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = (float)(int8_t)((w[i >> 2] >> (8 * (i & 3))) & 0xff);
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = 0.0f;
                }
                store_row16(sm.a, cr, ch, v);
            }
            // ---- B: weight quants (with the sub-block scale folded in) -> f16
            {
                const int n = n0 + cr;
                float v1[16], v2[16];
                if (n < N) {
                    const uint8_t* blk = W + (size_t)n * row_bytes + (size_t)sb * (Q6 ? mq::Q6K_BYTES : mq::Q4K_BYTES);
                    if (Q6) {
                        const int hh = j >> 2, tq = j & 3;
                        const int sc = sm.wsc[cr][2 * j + ch];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int l = 16 * ch + i;
                            const int lb = blk[64 * hh + l + 32 * (tq & 1)];
                            const int lo = (tq < 2) ? (lb & 15) : (lb >> 4);
                            const int hi = (blk[128 + 32 * hh + l] >> (2 * tq)) & 3;
                            v1[i] = (float)(sc * lo);
                            v2[i] = (float)(16 * sc * (hi - 2));
                        }
                    } else {
                        const int sc = sm.wsc[cr][j];
                        const uint8_t* qs = blk + 16 + 32 * (j >> 1) + 16 * ch;
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int q = (j & 1) ? (qs[i] >> 4) : (qs[i] & 15);
                            v1[i] = (float)(sc * q);
                        }
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v1[i] = v2[i] = 0.0f;
                }
                store_row16(sm.b[0], cr, ch, v1);
                if (Q6) store_row16(sm.b[1], cr, ch, v2);
            }
            tc::fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0) {
                tc::tc_fence_after();
                const uint32_t sa = tc::smem_u32(sm.a);
#pragma unroll
                for (int part = 0; part < (Q6 ? 2 : 1); ++part) {
                    const uint32_t sbase = tc::smem_u32(sm.b[part]);
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const uint64_t adesc = tc::smem_desc_noswizzle(sa + i * 2 * kLBO, kLBO, kSBO);
                        const uint64_t bdesc = tc::smem_desc_noswizzle(sbase + i * 2 * kLBO, kLBO, kSBO);
                        tc::mma_f16(tmem, adesc, bdesc, idesc, (part | i) ? 1u : 0u);
                    }
                }
                tc::mma_commit(&sm.bar);
            }
            if (!tc::mbar_wait(&sm.bar, phase, kWaitLimitNs)) {
                atomicOr(&g_gemm_error, 1u);
                sm.abort = 1;
            }
            phase ^= 1u;
            tc::tc_fence_after();
            const float da = (m < M) ? ad[(size_t)m * KB + kb] : 0.0f;
            if (!Q6) beta[j] = (m < M) ? da * (float)as[(size_t)m * KB + kb] : 0.0f;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t I[32];
                tc::tmem_ld32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(c0 + 32 * half), I);
                tc::tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 32; ++c) acc[32 * half + c] = fmaf(da, __uint_as_float(I[c]), acc[32 * half + c]);
            }
            tc::tc_fence_before();
            __syncthreads();
            if (sm.abort) break;
        }
        // super-block epilogue
#pragma unroll
        for (int c = 0; c < 64; ++c) {
            const int nl = c0 + c;
            outv[c] = fmaf(sm.wd[nl], acc[c], outv[c]);
            if (!Q6) {
                float t = 0.0f;
#pragma unroll
                for (int j = 0; j < 8; ++j) t = fmaf((float)sm.wmn[nl][j], beta[j], t);
                outv[c] = fmaf(-sm.wdmin[nl], t, outv[c]);
            }
        }
        __syncthreads();
    }

    if (m < M && !sm.abort) {
        float* orow = out + (size_t)m * N;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
            const int n = n0 + c0 + c;
            if (n < N) orow[n] = outv[c];
        }
    }
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

int check_gemm(const mq_q8_plane* a, const void* w, int N, const float* out) {
    if (!a) return MQ_ERR_NULL;
    if (N < 0 || a->M < 0 || !mq::valid_k(a->K)) return MQ_ERR_SHAPE;
    int rc = mq::check_plane(a, a->M, a->K);
    if (rc != MQ_OK || N == 0 || a->M == 0) return rc;
    if (!w || !out) return MQ_ERR_NULL;
    if (!mq::aligned16(w) || !mq::aligned16(out)) return MQ_ERR_ALIGN;
    return mq::check_arch();
}

template <bool Q6>
int launch_gemm(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream) {
    int rc = check_gemm(a, w, N, out);
    if (rc != MQ_OK || N == 0 || a->M == 0) return rc;
    static_assert(kSmemBytes <= kSmemRequest, "shared memory layout too large");
    if (cudaFuncSetAttribute(gemm_sync_kernel<Q6>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemRequest) != cudaSuccess)
        return MQ_ERR_LAUNCH;
    dim3 grid((N + BN - 1) / BN, (a->M + BM - 1) / BM);
    gemm_sync_kernel<Q6><<<grid, kThreads, kSmemRequest, stream>>>(a->qs, a->d, a->s,
                                                                    static_cast<const uint8_t*>(w), out, a->M, N,
                                                                    a->K);
    return mq::launch_status();
}

}  // namespace

namespace mq {
int take_gemm_device_error(cudaStream_t stream, unsigned* code) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MQ_ERR_LAUNCH;
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_gemm_error, sizeof(v)) != cudaSuccess) return MQ_ERR_LAUNCH;
    if (v) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(zero)) != cudaSuccess) return MQ_ERR_LAUNCH;
    }
    *code = v;
    return MQ_OK;
}
}  // namespace mq

extern "C" int mq_gemm_q4k(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream) {
    return launch_gemm<false>(a, w, N, out, stream);
}

extern "C" int mq_gemm_q6k(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream) {
    return launch_gemm<true>(a, w, N, out, stream);
}
