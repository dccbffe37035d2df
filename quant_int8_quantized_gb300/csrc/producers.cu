// q8 plane producers: standalone quantize, fused RMSNorm -> q8, fused SwiGLU -> q8.
//
// All three share the lane mapping of the pages' mode-2 kernels ("55 · r52 —
// skip-write mode 2", §3.2): a warp sweeps 128 consecutive floats per round,
// lane l owns float4 number l, so the 8 lanes of group l>>3 own one 32-block
// (block index 4*round + (l>>3)). amax and the int sum of a block are reduced
// with xor shuffles at 4, 2, 1 — exact in any order ("55 · r52", §2.2). Loads
// and the qs store of a round are 512 B / 128 B coalesced warp accesses
// ("55 · r52", §3.3 pitfall 2). No f32 intermediate is ever written.
//
// HBM roofline: quantize reads 4 B and writes 1.25 B per element; rms reads
// 4 B (x) and writes 1.25 B; swiglu reads 8 B (g, u) and writes 1.25 B.

#include "mq_internal.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kRoundsPerIter = 4;   // float4 loads in flight per lane (inputs of a few rows: 1, more warps)

__device__ __forceinline__ void store_round(uint32_t* __restrict__ qs, float* __restrict__ d,
                                            int32_t* __restrict__ s, uint2* __restrict__ qh, long long round,
                                            int lane, uint32_t q, float dd, int ss, uint2 h) {
    qs[round * 32 + lane] = q;
    if (qh) qh[round * 32 + lane] = h;
    if ((lane & 7) == 0) {
        const long long b = round * 4 + (lane >> 3);
        d[b] = dd;
        s[b] = ss;
    }
}

// x is viewed as a flat array of M*K floats (rows are contiguous, K % 128 == 0),
// so every round lies inside one row and the plane arrays are flat too.
template <int R>
__global__ void __launch_bounds__(kThreads) quantize_q8_kernel(const float4* __restrict__ x,
                                                               uint32_t* __restrict__ qs,
                                                               float* __restrict__ d,
                                                               int32_t* __restrict__ s,
                                                               uint2* __restrict__ qh, long long rounds) {
    mq_grid_release();
    mq_grid_wait();
    const int lane = threadIdx.x & 31;
    const long long warp = ((long long)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * kThreads) >> 5;
    for (long long r0 = warp * R; r0 < rounds; r0 += nwarps * R) {
        float4 v[R];
#pragma unroll
        for (int u = 0; u < R; ++u)
            if (r0 + u < rounds) v[u] = __ldcs(x + (r0 + u) * 32 + lane);
#pragma unroll
        for (int u = 0; u < R; ++u) {
            if (r0 + u < rounds) {   // warp-uniform
                float dd;
                int ss;
                uint2 h;
                const uint32_t q = mq_quant4_group8(v[u].x, v[u].y, v[u].z, v[u].w, dd, ss, h);
                store_round(qs, d, s, qh, r0 + u, lane, q, dd, ss, h);
            }
        }
    }
}

// e^x in f32 by Cody-Waite range reduction and the Taylor series, with every
// step one correctly rounded operation (a multiply, or a fused multiply-add), so
// that the result is fixed bit for bit:
//   n = rint(x * log2 e),  r = fma(-n, ln2_lo, fma(-n, ln2_hi, x)),
//   p = 1 + r (1 + r (1/2! + r (1/3! + ... + r / 7!)))  (Horner, one fma a step),
//   e^x = p * 2^n.
// ln2_hi = 0.693145751953125 has 16 significant bits; ln2_lo = ln 2 - ln2_hi. The
// coefficients are 1/k! rounded to f32. On [-86, 88] n lies in [-124, 127], so
// 2^n and p * 2^n are normal and the scaling is exact. Below -86, e^x < 2^-124
// vanishes next to 1 in 1 + e^x: 0 is returned; above 88, +inf. Within 0.91 ulp
// of e^x on [-86, 88].
__device__ __forceinline__ float exp_cw(float x) {
    if (x < -86.0f) return 0.0f;
    if (x > 88.0f) return __int_as_float(0x7f800000);
    const float n = rintf(__fmul_rn(x, 0x1.715476p+0f));
    const float r = __fmaf_rn(-n, 0x1.7f7d1cp-20f, __fmaf_rn(-n, 0x1.62e4p-1f, x));
    float p = 0x1.a01a02p-13f;              // 1/7!
    p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);   // 1/6!
    p = __fmaf_rn(p, r, 0x1.111112p-7f);    // 1/5!
    p = __fmaf_rn(p, r, 0x1.555556p-5f);    // 1/4!
    p = __fmaf_rn(p, r, 0x1.555556p-3f);    // 1/3!
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    return __fmul_rn(p, __int_as_float(((int)n + 127) << 23));
}

// (g / (1 + e^-g)) * u as the pages write it: an IEEE division and correctly
// rounded f32 operations, with the exp above, so the plane is bit-exact.
__device__ __forceinline__ float silu_mul(float g, float u) {
    return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, exp_cw(-g))), u);
}

template <int R>
__global__ void __launch_bounds__(kThreads) swiglu_quant_kernel(const float4* __restrict__ g,
                                                                const float4* __restrict__ u,
                                                                uint32_t* __restrict__ qs,
                                                                float* __restrict__ d,
                                                                int32_t* __restrict__ s,
                                                                uint2* __restrict__ qh, long long rounds) {
    mq_grid_release();
    mq_grid_wait();
    const int lane = threadIdx.x & 31;
    const long long warp = ((long long)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * kThreads) >> 5;
    for (long long r0 = warp * R; r0 < rounds; r0 += nwarps * R) {
        float4 gv[R], uv[R];
#pragma unroll
        for (int k = 0; k < R; ++k) {
            if (r0 + k < rounds) {
                gv[k] = __ldcs(g + (r0 + k) * 32 + lane);
                uv[k] = __ldcs(u + (r0 + k) * 32 + lane);
            }
        }
#pragma unroll
        for (int k = 0; k < R; ++k) {
            if (r0 + k < rounds) {
                float dd;
                int ss;
                uint2 h;
                const uint32_t q = mq_quant4_group8(silu_mul(gv[k].x, uv[k].x), silu_mul(gv[k].y, uv[k].y),
                                                    silu_mul(gv[k].z, uv[k].z), silu_mul(gv[k].w, uv[k].w),
                                                    dd, ss, h);
                store_round(qs, d, s, qh, r0 + k, lane, q, dd, ss, h);
            }
        }
    }
}

// RMSNorm scale of one row in the fixed order: lane l serially adds float4 l,
// l+32, ... (each as ((x0*x0 + x1*x1) + x2*x2) + x3*x3, every op separately
// rounded), then an xor butterfly 16, 8, 4, 2, 1; scale = 1 / sqrt(ss/K + eps)
// ("55 · r52", §3.2 phase 1; "72 · D3-7", §2c(i) and Excerpt C).
__device__ __forceinline__ float sum_sq4(float4 v) {
    float t = __fadd_rn(__fmul_rn(v.x, v.x), __fmul_rn(v.y, v.y));
    t = __fadd_rn(t, __fmul_rn(v.z, v.z));
    return __fadd_rn(t, __fmul_rn(v.w, v.w));
}

__device__ __forceinline__ float rms_scale_finish(float ss, int K, float eps) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, off));
    return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)K), eps)));
}

__device__ __forceinline__ float rms_scale_warp(const float4* __restrict__ xr, int K, float eps, int lane) {
    const int K4 = K >> 2;
    float ss = 0.0f;
#pragma unroll 8
    for (int i = lane; i < K4; i += 32) ss = __fadd_rn(ss, sum_sq4(mq_ld_dep(xr + i)));
    return rms_scale_finish(ss, K, eps);
}

__device__ __forceinline__ void rms_quant_one(float4 xv, float4 wv, float scale, uint32_t* __restrict__ qs,
                                              float* __restrict__ d, int32_t* __restrict__ s,
                                              uint2* __restrict__ qh, long long round, int lane) {
    float dd;
    int ss;
    uint2 h;
    const uint32_t q = mq_quant4_group8(__fmul_rn(__fmul_rn(xv.x, scale), wv.x), __fmul_rn(__fmul_rn(xv.y, scale), wv.y),
                                        __fmul_rn(__fmul_rn(xv.z, scale), wv.z), __fmul_rn(__fmul_rn(xv.w, scale), wv.w),
                                        dd, ss, h);
    store_round(qs, d, s, qh, round, lane, q, dd, ss, h);
}

// Rows of at most 32 * kRegRoundsMax rounds (K <= 16384): one block per row, round
// r held in registers by warp r % nw (at most kRegRounds rounds a warp), all of
// a row's loads in flight at once.
// Each lane leaves the sum of squares of its float4 of each round in shared
// memory; warp 0 adds them per lane in round order — the same sequence as
// rms_scale_warp — and the scale goes through shared memory. The row is read
// from HBM once ("72 · D3-7", Excerpt C: a wide block per decode row).
constexpr int kRegRoundsMax = 4;

template <bool kPrefetchW, int kRegRounds>
__global__ void __launch_bounds__(1024) rms_quant_staged_kernel(const float4* __restrict__ x,
                                                                const float4* __restrict__ w4,
                                                                uint32_t* __restrict__ qs,
                                                                float* __restrict__ d,
                                                                int32_t* __restrict__ s,
                                                                uint2* __restrict__ qh, int K, float eps) {
    mq_grid_release();
    mq_grid_wait();
    extern __shared__ float s_sq[];   // [rounds][32]
    __shared__ float s_scale;
    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int nrounds = K >> 7;
    const float4* xr = x + (long long)blockIdx.x * (K >> 2);
    float4 xv[kRegRounds];
#pragma unroll
    for (int i = 0; i < kRegRounds; ++i) {
        const int r = wid + i * nw;
        if (r < nrounds) xv[i] = __ldcs(xr + r * 32 + lane);
    }
#pragma unroll
    for (int i = 0; i < kRegRounds; ++i) {
        const int r = wid + i * nw;
        if (r < nrounds) s_sq[r * 32 + lane] = sum_sq4(xv[i]);
    }
    float4 wv[kRegRounds];   // for a few rows the weight row is fetched while warp 0 computes the scale
    if constexpr (kPrefetchW) {
#pragma unroll
        for (int i = 0; i < kRegRounds; ++i) {
            const int r = wid + i * nw;
            if (r < nrounds) wv[i] = __ldg(w4 + r * 32 + lane);
        }
    }
    __syncthreads();
    if (wid == 0) {
        float ss = 0.0f;
#pragma unroll 8
        for (int r = 0; r < nrounds; ++r) ss = __fadd_rn(ss, s_sq[r * 32 + lane]);
        const float sc = rms_scale_finish(ss, K, eps);
        if (lane == 0) s_scale = sc;
    }
    __syncthreads();
    const float scale = s_scale;
    const long long round0 = (long long)blockIdx.x * nrounds;
#pragma unroll
    for (int i = 0; i < kRegRounds; ++i) {
        const int r = wid + i * nw;
        if (r < nrounds)
            rms_quant_one(xv[i], kPrefetchW ? wv[i] : __ldg(w4 + r * 32 + lane), scale, qs, d, s, qh, round0 + r, lane);
    }
}

// Longer rows: one block per row with one warp per round (at most 32 warps, or 4
// when there are many rows; more rounds wrap around). Every warp loads its first
// round while warp 0 computes the scale with rms_scale_warp (the row is read
// twice, the second time mostly from cache).
__global__ void __launch_bounds__(1024) rms_quant_wide_kernel(const float4* __restrict__ x,
                                                              const float4* __restrict__ w4,
                                                              uint32_t* __restrict__ qs,
                                                              float* __restrict__ d,
                                                              int32_t* __restrict__ s,
                                                              uint2* __restrict__ qh, int K, float eps) {
    mq_grid_release();
    mq_grid_wait();
    __shared__ float s_scale;
    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int nrounds = K >> 7;
    const float4* xr = x + (long long)blockIdx.x * (K >> 2);
    const float4 x0 = mq_ld_dep(xr + wid * 32 + lane);   // wid < nrounds by construction of the launch
    const float4 w0 = __ldg(w4 + wid * 32 + lane);
    if (wid == 0) {
        const float sc = rms_scale_warp(xr, K, eps, lane);
        if (lane == 0) s_scale = sc;
    }
    __syncthreads();
    const float scale = s_scale;
    const long long round0 = (long long)blockIdx.x * nrounds;
    rms_quant_one(x0, w0, scale, qs, d, s, qh, round0 + wid, lane);
#pragma unroll 2
    for (int k = wid + nw; k < nrounds; k += nw)
        rms_quant_one(mq_ld_dep(xr + k * 32 + lane), __ldg(w4 + k * 32 + lane), scale, qs, d, s, qh, round0 + k, lane);
}

// Inputs that would not give every SM two blocks at four rounds a warp (decode
// rows) are spread one round per warp: the rounds' latencies then overlap across
// warps instead of queueing inside one.
bool few_rounds(long long rounds) { return rounds < 2LL * mq::num_sms() * (kThreads / 32) * kRoundsPerIter; }

int flat_grid(long long rounds, int rounds_per_iter) {
    const long long per_block = (kThreads / 32) * rounds_per_iter;
    long long blocks = (rounds + per_block - 1) / per_block;
    const long long cap = (long long)mq::num_sms() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return (int)blocks;
}

int check_producer(const void* a, const void* b, int M, int K, const mq_q8_plane* out) {
    if (M < 0 || !mq::valid_k(K)) return MQ_ERR_SHAPE;
    int rc = mq::check_plane(out, M, K);
    if (rc != MQ_OK || M == 0) return rc;
    if (!a || !b) return MQ_ERR_NULL;
    if (!mq::aligned16(a) || !mq::aligned16(b)) return MQ_ERR_ALIGN;
    return mq::check_arch();
}

}  // namespace

extern "C" int mq_quantize_q8(const float* x, int M, int K, const mq_q8_plane* out, cudaStream_t stream) {
    int rc = check_producer(x, x, M, K, out);
    if (rc != MQ_OK || M == 0) return rc;
    const long long rounds = (long long)M * K / 128;
    const bool few = few_rounds(rounds);
    return mq::launch_pdl(few ? quantize_q8_kernel<1> : quantize_q8_kernel<kRoundsPerIter>,
                          dim3(flat_grid(rounds, few ? 1 : kRoundsPerIter)), dim3(kThreads), 0, stream,
                          reinterpret_cast<const float4*>(x), reinterpret_cast<uint32_t*>(out->qs), out->d, out->s,
                          reinterpret_cast<uint2*>(out->qh), rounds);
}

extern "C" int mq_swiglu_quant(const float* g, const float* u, int M, int K, const mq_q8_plane* out,
                               cudaStream_t stream) {
    int rc = check_producer(g, u, M, K, out);
    if (rc != MQ_OK || M == 0) return rc;
    const long long rounds = (long long)M * K / 128;
    const bool few = few_rounds(rounds);
    return mq::launch_pdl(few ? swiglu_quant_kernel<1> : swiglu_quant_kernel<kRoundsPerIter>,
                          dim3(flat_grid(rounds, few ? 1 : kRoundsPerIter)), dim3(kThreads), 0, stream,
                          reinterpret_cast<const float4*>(g), reinterpret_cast<const float4*>(u),
                          reinterpret_cast<uint32_t*>(out->qs), out->d, out->s, reinterpret_cast<uint2*>(out->qh),
                          rounds);
}

extern "C" int mq_rms_quant(const float* x, const float* w, int M, int K, float eps, const mq_q8_plane* out,
                            cudaStream_t stream) {
    int rc = check_producer(x, w, M, K, out);
    if (rc != MQ_OK || M == 0) return rc;
    const float4* x4 = reinterpret_cast<const float4*>(x);
    const float4* w4 = reinterpret_cast<const float4*>(w);
    uint32_t* qs = reinterpret_cast<uint32_t*>(out->qs);
    uint2* qh = reinterpret_cast<uint2*>(out->qh);
    // One block per row. Rows of up to 128 rounds are read once into registers: one warp
    // per round for a few rows (decode); two rounds a warp (four for rows over 64 rounds)
    // once there are enough rows to fill the machine. Longer rows take the kernel that
    // reads them twice.
    const int rounds = K / 128;
    const bool many = M >= 4 * mq::num_sms();
    if (rounds <= 32 * kRegRoundsMax) {
        const size_t smem = (size_t)rounds * 32 * sizeof(float);
        if (!many)
            return mq::launch_pdl(rms_quant_staged_kernel<true, kRegRoundsMax>, dim3(M),
                                  dim3(32 * (rounds < 32 ? rounds : 32)), smem, stream, x4, w4, qs, out->d, out->s, qh,
                                  K, eps);
        if (rounds <= 64)   // two rounds a warp (measured faster than four at 3314 x 3584)
            return mq::launch_pdl(rms_quant_staged_kernel<false, 2>, dim3(M), dim3(32 * ((rounds + 1) / 2)), smem,
                                  stream, x4, w4, qs, out->d, out->s, qh, K, eps);
        return mq::launch_pdl(rms_quant_staged_kernel<false, kRegRoundsMax>, dim3(M),
                              dim3(32 * ((rounds + kRegRoundsMax - 1) / kRegRoundsMax)), smem, stream, x4, w4, qs, out->d,
                              out->s, qh, K, eps);
    }
    const int cap = many ? 4 : 32;
    const int warps = rounds < cap ? rounds : cap;
    return mq::launch_pdl(rms_quant_wide_kernel, dim3(M), dim3(32 * warps), 0, stream, x4, w4, qs, out->d, out->s, qh,
                          K, eps);
}
