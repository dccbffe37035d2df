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
// A plane may also carry the prefill GEMM's operand form (ah, ax, af; see mq.h).
// It is derived per super-block of 256, i.e. per pair of rounds (2p, 2p+1), which
// is why the kernels hand whole pairs to a warp: the super-block's largest block
// scale is a warp-wide max, the block sums of ah are xor-shuffle sums (exact:
// the values of one block are multiples of its smallest one's ulp and stay far
// below 2^24 of it).
//
// HBM roofline per element: quantize reads 4 B, rms 4 B (x), swiglu 8 B (g, u);
// the q8 arrays take 1.25 B, the operand arrays 2.25 B.

#include "mq_internal.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kRoundsPerIter = 4;   // float4 loads in flight per lane (inputs of a few rows: fewer, more warps)

// Where a producer writes: the q8 arrays (qs == nullptr: absent) and the operand
// arrays (ah == nullptr: absent). Plane arrays are flat: rows are contiguous and a
// round (128 elements) never crosses a row, nor a pair of rounds a super-block.
struct Out {
    uint32_t* qs;
    float* d;
    int32_t* s;
    uint2* ah;
    uint16_t* ax;
    float* af;
    int kr;     // rounds per row (K / 128)
    int mp;     // af row stride (M rounded up to a multiple of 4)
};

__device__ __forceinline__ void store_q8(const Out& o, long long round, int lane, uint32_t q, float dd, int ss) {
    o.qs[round * 32 + lane] = q;
    if ((lane & 7) == 0) {
        const long long b = round * 4 + (lane >> 3);
        o.d[b] = dd;
        o.s[b] = ss;
    }
}

// Quantize one round (q8 arrays only).
__device__ __forceinline__ void quant_round(const Out& o, long long round, int lane, float v0, float v1, float v2,
                                            float v3) {
    float dd;
    int ss, q[4];
    const uint32_t pq = mq_quant4_group8(v0, v1, v2, v3, dd, ss, q);
    store_q8(o, round, lane, pq, dd, ss);
}

// Quantize the two rounds of super-block `pair` (rounds 2 pair, 2 pair + 1) and write
// every array group the plane holds. v[r] is this lane's float4 of round r.
__device__ __forceinline__ void quant_pair(const Out& o, long long pair, int lane, const float4 (&v)[2]) {
    float dd[2];
    int ss[2], q[2][4];
    uint32_t pq[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) pq[r] = mq_quant4_group8(v[r].x, v[r].y, v[r].z, v[r].w, dd[r], ss[r], q[r]);
    const long long r0 = 2 * pair;
    if (o.qs) {
        store_q8(o, r0, lane, pq[0], dd[0], ss[0]);
        store_q8(o, r0 + 1, lane, pq[1], dd[1], ss[1]);
    }
    if (o.ah) {
        // e from the super-block's largest block scale D (a max, exact in any order):
        // D = f 2^E with f in [1/2, 1), e = 3 - E clamped to [-126, 126], e = 0 for D = 0.
        float D = fmaxf(dd[0], dd[1]);
        D = fmaxf(D, __shfl_xor_sync(0xffffffffu, D, 8));
        D = fmaxf(D, __shfl_xor_sync(0xffffffffu, D, 16));
        int e = 0;
        if (D >= 0x1p-126f) {   // normal: D = 1.m 2^(b - 127) = 0.1m 2^(b - 126)
            e = min(126, max(-126, 3 - (((int)(__float_as_uint(D) >> 23) & 0xff) - 126)));
        } else if (D != 0.0f) {
            int E;
            frexpf(D, &E);
            e = min(126, max(-126, 3 - E));
        }
        const float scale = __int_as_float((e + 127) << 23);      // 2^e, exact
        float sig[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            // f16(f32(d q) 2^e), two values per packed multiply; the block sum of these binary16
            // values is exact in f32 in any order (see above), so it is taken pairwise
            const float2 p01 = f2_mul(f2_mul(f2_dup(dd[r]), make_float2((float)q[r][0], (float)q[r][1])), f2_dup(scale));
            const float2 p23 = f2_mul(f2_mul(f2_dup(dd[r]), make_float2((float)q[r][2], (float)q[r][3])), f2_dup(scale));
            const __half2 h01 = __floats2half2_rn(p01.x, p01.y), h23 = __floats2half2_rn(p23.x, p23.y);
            const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
            const float2 pr = f2_add(f01, f23);
            float part = __fadd_rn(pr.x, pr.y);
            o.ah[(r0 + r) * 32 + lane] = make_uint2(*reinterpret_cast<const uint32_t*>(&h01),
                                                    *reinterpret_cast<const uint32_t*>(&h23));
            part = __fadd_rn(part, __shfl_xor_sync(0xffffffffu, part, 4));
            part = __fadd_rn(part, __shfl_xor_sync(0xffffffffu, part, 2));
            part = __fadd_rn(part, __shfl_xor_sync(0xffffffffu, part, 1));
            sig[r] = part;
        }
        if ((lane & 7) == 0) {   // block j = 4r + lane/8 of the super-block: slots j (hi), 8 + j (lo)
            uint16_t* rec = o.ax + pair * 16;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const __half hi = __float2half_rn(sig[r]);
                const __half lo = __float2half_rn(__fsub_rn(sig[r], __half2float(hi)));
                const int j = 4 * r + (lane >> 3);
                rec[j] = __half_as_ushort(hi);
                rec[8 + j] = __half_as_ushort(lo);
            }
        }
        if (lane == 0) {
            const int spr = o.kr >> 1;                                 // super-blocks per row
            const long long row = pair / spr;
            const int t = (int)(pair - row * spr);
            o.af[(long long)t * o.mp + row] = __int_as_float((127 - e) << 23);   // 2^-e
        }
    }
}

// x is viewed as a flat array of M*K floats (rows are contiguous, K % 256 == 0).
// R rounds per warp and iteration; R >= 2 is even, so every pair of rounds is one
// super-block (required when the plane holds the operand form). R == 1 writes the q8
// arrays only.
template <int R>
__global__ void __launch_bounds__(kThreads, 4) quantize_q8_kernel(const float4* __restrict__ x, Out o, long long rounds) {
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
        if constexpr (R == 1) {
            quant_round(o, r0, lane, v[0].x, v[0].y, v[0].z, v[0].w);
        } else {
#pragma unroll
            for (int u = 0; u < R; u += 2) {
                if (r0 + u < rounds) {   // warp-uniform; rounds is even, so the pair is whole
                    const float4 pv[2] = {v[u], v[u + 1]};
                    quant_pair(o, (r0 + u) >> 1, lane, pv);
                }
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
__device__ __forceinline__ float2 exp_cw2(float2 x) {   // two values, packed arithmetic
    const float2 t = f2_mul(x, f2_dup(0x1.715476p+0f));
    const float2 n = make_float2(rintf(t.x), rintf(t.y));
    const float2 r = f2_fma(n, f2_dup(-0x1.7f7d1cp-20f), f2_fma(n, f2_dup(-0x1.62e4p-1f), x));
    float2 p = f2_dup(0x1.a01a02p-13f);                 // 1/7!
    p = f2_fma(p, r, f2_dup(0x1.6c16c2p-10f));          // 1/6!
    p = f2_fma(p, r, f2_dup(0x1.111112p-7f));           // 1/5!
    p = f2_fma(p, r, f2_dup(0x1.555556p-5f));           // 1/4!
    p = f2_fma(p, r, f2_dup(0x1.555556p-3f));           // 1/3!
    p = f2_fma(p, r, f2_dup(0.5f));
    p = f2_fma(p, r, f2_dup(1.0f));
    p = f2_fma(p, r, f2_dup(1.0f));
    // 2^n is formed for every x; outside [-86, 88] the result is replaced below
    float2 e = f2_mul(p, make_float2(__int_as_float(((int)n.x + 127) << 23), __int_as_float(((int)n.y + 127) << 23)));
    if (x.x < -86.0f) e.x = 0.0f;
    if (x.x > 88.0f) e.x = __int_as_float(0x7f800000);
    if (x.y < -86.0f) e.y = 0.0f;
    if (x.y > 88.0f) e.y = __int_as_float(0x7f800000);
    return e;
}

// (g / (1 + e^-g)) * u as the pages write it: an IEEE division and correctly
// rounded f32 operations, with the exp above, so the plane is bit-exact.
__device__ __forceinline__ float2 silu_mul2(float2 g, float2 u) {
    const float2 den = f2_add(f2_dup(1.0f), exp_cw2(make_float2(-g.x, -g.y)));
    return f2_mul(make_float2(__fdiv_rn(g.x, den.x), __fdiv_rn(g.y, den.y)), u);
}

__device__ __forceinline__ float4 silu_mul4(float4 g, float4 u) {
    const float2 a = silu_mul2(make_float2(g.x, g.y), make_float2(u.x, u.y));
    const float2 b = silu_mul2(make_float2(g.z, g.w), make_float2(u.z, u.w));
    return make_float4(a.x, a.y, b.x, b.y);
}

template <int R>
__global__ void __launch_bounds__(kThreads, 4) swiglu_quant_kernel(const float4* __restrict__ g,
                                                                const float4* __restrict__ u, Out o,
                                                                long long rounds) {
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
        if constexpr (R == 1) {
            const float4 v = silu_mul4(gv[0], uv[0]);
            quant_round(o, r0, lane, v.x, v.y, v.z, v.w);
        } else {
#pragma unroll
            for (int k = 0; k < R; k += 2) {
                if (r0 + k < rounds) {
                    const float4 pv[2] = {silu_mul4(gv[k], uv[k]), silu_mul4(gv[k + 1], uv[k + 1])};
                    quant_pair(o, (r0 + k) >> 1, lane, pv);
                }
            }
        }
    }
}

// RMSNorm scale of one row in the fixed order: lane l serially adds float4 l,
// l+32, ... (each as ((x0*x0 + x1*x1) + x2*x2) + x3*x3, every op separately
// rounded), then an xor butterfly 16, 8, 4, 2, 1; scale = 1 / sqrt(ss/K + eps)
// ("55 · r52", §3.2 phase 1; "72 · D3-7", §2c(i) and Excerpt C).
__device__ __forceinline__ float sum_sq4(float4 v) {
    const float2 a = f2_mul(make_float2(v.x, v.y), make_float2(v.x, v.y));
    const float2 b = f2_mul(make_float2(v.z, v.w), make_float2(v.z, v.w));
    return __fadd_rn(__fadd_rn(__fadd_rn(a.x, a.y), b.x), b.y);
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

__device__ __forceinline__ float4 rms_apply(float4 xv, float4 wv, float scale) {   // (x scale) w
    const float2 a = f2_mul(f2_mul(make_float2(xv.x, xv.y), f2_dup(scale)), make_float2(wv.x, wv.y));
    const float2 b = f2_mul(f2_mul(make_float2(xv.z, xv.w), f2_dup(scale)), make_float2(wv.z, wv.w));
    return make_float4(a.x, a.y, b.x, b.y);
}

// Rows of at most 64 * kRegPairsMax rounds (K <= 16384): one block per row; pair p
// (rounds 2p, 2p+1) is held in registers by warp p % nw, at most kRegPairs pairs a
// warp, all of a row's loads in flight at once.
// Each lane leaves the sum of squares of its float4 of each round in shared
// memory; warp 0 adds them per lane in round order — the same sequence as
// rms_scale_warp — and the scale goes through shared memory. The row is read
// from HBM once ("72 · D3-7", Excerpt C: a wide block per decode row).
constexpr int kRegPairsMax = 2;

template <bool kPrefetchW, int kRegPairs>
__global__ void __launch_bounds__(1024) rms_quant_staged_kernel(const float4* __restrict__ x,
                                                                const float4* __restrict__ w4, Out o, int K,
                                                                float eps) {
    mq_grid_release();
    mq_grid_wait();
    extern __shared__ float s_sq[];   // [rounds][32]
    __shared__ float s_scale;
    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int nrounds = K >> 7, npairs = nrounds >> 1;
    const float4* xr = x + (long long)blockIdx.x * (K >> 2);
    float4 xv[kRegPairs][2];
#pragma unroll
    for (int i = 0; i < kRegPairs; ++i) {
        const int p = wid + i * nw;
        if (p < npairs) {
            xv[i][0] = __ldcs(xr + (2 * p) * 32 + lane);
            xv[i][1] = __ldcs(xr + (2 * p + 1) * 32 + lane);
        }
    }
#pragma unroll
    for (int i = 0; i < kRegPairs; ++i) {
        const int p = wid + i * nw;
        if (p < npairs) {
            s_sq[(2 * p) * 32 + lane] = sum_sq4(xv[i][0]);
            s_sq[(2 * p + 1) * 32 + lane] = sum_sq4(xv[i][1]);
        }
    }
    float4 wv[kRegPairs][2];   // for a few rows the weight row is fetched while warp 0 computes the scale
    if constexpr (kPrefetchW) {
#pragma unroll
        for (int i = 0; i < kRegPairs; ++i) {
            const int p = wid + i * nw;
            if (p < npairs) {
                wv[i][0] = __ldg(w4 + (2 * p) * 32 + lane);
                wv[i][1] = __ldg(w4 + (2 * p + 1) * 32 + lane);
            }
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
    const long long pair0 = (long long)blockIdx.x * npairs;
#pragma unroll
    for (int i = 0; i < kRegPairs; ++i) {
        const int p = wid + i * nw;
        if (p < npairs) {
            const float4 w0 = kPrefetchW ? wv[i][0] : __ldg(w4 + (2 * p) * 32 + lane);
            const float4 w1 = kPrefetchW ? wv[i][1] : __ldg(w4 + (2 * p + 1) * 32 + lane);
            const float4 pv[2] = {rms_apply(xv[i][0], w0, scale), rms_apply(xv[i][1], w1, scale)};
            quant_pair(o, pair0 + p, lane, pv);
        }
    }
}

// Longer rows: one block per row with one warp per pair of rounds (at most 32 warps,
// or 4 when there are many rows; more pairs wrap around). Every warp loads its first
// pair while warp 0 computes the scale with rms_scale_warp (the row is read twice,
// the second time mostly from cache).
__global__ void __launch_bounds__(1024) rms_quant_wide_kernel(const float4* __restrict__ x,
                                                              const float4* __restrict__ w4, Out o, int K,
                                                              float eps) {
    mq_grid_release();
    mq_grid_wait();
    __shared__ float s_scale;
    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int npairs = K >> 8;
    const float4* xr = x + (long long)blockIdx.x * (K >> 2);
    // wid < npairs by construction of the launch
    const float4 x0 = mq_ld_dep(xr + (2 * wid) * 32 + lane), x1 = mq_ld_dep(xr + (2 * wid + 1) * 32 + lane);
    const float4 w0 = __ldg(w4 + (2 * wid) * 32 + lane), w1 = __ldg(w4 + (2 * wid + 1) * 32 + lane);
    if (wid == 0) {
        const float sc = rms_scale_warp(xr, K, eps, lane);
        if (lane == 0) s_scale = sc;
    }
    __syncthreads();
    const float scale = s_scale;
    const long long pair0 = (long long)blockIdx.x * npairs;
    {
        const float4 pv[2] = {rms_apply(x0, w0, scale), rms_apply(x1, w1, scale)};
        quant_pair(o, pair0 + wid, lane, pv);
    }
#pragma unroll 2
    for (int p = wid + nw; p < npairs; p += nw) {
        const float4 pv[2] = {rms_apply(mq_ld_dep(xr + (2 * p) * 32 + lane), __ldg(w4 + (2 * p) * 32 + lane), scale),
                              rms_apply(mq_ld_dep(xr + (2 * p + 1) * 32 + lane), __ldg(w4 + (2 * p + 1) * 32 + lane),
                                        scale)};
        quant_pair(o, pair0 + p, lane, pv);
    }
}

// Inputs that would not give every SM two blocks at four rounds a warp (decode
// rows) are spread one round per warp (two when the operand form is written): the
// rounds' latencies then overlap across warps instead of queueing inside one.
bool few_rounds(long long rounds) { return rounds < 2LL * mq::num_sms() * (kThreads / 32) * kRoundsPerIter; }

// One wave: as many blocks as are resident at once (the warps stride over the rounds),
// never more than the rounds need.
template <typename Kern>
int flat_grid(long long rounds, int rounds_per_iter, Kern kern) {
    const long long per_block = (kThreads / 32) * rounds_per_iter;
    long long blocks = (rounds + per_block - 1) / per_block;
    const long long cap = (long long)mq::num_sms() * mq::resident_blocks(reinterpret_cast<const void*>(kern), kThreads, 0);
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

Out out_of(const mq_q8_plane* p) {
    return Out{reinterpret_cast<uint32_t*>(p->qs), p->d, p->s, reinterpret_cast<uint2*>(p->ah), p->ax, p->af,
               p->K / 128, mq::af_stride(p->M)};
}

// Rounds per warp and iteration of the flat kernels.
int flat_rounds(long long rounds, const mq_q8_plane* out) {
    if (!few_rounds(rounds)) return kRoundsPerIter;
    return mq::has_op(out) ? 2 : 1;
}

}  // namespace

extern "C" int mq_quantize_q8(const float* x, int M, int K, const mq_q8_plane* out, cudaStream_t stream) {
    int rc = check_producer(x, x, M, K, out);
    if (rc != MQ_OK || M == 0) return rc;
    const long long rounds = (long long)M * K / 128;
    const int R = flat_rounds(rounds, out);
    auto kern = R == 1 ? quantize_q8_kernel<1> : R == 2 ? quantize_q8_kernel<2> : quantize_q8_kernel<kRoundsPerIter>;
    return mq::launch_pdl(kern, dim3(flat_grid(rounds, R, kern)), dim3(kThreads), 0, stream,
                          reinterpret_cast<const float4*>(x), out_of(out), rounds);
}

extern "C" int mq_swiglu_quant(const float* g, const float* u, int M, int K, const mq_q8_plane* out,
                               cudaStream_t stream) {
    int rc = check_producer(g, u, M, K, out);
    if (rc != MQ_OK || M == 0) return rc;
    const long long rounds = (long long)M * K / 128;
    const int R = flat_rounds(rounds, out);
    auto kern = R == 1 ? swiglu_quant_kernel<1> : R == 2 ? swiglu_quant_kernel<2> : swiglu_quant_kernel<kRoundsPerIter>;
    return mq::launch_pdl(kern, dim3(flat_grid(rounds, R, kern)), dim3(kThreads), 0, stream,
                          reinterpret_cast<const float4*>(g), reinterpret_cast<const float4*>(u), out_of(out), rounds);
}

extern "C" int mq_rms_quant(const float* x, const float* w, int M, int K, float eps, const mq_q8_plane* out,
                            cudaStream_t stream) {
    int rc = check_producer(x, w, M, K, out);
    if (rc != MQ_OK || M == 0) return rc;
    const float4* x4 = reinterpret_cast<const float4*>(x);
    const float4* w4 = reinterpret_cast<const float4*>(w);
    const Out o = out_of(out);
    // One block per row. Rows of up to 64 pairs of rounds are read once into registers:
    // one warp per pair for a few rows (decode) and for rows of up to 32 pairs; two pairs
    // a warp for longer rows when there are enough rows to fill the machine. Longer rows
    // take the kernel that reads them twice.
    const int rounds = K / 128, pairs = rounds / 2;
    const bool many = M >= 4 * mq::num_sms();
    if (pairs <= 32 * kRegPairsMax) {
        const size_t smem = (size_t)rounds * 32 * sizeof(float);
        if (!many)
            return mq::launch_pdl(rms_quant_staged_kernel<true, kRegPairsMax>, dim3(M),
                                  dim3(32 * (pairs < 32 ? pairs : 32)), smem, stream, x4, w4, o, K, eps);
        if (pairs <= 32)   // one pair (two rounds) a warp: measured fastest at 3314 x 3584
            return mq::launch_pdl(rms_quant_staged_kernel<false, 1>, dim3(M), dim3(32 * pairs), smem, stream, x4,
                                  w4, o, K, eps);
        return mq::launch_pdl(rms_quant_staged_kernel<false, kRegPairsMax>, dim3(M),
                              dim3(32 * ((pairs + kRegPairsMax - 1) / kRegPairsMax)), smem, stream, x4, w4, o, K,
                              eps);
    }
    const int cap = many ? 4 : 32;
    const int warps = pairs < cap ? pairs : cap;
    return mq::launch_pdl(rms_quant_wide_kernel, dim3(M), dim3(32 * warps), 0, stream, x4, w4, o, K, eps);
}
