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
//   B (q4_K):        sc * q with sc in 0..63, q in 0..15 (at most 945).
//   B (q6_K):        sc * (q - 32) = sc*lo + 16*sc*(hi - 2) with q = lo + 16*hi,
//                    two exact operands (|.| <= 1920, and a multiple of 16 with
//                    |.| <= 4096), accumulated into the same block sum.
// Per 32-wide activation block one MMA group yields the exact integer block dot
// I (partial sums are integers below 2^24) in a TMEM slot. The epilogue applies
// the scales: per block acc += d_a * I (one packed FMA per two outputs), per
// super-block out += d * acc, and for q4_K out -= dmin * MS where
// MS = sum_j m_j * (d_a,j * s_j) comes from two small tf32 MMAs (the f32 factor
// d_a*s split into two tf32 parts; m_j is exact).
//
// Kernel structure (one persistent CTA per SM, 5 warpgroups, 640 threads):
//   warp 0      TMA producer: activation quants (2-D tensor map, 64 K per
//               stage), activation d and s planes (2-D, one super-block per
//               stage), weight rows (1-D bulk copies, one super-block per stage);
//   warp 1      MMA issuer (tcgen05.mma, one thread);
//   warp 2      TMEM allocator;
//   warps 4-7   A converters: int8 quants -> f16 operand tiles; q4_K min-term
//               activation operand;
//   warps 8-11  B converters: 4/6-bit quants (+ sub-block scales) -> f16
//               operand tiles, per-row super-block scales, q4_K min operand;
//   warps 12-19 epilogue: TMEM -> registers, scale, accumulate; the running
//               output tile lives in TMEM columns [0, 128).
// Operand tiles use the no-swizzle K-major layout (8 rows x 16 B core
// matrices). Within every group of 4 K positions both operands store the
// order (0, 2, 1, 3), which leaves every dot product unchanged.
// Every mbarrier wait is bounded; on timeout the kernel records an error,
// stops, drains its own copies and MMAs, frees TMEM and returns.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <mutex>

#include "mq_internal.cuh"
#include "tc.cuh"

namespace {

__device__ unsigned int g_gemm_error;   // bit 0: a bounded wait gave up

constexpr int BM = 128;                 // activation rows per tile (MMA M)
constexpr int BN = 128;                 // weight rows per tile (MMA N)
constexpr int RA = 4;                   // activation-quant stages (64 K each)
constexpr int RB = 2;                   // weight stages (one super-block each)
constexpr int RD = 2;                   // d/s plane stages (one super-block each)
constexpr int RF = 4;                   // converted operand slots (one 32-block each)
constexpr int RM = 2;                   // q4_K min-term operand slots
constexpr int RS = 2;                   // per-row super-block scale slots
constexpr int RT = 3;                   // TMEM accumulator slots (128 columns each)
constexpr int kThreads = 640;
constexpr int kLaunchRegs = 96;         // 65536 / 640, rounded down to the allocation unit
constexpr int kRegsWG0 = 48, kRegsConv = 80, kRegsEpi = 136;
static_assert(128 * kRegsWG0 + 256 * kRegsConv + 256 * kRegsEpi <= kThreads * kLaunchRegs, "register split");
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kLBO = 128;          // K-adjacent core matrices
constexpr uint32_t kSBO = 512;          // 8-row groups (4 core matrices per row group)
constexpr int kTile = 8192;             // 128 rows x 32 f16 (or 16 tf32)
constexpr int kARaw = BM * 64;          // two 32-blocks of int8 quants
constexpr int kDRaw = BM * 8 * 4;       // one super-block of d (or s)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOutCol = 0, kSlotCol0 = 128;

template <bool Q6>
struct Cfg {
    static constexpr int kSB = Q6 ? mq::Q6K_BYTES : mq::Q4K_BYTES;
    static constexpr int kBStride = Q6 ? 224 : 144;       // bytes per weight row in a stage
    static constexpr int kBRaw = BN * kBStride;
    static constexpr int kBTiles = Q6 ? 2 : 1;
    static constexpr int kFSlot = kTile * (1 + kBTiles);  // A tile, then B tile(s)
    static constexpr int kMS = Q6 ? 1 : RM;
};

template <bool Q6>
struct Smem {
    uint8_t f16[RF][Cfg<Q6>::kFSlot];
    uint8_t ms[Cfg<Q6>::kMS][Q6 ? 1024 : 2 * kTile];      // q4_K: A_ms tile, B_ms tile
    uint8_t araw[RA][kARaw];
    uint8_t draw[RD][2 * kDRaw];                           // d tile, then s tile
    uint8_t braw[RB][Cfg<Q6>::kBRaw];
    float wd[RS][BN];
    float wdmin[RS][BN];
    uint64_t fullA[RA], emptyA[RA], fullB[RB], emptyB[RB], fullD[RD], emptyD[RD];
    uint64_t fullF[RF], emptyF[RF], fullM[RM], emptyM[RM], fullS[RS], emptyS[RS];
    uint64_t tfull[RT], tempty[RT], mma_done;
    uint32_t tmem;
    int abort;
};

struct Ring {
    int i = 0;
    uint32_t ph = 0;
    __device__ __forceinline__ void next(int n) {
        if (++i == n) {
            i = 0;
            ph ^= 1u;
        }
    }
};

__device__ __forceinline__ uint32_t tile_off(int r, int kg) {
    return (uint32_t)((r >> 3) * kSBO + kg * kLBO + (r & 7) * 16);
}

template <bool Q6>
__device__ __forceinline__ bool wait_or_abort(Smem<Q6>& sm, uint64_t* bar, uint32_t parity) {
    if (tc::mbar_wait(bar, parity, kWaitLimitNs)) return true;
    atomicOr(&g_gemm_error, 1u);
    *(volatile int*)&sm.abort = 1;
    return false;
}

template <bool Q6>
__device__ __forceinline__ bool aborted(Smem<Q6>& sm) {
    return *(volatile int*)&sm.abort != 0;
}

// Whole-warp variants: every lane waits, and the outcome is made warp-uniform
// so that the warp never diverges in front of a warp-collective operation.
template <bool Q6>
__device__ __forceinline__ bool wwait(Smem<Q6>& sm, uint64_t* bar, uint32_t parity) {
    const bool ok = __all_sync(0xffffffffu, tc::mbar_wait(bar, parity, kWaitLimitNs));
    if (!ok) {
        if ((threadIdx.x & 31) == 0) atomicOr(&g_gemm_error, 1u);
        *(volatile int*)&sm.abort = 1;
    }
    return ok;
}

template <bool Q6>
__device__ __forceinline__ bool waborted(Smem<Q6>& sm) {
    return __any_sync(0xffffffffu, aborted(sm));
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Four int8 quants (one word, K positions 0..3) -> two f16x2 words holding
// positions (0, 2) and (1, 3). Byte b of a quant q is biased to q + 128 and
// placed in the mantissa of 1024.0, then 1152 is subtracted (exact).
__device__ __forceinline__ void a_word_to_f16(uint32_t w, uint32_t& p02, uint32_t& p13) {
    const __half2 bias = __floats2half2_rn(-1152.0f, -1152.0f);
    const uint32_t x02 = (w & 0x00FF00FFu) ^ 0x64806480u;
    const uint32_t x13 = ((w >> 8) & 0x00FF00FFu) ^ 0x64806480u;
    p02 = h2_bits(__hadd2(bits_h2(x02), bias));
    p13 = h2_bits(__hadd2(bits_h2(x13), bias));
}

// q4_K: four 4-bit quants in the low nibble of each byte of `nib` (bytes 0..3 =
// K positions 0..3) -> f16 pairs (0, 2), (1, 3) of sc * q.
// (1024 + q) * sc - 1024 * sc = sc * q exactly (|1024 sc| <= 64512 fits in f16).
__device__ __forceinline__ void q4_word_to_f16(uint32_t nib, __half2 sc2, __half2 nbias2, uint32_t& p02,
                                               uint32_t& p13) {
    const uint32_t x02 = (nib & 0x000F000Fu) | 0x64006400u;
    const uint32_t x13 = ((nib >> 8) & 0x000F000Fu) | 0x64006400u;
    p02 = h2_bits(__hfma2(bits_h2(x02), sc2, nbias2));
    p13 = h2_bits(__hfma2(bits_h2(x13), sc2, nbias2));
}

// q6_K: four values v (0..15 for the low part, 0..3 for the high part) in
// bits [0,4) of each byte of `v4` -> f16 pairs of mul * v + add, built as
// (1 + v/16) * (16 mul) - 16 mul + add so that no intermediate overflows f16.
__device__ __forceinline__ void small_word_to_f16(uint32_t v4, __half2 mul16, __half2 add2, uint32_t& p02,
                                                  uint32_t& p13) {
    const uint32_t x02 = ((v4 & 0x000F000Fu) << 6) | 0x3C003C00u;
    const uint32_t x13 = ((v4 >> 2) & 0x03C003C0u) | 0x3C003C00u;
    p02 = h2_bits(__hfma2(bits_h2(x02), mul16, add2));
    p13 = h2_bits(__hfma2(bits_h2(x13), mul16, add2));
}

// Two little-endian words starting at a 2-byte aligned shared-memory address.
__device__ __forceinline__ void lds8_unaligned(const uint8_t* p, uint32_t& w0, uint32_t& w1) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~(uintptr_t)3);
    const uint32_t sh = (uint32_t)(a & 3) * 8;
    const uint32_t v0 = w[0], v1 = w[1], v2 = w[2];
    w0 = __funnelshift_r(v0, v1, sh);
    w1 = __funnelshift_r(v1, v2, sh);
}

template <bool Q6>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                                                           const __grid_constant__ CUtensorMap tmD,
                                                           const __grid_constant__ CUtensorMap tmS,
                                                           const uint8_t* __restrict__ W, float* __restrict__ out,
                                                           int M, int N, int K, unsigned long long wstride,
                                                           unsigned long long wtotal) {
    using C = Cfg<Q6>;
    extern __shared__ uint8_t smem_raw[];
    Smem<Q6>& sm = *reinterpret_cast<Smem<Q6>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = K / mq::QK_K;
    const int num_mt = (M + BM - 1) / BM, num_nt = (N + BN - 1) / BN;
    const int tiles = num_mt * num_nt;

    if (tid == 0) {
        for (int i = 0; i < RA; ++i) { tc::mbar_init(&sm.fullA[i], 1); tc::mbar_init(&sm.emptyA[i], 4); }
        for (int i = 0; i < RB; ++i) { tc::mbar_init(&sm.fullB[i], 1); tc::mbar_init(&sm.emptyB[i], 4); }
        for (int i = 0; i < RD; ++i) { tc::mbar_init(&sm.fullD[i], 1); tc::mbar_init(&sm.emptyD[i], Q6 ? 8 : 12); }
        for (int i = 0; i < RF; ++i) { tc::mbar_init(&sm.fullF[i], 8); tc::mbar_init(&sm.emptyF[i], 1); }
        for (int i = 0; i < RM; ++i) { tc::mbar_init(&sm.fullM[i], 8); tc::mbar_init(&sm.emptyM[i], 1); }
        for (int i = 0; i < RS; ++i) { tc::mbar_init(&sm.fullS[i], 4); tc::mbar_init(&sm.emptyS[i], 8); }
        for (int i = 0; i < RT; ++i) { tc::mbar_init(&sm.tfull[i], 1); tc::mbar_init(&sm.tempty[i], 8); }
        tc::mbar_init(&sm.mma_done, 1);
        sm.abort = 0;
        tc::fence_mbar_init();
    }
    if (warp == 2) tc::tmem_alloc(&sm.tmem, kTmemCols);
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tbase = sm.tmem;

    if (warp < 4) {
        // ============================================================ warpgroup 0
        tc::setmaxnreg_dec<kRegsWG0>();
        if (warp == 0) {
            // ---------------------------------------------------- TMA producer
            Ring ra, rb, rd;
            int issA[RA], issB[RB], issD[RD];
            uint32_t phA[RA], phB[RB], phD[RD];
            for (int i = 0; i < RA; ++i) issA[i] = 0;
            for (int i = 0; i < RB; ++i) issB[i] = 0;
            for (int i = 0; i < RD; ++i) issD[i] = 0;
            const unsigned long long wend16 = wtotal & ~15ull;
            for (int t = blockIdx.x; t < tiles && !waborted(sm); t += gridDim.x) {
                const int m0 = (t % num_mt) * BM, n0 = (t / num_mt) * BN;
                for (int sb = 0; sb < S && !waborted(sm); ++sb) {
                    // activation d and s of this super-block
                    if (lane == 0 && wait_or_abort(sm, &sm.emptyD[rd.i], rd.ph ^ 1u)) {
                        tc::mbar_arrive_expect_tx(&sm.fullD[rd.i], 2 * kDRaw);
                        tc::tma_load_2d(sm.draw[rd.i], &tmD, sb * 8, m0, &sm.fullD[rd.i]);
                        tc::tma_load_2d(sm.draw[rd.i] + kDRaw, &tmS, sb * 8, m0, &sm.fullD[rd.i]);
                        issD[rd.i] = 1;
                        phD[rd.i] = rd.ph;
                    }
                    rd.next(RD);
                    // weight rows n0..n0+127 of this super-block
                    bool ok = true;
                    if (lane == 0) ok = wait_or_abort(sm, &sm.emptyB[rb.i], rb.ph ^ 1u);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok || waborted(sm)) break;
                    uint32_t bytes = 0;
                    uint8_t* stage = sm.braw[rb.i];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int r = lane + 32 * k, n = n0 + r;
                        if (n < N) {
                            const unsigned long long start = (unsigned long long)n * wstride + (unsigned long long)sb * C::kSB;
                            const unsigned long long a0 = start & ~15ull;
                            unsigned long long sz = Q6 ? 224ull : 144ull;
                            if (a0 + sz > wend16) {   // only the last bytes of the buffer
                                sz = wend16 - a0;
                                for (unsigned long long b = wend16; b < start + C::kSB; ++b)
                                    stage[r * C::kBStride + (b - a0)] = W[b];
                            }
                            bytes += (uint32_t)sz;
                        }
                    }
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, off);
                    __syncwarp();
                    if (lane == 0) {
                        tc::mbar_arrive_expect_tx(&sm.fullB[rb.i], bytes);
                        issB[rb.i] = 1;
                        phB[rb.i] = rb.ph;
                    }
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int r = lane + 32 * k, n = n0 + r;
                        if (n < N) {
                            const unsigned long long start = (unsigned long long)n * wstride + (unsigned long long)sb * C::kSB;
                            const unsigned long long a0 = start & ~15ull;
                            unsigned long long sz = Q6 ? 224ull : 144ull;
                            if (a0 + sz > wend16) sz = wend16 - a0;
                            if (sz) tc::bulk_load(stage + r * C::kBStride, W + a0, (uint32_t)sz, &sm.fullB[rb.i]);
                        }
                    }
                    rb.next(RB);
                    // activation quants, four stages of 64 K
                    for (int a = 0; a < 4; ++a) {
                        if (lane == 0 && wait_or_abort(sm, &sm.emptyA[ra.i], ra.ph ^ 1u)) {
                            tc::mbar_arrive_expect_tx(&sm.fullA[ra.i], kARaw);
                            tc::tma_load_2d(sm.araw[ra.i], &tmA, sb * 256 + a * 64, m0, &sm.fullA[ra.i]);
                            issA[ra.i] = 1;
                            phA[ra.i] = ra.ph;
                        }
                        ra.next(RA);
                    }
                }
            }
            if (aborted(sm) && lane == 0) {   // let every copy already issued land before the CTA exits
                for (int i = 0; i < RA; ++i) if (issA[i]) tc::mbar_wait(&sm.fullA[i], phA[i], kWaitLimitNs);
                for (int i = 0; i < RB; ++i) if (issB[i]) tc::mbar_wait(&sm.fullB[i], phB[i], kWaitLimitNs);
                for (int i = 0; i < RD; ++i) if (issD[i]) tc::mbar_wait(&sm.fullD[i], phD[i], kWaitLimitNs);
            }
        } else if (warp == 1) {
            // ---------------------------------------------------- MMA issuer
            if (lane == 0) {
                Ring rf, rm, rt;
                const uint32_t idesc = tc::instr_desc(BM, BN, 0);
                const uint32_t idesc32 = tc::instr_desc(BM, BN, 2);
                bool issued = false;
                for (int t = blockIdx.x; t < tiles && !aborted(sm); t += gridDim.x) {
                    for (int sb = 0; sb < S && !aborted(sm); ++sb) {
                        for (int j = 0; j < 8; ++j) {
                            if (!wait_or_abort(sm, &sm.fullF[rf.i], rf.ph)) break;
                            if (!wait_or_abort(sm, &sm.tempty[rt.i], rt.ph ^ 1u)) break;
                            tc::tc_fence_after();
                            const uint32_t d = tbase + kSlotCol0 + 128u * rt.i;
                            const uint32_t sa = tc::smem_u32(sm.f16[rf.i]);
#pragma unroll
                            for (int part = 0; part < C::kBTiles; ++part) {
                                const uint32_t sbb = sa + kTile * (1 + part);
#pragma unroll
                                for (int k = 0; k < 2; ++k)
                                    tc::mma_f16(d, tc::smem_desc_noswizzle(sa + k * 2 * kLBO, kLBO, kSBO),
                                                tc::smem_desc_noswizzle(sbb + k * 2 * kLBO, kLBO, kSBO), idesc,
                                                (part | k) ? 1u : 0u);
                            }
                            tc::mma_commit(&sm.emptyF[rf.i]);
                            tc::mma_commit(&sm.tfull[rt.i]);
                            issued = true;
                            rf.next(RF);
                            rt.next(RT);
                        }
                        if constexpr (!Q6) {
                            if (aborted(sm)) break;
                            if (!wait_or_abort(sm, &sm.fullM[rm.i], rm.ph)) break;
                            if (!wait_or_abort(sm, &sm.tempty[rt.i], rt.ph ^ 1u)) break;
                            tc::tc_fence_after();
                            const uint32_t d = tbase + kSlotCol0 + 128u * rt.i;
                            const uint32_t sa = tc::smem_u32(sm.ms[rm.i]);
#pragma unroll
                            for (int k = 0; k < 2; ++k)
                                tc::mma_tf32(d, tc::smem_desc_noswizzle(sa + k * 2 * kLBO, kLBO, kSBO),
                                             tc::smem_desc_noswizzle(sa + kTile + k * 2 * kLBO, kLBO, kSBO), idesc32,
                                             k ? 1u : 0u);
                            tc::mma_commit(&sm.emptyM[rm.i]);
                            tc::mma_commit(&sm.tfull[rt.i]);
                            rm.next(RM);
                            rt.next(RT);
                        }
                    }
                }
                if (issued) {   // every MMA of this CTA has completed before TMEM is freed
                    tc::mma_commit(&sm.mma_done);
                    tc::mbar_wait(&sm.mma_done, 0, kWaitLimitNs);
                }
                tc::tc_fence_before();
            }
            __syncwarp();
        }
    } else if (warp < 8) {
        // ============================================================ A converters
        tc::setmaxnreg_dec<kRegsConv>();
        const int t = tid - 128;
        Ring ra, rd, rf, rm;
        for (int tt = blockIdx.x; tt < tiles && !waborted(sm); tt += gridDim.x) {
            for (int sb = 0; sb < S && !waborted(sm); ++sb) {
                if constexpr (!Q6) {
                    // min-term operand: row t, K' = j (hi part of d_a,j * s_j) and 8 + j (lo part)
                    if (!wwait(sm, &sm.fullD[rd.i], rd.ph)) break;
                    if (!wwait(sm, &sm.emptyM[rm.i], rm.ph ^ 1u)) break;
                    const float* drow = reinterpret_cast<const float*>(sm.draw[rd.i]) + t * 8;
                    const int* srow = reinterpret_cast<const int*>(sm.draw[rd.i] + kDRaw) + t * 8;
                    float hi[8], lo[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float beta = drow[j] * (float)srow[j];
                        hi[j] = __uint_as_float(__float_as_uint(beta) & 0xFFFFE000u);
                        lo[j] = beta - hi[j];
                    }
                    uint8_t* tile = sm.ms[rm.i];
                    *reinterpret_cast<float4*>(tile + tile_off(t, 0)) = make_float4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<float4*>(tile + tile_off(t, 1)) = make_float4(hi[4], hi[5], hi[6], hi[7]);
                    *reinterpret_cast<float4*>(tile + tile_off(t, 2)) = make_float4(lo[0], lo[1], lo[2], lo[3]);
                    *reinterpret_cast<float4*>(tile + tile_off(t, 3)) = make_float4(lo[4], lo[5], lo[6], lo[7]);
                    tc::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tc::mbar_arrive(&sm.fullM[rm.i]);
                        tc::mbar_arrive(&sm.emptyD[rd.i]);
                    }
                    rd.next(RD);
                    rm.next(RM);
                }
                for (int a = 0; a < 4; ++a) {
                    if (!wwait(sm, &sm.fullA[ra.i], ra.ph)) break;
                    const int f0 = rf.i;
                    if (!wwait(sm, &sm.emptyF[rf.i], rf.ph ^ 1u)) break;
                    rf.next(RF);
                    const int f1 = rf.i;
                    if (!wwait(sm, &sm.emptyF[rf.i], rf.ph ^ 1u)) break;
                    rf.next(RF);
                    const uint8_t* raw = sm.araw[ra.i];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int q = i * 128 + t;           // 16-byte chunk of the 128 x 64 B stage
                        const int r = q >> 2, c = q & 3;
                        const uint4 v = *reinterpret_cast<const uint4*>(raw + q * 16);
                        uint8_t* tile = sm.f16[(c >> 1) ? f1 : f0];
                        uint4 o0, o1;
                        a_word_to_f16(v.x, o0.x, o0.y);
                        a_word_to_f16(v.y, o0.z, o0.w);
                        a_word_to_f16(v.z, o1.x, o1.y);
                        a_word_to_f16(v.w, o1.z, o1.w);
                        *reinterpret_cast<uint4*>(tile + tile_off(r, 2 * (c & 1))) = o0;
                        *reinterpret_cast<uint4*>(tile + tile_off(r, 2 * (c & 1) + 1)) = o1;
                    }
                    tc::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tc::mbar_arrive(&sm.fullF[f0]);
                        tc::mbar_arrive(&sm.fullF[f1]);
                        tc::mbar_arrive(&sm.emptyA[ra.i]);
                    }
                    ra.next(RA);
                }
            }
        }
    } else if (warp < 12) {
        // ============================================================ B converters
        tc::setmaxnreg_dec<kRegsConv>();
        const int t = tid - 256;
        const int c = t & 3;                    // 8-position part of a 32-block
        Ring rb, rf, rm, rs;
        for (int tt = blockIdx.x; tt < tiles && !waborted(sm); tt += gridDim.x) {
            const int n0 = (tt / num_mt) * BN;
            for (int sb = 0; sb < S && !waborted(sm); ++sb) {
                if (!wwait(sm, &sm.fullB[rb.i], rb.ph)) break;
                if (!wwait(sm, &sm.emptyS[rs.i], rs.ph ^ 1u)) break;
                if (!Q6 && !wwait(sm, &sm.emptyM[rm.i], rm.ph ^ 1u)) break;
                const uint8_t* stage = sm.braw[rb.i];
                int delta[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int r = 32 * k + (t >> 2), n = n0 + r;
                    delta[k] = Q6 ? (int)(((unsigned long long)n * wstride + (unsigned long long)sb * C::kSB) & 15ull) : 0;
                    const uint8_t* blk = stage + r * C::kBStride + delta[k];
                    const bool valid = n < N;
                    if constexpr (Q6) {
                        if (c == 0) {
                            sm.wd[rs.i][r] = valid ? __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(blk + 208))) : 0.0f;
                        }
                    } else {
                        uint32_t s0 = 0, s1 = 0, s2 = 0;
                        if (valid) {
                            const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
                            s0 = hdr.y; s1 = hdr.z; s2 = hdr.w;
                            if (c == 0) {
                                sm.wd[rs.i][r] = __half2float(__ushort_as_half((unsigned short)(hdr.x & 0xffffu)));
                                sm.wdmin[rs.i][r] = __half2float(__ushort_as_half((unsigned short)(hdr.x >> 16)));
                            }
                        } else if (c == 0) {
                            sm.wd[rs.i][r] = 0.0f;
                            sm.wdmin[rs.i][r] = 0.0f;
                        }
                        // mins of sub-blocks 4*(c&1) .. 4*(c&1)+3 -> K' positions 4c .. 4c+3 of B_ms
                        float mv[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int j = 4 * (c & 1) + u;
                            const uint32_t bj4 = (j < 4) ? ((s1 >> (8 * j)) & 0xffu) : ((s2 >> (8 * (j - 4))) & 0xffu);
                            const uint32_t hbits = (j < 4) ? 0u : (((j < 4 ? 0u : ((s1 >> (8 * (j - 4))) & 0xffu)) >> 6) << 4);
                            const uint32_t m = (j < 4) ? (bj4 & 63u) : ((bj4 >> 4) | hbits);
                            mv[u] = (float)m;
                        }
                        *reinterpret_cast<float4*>(sm.ms[rm.i] + kTile + tile_off(r, c)) = make_float4(mv[0], mv[1], mv[2], mv[3]);
                    }
                }
                if (!Q6) tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tc::mbar_arrive(&sm.fullS[rs.i]);
                    if (!Q6) tc::mbar_arrive(&sm.fullM[rm.i]);
                }
                rs.next(RS);
                if (!Q6) rm.next(RM);

                for (int P = 0; P < 4 && !waborted(sm); ++P) {
                    const int f0 = rf.i;
                    if (!wwait(sm, &sm.emptyF[rf.i], rf.ph ^ 1u)) break;
                    rf.next(RF);
                    const int f1 = rf.i;
                    if (!wwait(sm, &sm.emptyF[rf.i], rf.ph ^ 1u)) break;
                    rf.next(RF);
                    uint8_t* b0 = sm.f16[f0] + kTile;
                    uint8_t* b1 = sm.f16[f1] + kTile;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int r = 32 * k + (t >> 2), n = n0 + r;
                        const uint8_t* blk = stage + r * C::kBStride + delta[k];
                        uint4 o0 = make_uint4(0, 0, 0, 0), o1 = o0, o2 = o0, o3 = o0;
                        if (n < N) {
                            if constexpr (!Q6) {
                                // sub-blocks 2P (low nibbles) and 2P+1 (high nibbles), positions 8c..8c+7
                                const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
                                int sc[2];
#pragma unroll
                                for (int u = 0; u < 2; ++u) {
                                    const int j = 2 * P + u;
                                    const uint32_t bj = (j < 4) ? ((hdr.y >> (8 * j)) & 0xffu) : ((hdr.w >> (8 * (j - 4))) & 0xffu);
                                    const uint32_t bjm4 = (j < 4) ? 0u : ((hdr.y >> (8 * (j - 4))) & 0xffu);
                                    sc[u] = (j < 4) ? (int)(bj & 63u) : (int)((bj & 15u) | ((bjm4 >> 6) << 4));
                                }
                                const uint2 q = *reinterpret_cast<const uint2*>(blk + 16 + 32 * P + 8 * c);
                                const __half2 s0 = __float2half2_rn((float)sc[0]), s1 = __float2half2_rn((float)sc[1]);
                                const __half2 nb0 = __float2half2_rn(-1024.0f * sc[0]), nb1 = __float2half2_rn(-1024.0f * sc[1]);
                                q4_word_to_f16(q.x, s0, nb0, o0.x, o0.y);
                                q4_word_to_f16(q.y, s0, nb0, o0.z, o0.w);
                                q4_word_to_f16(q.x >> 4, s1, nb1, o1.x, o1.y);
                                q4_word_to_f16(q.y >> 4, s1, nb1, o1.z, o1.w);
                            } else {
                                // blocks 2P, 2P+1: half h, quarters tq0 = 2(P&1), tq0+1
                                const int h = P >> 1, tq0 = 2 * (P & 1);
                                uint32_t l0a, l0b, l1a, l1b, qa, qb;
                                lds8_unaligned(blk + 64 * h + 8 * c, l0a, l0b);
                                lds8_unaligned(blk + 64 * h + 32 + 8 * c, l1a, l1b);
                                lds8_unaligned(blk + 128 + 32 * h + 8 * c, qa, qb);
                                const int nsh = (P & 1) ? 4 : 0;   // low nibbles for quarters 0, 1
                                const int sc0 = (int)(int8_t)blk[192 + 4 * P + (c >> 1)];
                                const int sc1 = (int)(int8_t)blk[192 + 4 * P + 2 + (c >> 1)];
                                const __half2 m0 = __float2half2_rn(16.0f * sc0), a0 = __float2half2_rn(-16.0f * sc0);
                                const __half2 m1 = __float2half2_rn(16.0f * sc1), a1 = __float2half2_rn(-16.0f * sc1);
                                const __half2 hm0 = __float2half2_rn(256.0f * sc0), ha0 = __float2half2_rn(-288.0f * sc0);
                                const __half2 hm1 = __float2half2_rn(256.0f * sc1), ha1 = __float2half2_rn(-288.0f * sc1);
                                const uint32_t m4 = 0x0F0F0F0Fu, m2 = 0x03030303u;
                                // block 2P: B1 = sc*lo -> o0, B2 = 16 sc (hi-2) -> o1
                                small_word_to_f16((l0a >> nsh) & m4, m0, a0, o0.x, o0.y);
                                small_word_to_f16((l0b >> nsh) & m4, m0, a0, o0.z, o0.w);
                                small_word_to_f16((qa >> (2 * tq0)) & m2, hm0, ha0, o1.x, o1.y);
                                small_word_to_f16((qb >> (2 * tq0)) & m2, hm0, ha0, o1.z, o1.w);
                                // block 2P+1 -> o2, o3
                                small_word_to_f16((l1a >> nsh) & m4, m1, a1, o2.x, o2.y);
                                small_word_to_f16((l1b >> nsh) & m4, m1, a1, o2.z, o2.w);
                                small_word_to_f16((qa >> (2 * tq0 + 2)) & m2, hm1, ha1, o3.x, o3.y);
                                small_word_to_f16((qb >> (2 * tq0 + 2)) & m2, hm1, ha1, o3.z, o3.w);
                            }
                        }
                        if (!Q6) {
                            *reinterpret_cast<uint4*>(b0 + tile_off(r, c)) = o0;
                            *reinterpret_cast<uint4*>(b1 + tile_off(r, c)) = o1;
                        } else {
                            *reinterpret_cast<uint4*>(b0 + tile_off(r, c)) = o0;
                            *reinterpret_cast<uint4*>(b0 + kTile + tile_off(r, c)) = o1;
                            *reinterpret_cast<uint4*>(b1 + tile_off(r, c)) = o2;
                            *reinterpret_cast<uint4*>(b1 + kTile + tile_off(r, c)) = o3;
                        }
                    }
                    tc::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tc::mbar_arrive(&sm.fullF[f0]);
                        tc::mbar_arrive(&sm.fullF[f1]);
                    }
                }
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&sm.emptyB[rb.i]);
                rb.next(RB);
            }
        }
    } else {
        // ============================================================ epilogue
        tc::setmaxnreg_inc<kRegsEpi>();
        const int q = warp & 3;                 // TMEM lane quarter
        const int ch = (warp - 12) >> 2;        // column half: 64 * ch .. 64 * ch + 63
        const int rloc = 32 * q + lane;
        const uint32_t lane_bits = (uint32_t)(32 * q) << 16;
        Ring rd, rt, rs;
        for (int tt = blockIdx.x; tt < tiles && !waborted(sm); tt += gridDim.x) {
            const int m0 = (tt % num_mt) * BM, n0 = (tt / num_mt) * BN;
            const int m = m0 + rloc;
            for (int sb = 0; sb < S && !waborted(sm); ++sb) {
                if (!wwait(sm, &sm.fullD[rd.i], rd.ph)) break;
                float da[8];
                {
                    const float4* dp = reinterpret_cast<const float4*>(sm.draw[rd.i] + rloc * 32);
                    const float4 x0 = dp[0], x1 = dp[1];
                    da[0] = x0.x; da[1] = x0.y; da[2] = x0.z; da[3] = x0.w;
                    da[4] = x1.x; da[5] = x1.y; da[6] = x1.z; da[7] = x1.w;
                }
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&sm.emptyD[rd.i]);
                rd.next(RD);

                float2 acc[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) acc[c] = make_float2(0.0f, 0.0f);
                bool ok = true;
#pragma unroll 1
                for (int j = 0; j < 8; ++j) {
                    if (!wwait(sm, &sm.tfull[rt.i], rt.ph)) { ok = false; break; }
                    tc::tc_fence_after();
                    const uint32_t ta = tbase + lane_bits + kSlotCol0 + 128u * rt.i + 64u * ch;
                    const float2 d2 = make_float2(da[j], da[j]);
                    uint32_t I[32];
                    tc::tmem_ld32(ta, I);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        acc[c] = tc::ffma2(d2, make_float2(__uint_as_float(I[2 * c]), __uint_as_float(I[2 * c + 1])), acc[c]);
                    tc::tmem_ld32(ta + 32, I);
                    tc::tmem_ld_wait();
                    tc::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&sm.tempty[rt.i]);
                    rt.next(RT);
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        acc[16 + c] = tc::ffma2(d2, make_float2(__uint_as_float(I[2 * c]), __uint_as_float(I[2 * c + 1])), acc[16 + c]);
                }
                if (!ok) break;
                uint32_t ms_slot = 0;
                if (!Q6) {
                    if (!wwait(sm, &sm.tfull[rt.i], rt.ph)) break;
                    tc::tc_fence_after();
                    ms_slot = kSlotCol0 + 128u * rt.i;
                }
                if (!wwait(sm, &sm.fullS[rs.i], rs.ph)) break;
                const bool last = (sb == S - 1);
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const int col = 64 * ch + 16 * h;
                    uint32_t o[16], mv[16];
                    if (sb > 0) tc::tmem_ld16(tbase + lane_bits + kOutCol + col, o);
                    if (!Q6) tc::tmem_ld16(tbase + lane_bits + ms_slot + col, mv);
                    tc::tmem_ld_wait();
                    const float4* wdp = reinterpret_cast<const float4*>(&sm.wd[rs.i][col]);
                    const float4* wmp = reinterpret_cast<const float4*>(&sm.wdmin[rs.i][col]);
                    float res[16];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float4 wv = wdp[u];
                        const float w4[4] = {wv.x, wv.y, wv.z, wv.w};
                        float m4v[4] = {0.f, 0.f, 0.f, 0.f};
                        if (!Q6) {
                            const float4 mm = wmp[u];
                            m4v[0] = mm.x; m4v[1] = mm.y; m4v[2] = mm.z; m4v[3] = mm.w;
                        }
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int cc = 4 * u + e;                 // 0..15 within the chunk
                            const int ai = 8 * h + (cc >> 1);         // float2 index in acc
                            const float av = (cc & 1) ? acc[ai].y : acc[ai].x;
                            float v = (sb > 0) ? __uint_as_float(o[cc]) : 0.0f;
                            v = fmaf(w4[e], av, v);
                            if (!Q6) v = fmaf(-m4v[e], __uint_as_float(mv[cc]), v);
                            res[cc] = v;
                        }
                    }
                    if (last) {
                        if (m < M) {
                            float* orow = out + (size_t)m * N + n0 + col;
                            if (n0 + col + 16 <= N && (N & 3) == 0) {
#pragma unroll
                                for (int u = 0; u < 4; ++u)
                                    reinterpret_cast<float4*>(orow)[u] = make_float4(res[4 * u], res[4 * u + 1], res[4 * u + 2], res[4 * u + 3]);
                            } else {
                                for (int u = 0; u < 16; ++u)
                                    if (n0 + col + u < N) orow[u] = res[u];
                            }
                        }
                    } else {
                        uint32_t ob[16];
#pragma unroll
                        for (int u = 0; u < 16; ++u) ob[u] = __float_as_uint(res[u]);
                        tc::tmem_st16(tbase + lane_bits + kOutCol + col, ob);
                    }
                }
                tc::tmem_st_wait();
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    tc::mbar_arrive(&sm.emptyS[rs.i]);
                    if (!Q6) tc::mbar_arrive(&sm.tempty[rt.i]);
                }
                rs.next(RS);
                if (!Q6) rt.next(RT);
            }
        }
    }

    __syncthreads();
    if (warp == 2) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tbase, kTmemCols);
    }
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool make_map(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
              uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
    const int M = a->M, K = a->K;
    // The register split between warpgroups assumes the launch register count.
    static int regs_ok = -1;
    if (regs_ok < 0) {
        cudaFuncAttributes fa;
        regs_ok = (cudaFuncGetAttributes(&fa, gemm_kernel<Q6>) == cudaSuccess && fa.numRegs == kLaunchRegs) ? 1 : 0;
    }
    if (!regs_ok) return MQ_ERR_LAUNCH;
    CUtensorMap tmA, tmD, tmS;
    if (!make_map(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, a->qs, (uint64_t)K, (uint64_t)M, (uint64_t)K, 64, BM) ||
        !make_map(&tmD, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a->d, (uint64_t)K / 32, (uint64_t)M, (uint64_t)K / 8, 8, BM) ||
        !make_map(&tmS, CU_TENSOR_MAP_DATA_TYPE_INT32, a->s, (uint64_t)K / 32, (uint64_t)M, (uint64_t)K / 8, 8, BM))
        return MQ_ERR_LAUNCH;
    const size_t smem = sizeof(Smem<Q6>) + 1024;
    if (cudaFuncSetAttribute(gemm_kernel<Q6>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return MQ_ERR_LAUNCH;
    const long long tiles = (long long)((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    const int grid = (int)(tiles < mq::num_sms() ? tiles : mq::num_sms());
    const unsigned long long row = (unsigned long long)(K / mq::QK_K) * Cfg<Q6>::kSB;
    gemm_kernel<Q6><<<grid, kThreads, smem, stream>>>(tmA, tmD, tmS, static_cast<const uint8_t*>(w), out, M, N, K,
                                                      row, row * (unsigned long long)N);
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
