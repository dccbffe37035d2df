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
//   A (activations): q_a in [-127, 127] — the plane's binary16 copy (qh),
//                    loaded by TMA straight into the MMA operand layout.
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
//   warp 0      TMA producer: activation f16 quants (2-D map, 64-byte swizzle,
//               one 32-block per operand slot), activation d and s planes
//               (2-D, one super-block per stage), weight rows (1-D bulk
//               copies, one super-block per stage);
//   warp 1      MMA issuer (tcgen05.mma, one thread);
//   warp 2      TMEM allocator;
//   warps 4-11  B converters: 4/6-bit quants (+ sub-block scales) -> f16
//               operand tiles, per-row super-block scales, q4_K min operand;
//   warps 12-19 epilogue: TMEM -> registers, scale, accumulate (each warp one
//               TMEM lane quarter x 64 columns); the running output tile lives
//               in TMEM columns [0, 128); q4_K min-term activation operand.
// Weight operand tiles use the no-swizzle K-major layout (8 rows x 16 B core
// matrices). Every mbarrier wait is bounded; on timeout the kernel records an
// error, stops, drains its own copies and MMAs, frees TMEM and returns.

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
constexpr int RB = 2;                   // weight stages (one super-block each)
constexpr int RD = 2;                   // d/s plane stages (one super-block each)
constexpr int RM = 2;                   // q4_K min-term operand slots
constexpr int RS = 2;                   // per-row super-block scale slots
constexpr int RT = 3;                   // TMEM accumulator slots (128 columns each)
constexpr int kConvWarps = 8;
constexpr int kConvRows = BN / (8 * kConvWarps);   // weight rows per converter thread
constexpr int kEpiWarps = 8;            // 2 per TMEM lane quarter, 64 columns each
constexpr int kThreads = 128 + 32 * kConvWarps + 32 * kEpiWarps;
constexpr int kLaunchRegs = 96;         // 65536 / 640, rounded down to the allocation unit
#ifndef MQ_REGS_OVERRIDE
constexpr int kRegsWG0 = 48, kRegsConv = 64, kRegsEpi = 152;   // measured best of the splits that fit
#else
constexpr int kRegsWG0 = MQ_R0, kRegsConv = MQ_RC, kRegsEpi = MQ_RE;
#endif
static_assert(128 * kRegsWG0 + 32 * kConvWarps * kRegsConv + 32 * kEpiWarps * kRegsEpi <= kThreads * kLaunchRegs,
              "register split");
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kLBO = 128;          // K-adjacent core matrices (no-swizzle tiles)
constexpr uint32_t kSBO = 512;          // 8-row groups
constexpr int kTile = 8192;             // 128 rows x 32 f16 (or 16 tf32)
constexpr int kDRaw = BM * 8 * 4;       // one super-block of d (or s)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOutCol = 0, kSlotCol0 = 128;

template <bool Q6>
struct Cfg {
    static constexpr int kSB = Q6 ? mq::Q6K_BYTES : mq::Q4K_BYTES;
    static constexpr int kBStride = Q6 ? 240 : 144;       // bytes per weight row in a stage (8 rows: distinct banks)
    static constexpr int kBRaw = BN * kBStride;
    static constexpr int kBTiles = Q6 ? 2 : 1;
    static constexpr int kFSlot = kTile * (1 + kBTiles);  // A tile, then B tile(s)
    static constexpr int RF = Q6 ? 5 : 6;                 // operand slots (one 32-block each)
    static constexpr int kMS = Q6 ? 1 : RM;
};

template <bool Q6>
struct Smem {
    uint8_t f16[Cfg<Q6>::RF][Cfg<Q6>::kFSlot];
    uint8_t ms[Cfg<Q6>::kMS][Q6 ? 1024 : 2 * kTile];      // q4_K: A_ms tile, B_ms tile
    uint8_t draw[RD][2 * kDRaw];                           // d tile, then s tile
    uint8_t braw[RB][Cfg<Q6>::kBRaw];
    uint2 scpack[Q6 ? 1 : BN][8];                          // q4_K: per row and sub-block {sc x2, -1024 sc x2} as f16
    float wd[RS][BN];
    float wdmin[RS][BN];
    uint64_t fullB[RB], emptyB[RB], fullD[RD], emptyD[RD];
    uint64_t fullF[Cfg<Q6>::RF], emptyF[Cfg<Q6>::RF], fullM[RM], emptyM[RM], fullS[RS], emptyS[RS];
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

// A work unit: one output tile and one slice [sb0, sb1) of its super-blocks. Tiles
// are numbered m-fastest; units that share a tile add their partial sums into the
// output, which the host zeroed beforehand.
//   q4_K: every tile is split into `splits` slices (1 unless there are fewer tiles
//         than SMs); unit u is slice u % splits of tile u / splits.
//   q6_K: the first `whole` units are whole tiles (full waves over the CTAs); each
//         tile of the last, partial wave is split into `splits` slices.
// (The q4_K kernel keeps the plain mapping: the same hybrid there measured slower
// through the code it makes, not through its schedule.)
struct Work {
    int m0, n0, sb0, sb1;
};
template <bool Q6>
__device__ __forceinline__ Work work_of(int u, int whole, int splits, int num_mt, int S) {
    if constexpr (!Q6) {
        const int t = u / splits, sp = u - t * splits;
        return Work{(t % num_mt) * BM, (t / num_mt) * BN, (sp * S) / splits, ((sp + 1) * S) / splits};
    } else {
        int t = u, sp = 0, ns = 1;
        if (u >= whole) {
            const int v = u - whole;
            t = whole + v / splits;
            sp = v - (t - whole) * splits;
            ns = splits;
        }
        return Work{(t % num_mt) * BM, (t / num_mt) * BN, (sp * S) / ns, ((sp + 1) * S) / ns};
    }
}

__device__ __forceinline__ uint32_t tile_off(int r, int kg) {
    return (uint32_t)((r >> 3) * kSBO + kg * kLBO + (r & 7) * 16);
}

// Non-suspending test of a phase (acquire semantics, like the waits). A phase that
// has already completed is seen sooner this way than by a suspending try_wait.
__device__ __forceinline__ bool mbar_ready(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok)
                 : "r"(tc::smem_u32(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

template <bool Q6>
__device__ __forceinline__ bool wait_or_abort(Smem<Q6>& sm, uint64_t* bar, uint32_t parity) {
    if (mbar_ready(bar, parity) || tc::mbar_wait(bar, parity, kWaitLimitNs)) return true;
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
    const bool ok = __all_sync(0xffffffffu, mbar_ready(bar, parity) || tc::mbar_wait(bar, parity, kWaitLimitNs));
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

// f16 bit pattern of a small integer (|v| <= 2048, exact), replicated in both halves.
__device__ __forceinline__ uint32_t h2_of_int(int v) {
    const uint32_t h = (uint32_t)__half_as_ushort(__int2half_rn(v));
    return h | (h << 16);
}

// Four 4-bit values in the low nibble of each byte of `x` (byte i = K position
// i) -> f16 pairs (0, 1), (2, 3) of mul * v + add. The value v is placed in the
// mantissa of 1024.0 (1024 + v), so mul * v + add with add = -1024 * mul gives
// mul * v exactly for the q4_K range (|1024 * sc| <= 64512 fits in f16).
__device__ __forceinline__ void nib4_to_f16_1024(uint32_t x, uint32_t mul2, uint32_t add2, uint32_t& p01,
                                                 uint32_t& p23) {
    p01 = tc::hfma2(tc::prmt(x, 0x64u, 0x4140u), mul2, add2);
    p23 = tc::hfma2(tc::prmt(x, 0x64u, 0x4342u), mul2, add2);
}

// Same for q6_K, where the multipliers reach 16 * 128: v (0..15) is placed as
// 1 + v/16, and mul16 = 16 * mul, add = -16 * mul + offset never overflow f16.
__device__ __forceinline__ void nib4_to_f16_one(uint32_t x, uint32_t mul16, uint32_t add2, uint32_t& p01,
                                                uint32_t& p23) {
    const uint32_t t01 = (tc::prmt(x, 0u, 0x4140u) << 6) | 0x3C003C00u;
    const uint32_t t23 = (tc::prmt(x, 0u, 0x4342u) << 6) | 0x3C003C00u;
    p01 = tc::hfma2(t01, mul16, add2);
    p23 = tc::hfma2(t23, mul16, add2);
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

__device__ __forceinline__ uint32_t byte_at(uint32_t w0, uint32_t w1, uint32_t w2, int i) {
    const uint32_t w = (i < 4) ? w0 : (i < 8 ? w1 : w2);
    return (w >> (8 * (i & 3))) & 0xffu;
}

// q6_K weight rows are only 2-byte aligned, so they are staged by the converter
// threads themselves: for each of its rows, part c of the 4 threads sharing a
// row copies 16-byte chunks c, c+4, ... of the aligned window that holds the
// row's 210-byte super-block (chunk copies never cross the last 16-byte
// boundary of the buffer; the few bytes past it are copied one by one).
// The copies form one commit group per super-block.
__device__ __forceinline__ void q6_fetch(uint8_t* stage, const uint8_t* __restrict__ W, int n0, int sb, int N,
                                         unsigned long long wstride, unsigned long long wtotal, int rbase, int c) {
    const unsigned long long wend16 = wtotal & ~15ull;
#pragma unroll
    for (int k = 0; k < kConvRows; ++k) {
        const int r = 8 * kConvWarps * k + rbase, n = n0 + r;
        if (n < N) {
            const unsigned long long start = (unsigned long long)n * wstride + (unsigned long long)sb * mq::Q6K_BYTES;
            const unsigned long long a0 = start & ~15ull, end = start + mq::Q6K_BYTES;
            uint8_t* dst = stage + r * Cfg<true>::kBStride;
            for (int ch = c; ch < 14; ch += 4) {
                const unsigned long long src = a0 + 16ull * ch;
                if (src >= end) break;
                if (src + 16 <= wend16) {
                    tc::cp_async16(dst + 16 * ch, W + src);
                } else {
                    for (unsigned long long b = src; b < end; ++b) dst[b - a0] = W[b];
                }
            }
        }
    }
    tc::cp_async_commit();
}

template <bool Q6>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                                                           const __grid_constant__ CUtensorMap tmD,
                                                           const __grid_constant__ CUtensorMap tmS,
                                                           const __grid_constant__ CUtensorMap tmW,
                                                           const uint8_t* __restrict__ W, float* __restrict__ out,
                                                           int M, int N, int K, int whole, int splits,
                                                           unsigned long long wstride, unsigned long long wtotal) {
    using C = Cfg<Q6>;
    constexpr int RF = C::RF;
    extern __shared__ uint8_t smem_raw[];
    Smem<Q6>& sm = *reinterpret_cast<Smem<Q6>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = K / mq::QK_K;
    const int num_mt = (M + BM - 1) / BM, num_nt = (N + BN - 1) / BN;
    const int units = Q6 ? whole + (num_mt * num_nt - whole) * splits : num_mt * num_nt * splits;

    if (tid == 0) {
        for (int i = 0; i < RB; ++i) { tc::mbar_init(&sm.fullB[i], 1); tc::mbar_init(&sm.emptyB[i], kConvWarps); }
        for (int i = 0; i < RD; ++i) { tc::mbar_init(&sm.fullD[i], 1); tc::mbar_init(&sm.emptyD[i], kEpiWarps); }
        for (int i = 0; i < RF; ++i) { tc::mbar_init(&sm.fullF[i], 1 + kConvWarps); tc::mbar_init(&sm.emptyF[i], 1); }
        for (int i = 0; i < RM; ++i) { tc::mbar_init(&sm.fullM[i], 4 + kConvWarps); tc::mbar_init(&sm.emptyM[i], 1); }
        for (int i = 0; i < RS; ++i) { tc::mbar_init(&sm.fullS[i], kConvWarps); tc::mbar_init(&sm.emptyS[i], kEpiWarps); }
        for (int i = 0; i < RT; ++i) { tc::mbar_init(&sm.tfull[i], 1); tc::mbar_init(&sm.tempty[i], kEpiWarps); }
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
            Ring rb, rd, rf;
            uint32_t issB = 0, issD = 0, issF = 0;        // bit i: stage i has a copy in flight
            uint32_t phB = 0, phD = 0, phF = 0;           // bit i: parity of that copy
            for (int u = blockIdx.x; u < units && !waborted(sm); u += gridDim.x) {
                const Work wk = work_of<Q6>(u, whole, splits, num_mt, S);
                const int m0 = wk.m0, n0 = wk.n0;
                for (int sb = wk.sb0; sb < wk.sb1 && !waborted(sm); ++sb) {
                    // activation d and s of this super-block
                    if (lane == 0 && wait_or_abort(sm, &sm.emptyD[rd.i], rd.ph ^ 1u)) {
                        tc::mbar_arrive_expect_tx(&sm.fullD[rd.i], 2 * kDRaw);
                        tc::tma_load_2d(sm.draw[rd.i], &tmD, sb * 8, m0, &sm.fullD[rd.i]);
                        tc::tma_load_2d(sm.draw[rd.i] + kDRaw, &tmS, sb * 8, m0, &sm.fullD[rd.i]);
                        issD |= 1u << rd.i;
                        phD = (phD & ~(1u << rd.i)) | (rd.ph << rd.i);
                    }
                    rd.next(RD);
                    // q4_K weight rows n0..n0+127 of this super-block: one 2-D copy (rows >= N read as zeros).
                    // q6_K rows are only 2-byte aligned; the converters fetch them themselves.
                    if constexpr (!Q6) {
                        if (lane == 0 && wait_or_abort(sm, &sm.emptyB[rb.i], rb.ph ^ 1u)) {
                            tc::mbar_arrive_expect_tx(&sm.fullB[rb.i], C::kBRaw);
                            tc::tma_load_2d(sm.braw[rb.i], &tmW, sb * C::kSB, n0, &sm.fullB[rb.i]);
                            issB |= 1u << rb.i;
                            phB = (phB & ~(1u << rb.i)) | (rb.ph << rb.i);
                        }
                        rb.next(RB);
                    }
                    // activation f16 quants: one 32-block per operand slot
                    for (int j = 0; j < 8; ++j) {
                        if (lane == 0 && wait_or_abort(sm, &sm.emptyF[rf.i], rf.ph ^ 1u)) {
                            tc::mbar_arrive_expect_tx(&sm.fullF[rf.i], kTile);
                            tc::tma_load_2d(sm.f16[rf.i], &tmA, sb * 256 + 32 * j, m0, &sm.fullF[rf.i]);
                            issF |= 1u << rf.i;
                            phF = (phF & ~(1u << rf.i)) | (rf.ph << rf.i);
                        }
                        rf.next(RF);
                    }
                }
            }
            if (aborted(sm) && lane == 0) {   // let every copy already issued land before the CTA exits
                for (int i = 0; i < RF; ++i) if (issF >> i & 1u) tc::mbar_wait(&sm.fullF[i], phF >> i & 1u, kWaitLimitNs);
                for (int i = 0; i < RB; ++i) if (issB >> i & 1u) tc::mbar_wait(&sm.fullB[i], phB >> i & 1u, kWaitLimitNs);
                for (int i = 0; i < RD; ++i) if (issD >> i & 1u) tc::mbar_wait(&sm.fullD[i], phD >> i & 1u, kWaitLimitNs);
            }
        } else if (warp == 1) {
            // ---------------------------------------------------- MMA issuer
            // The whole warp runs the loop and waits; lane 0 issues. (A warp whose other 31
            // lanes stay parked while one lane runs the kernel-long loop slows every warp of
            // its SM sub-partition.)
            Ring rf, rm, rt;
            const uint32_t idesc = tc::instr_desc(BM, BN, 0);
            const uint32_t idesc32 = tc::instr_desc(BM, BN, 2);
            bool issued = false;
            for (int u = blockIdx.x; u < units && !waborted(sm); u += gridDim.x) {
                const Work wk = work_of<Q6>(u, whole, splits, num_mt, S);
                for (int sb = wk.sb0; sb < wk.sb1 && !waborted(sm); ++sb) {
                    for (int j = 0; j < 8; ++j) {
                        if (!wwait(sm, &sm.fullF[rf.i], rf.ph)) break;
                        if (!wwait(sm, &sm.tempty[rt.i], rt.ph ^ 1u)) break;
                        tc::tc_fence_after();
                        if (lane == 0) {
                            const uint32_t d = tbase + kSlotCol0 + 128u * rt.i;
                            const uint32_t sa = tc::smem_u32(sm.f16[rf.i]);
#pragma unroll
                            for (int part = 0; part < C::kBTiles; ++part) {
                                const uint32_t sbb = sa + kTile * (1 + part);
#pragma unroll
                                for (int k = 0; k < 2; ++k)
                                    tc::mma_f16(d, tc::smem_desc_sw64(sa + 32 * k, 512),
                                                tc::smem_desc_noswizzle(sbb + k * 2 * kLBO, kLBO, kSBO), idesc,
                                                (part | k) ? 1u : 0u);
                            }
                            tc::mma_commit(&sm.emptyF[rf.i]);
                            tc::mma_commit(&sm.tfull[rt.i]);
                        }
                        __syncwarp();
                        issued = true;
                        rf.next(RF);
                        rt.next(RT);
                    }
                    if constexpr (!Q6) {
                        if (waborted(sm)) break;
                        if (!wwait(sm, &sm.fullM[rm.i], rm.ph)) break;
                        if (!wwait(sm, &sm.tempty[rt.i], rt.ph ^ 1u)) break;
                        tc::tc_fence_after();
                        if (lane == 0) {
                            const uint32_t d = tbase + kSlotCol0 + 128u * rt.i;
                            const uint32_t sa = tc::smem_u32(sm.ms[rm.i]);
#pragma unroll
                            for (int k = 0; k < 2; ++k)
                                tc::mma_tf32(d, tc::smem_desc_noswizzle(sa + k * 2 * kLBO, kLBO, kSBO),
                                             tc::smem_desc_noswizzle(sa + kTile + k * 2 * kLBO, kLBO, kSBO), idesc32,
                                             k ? 1u : 0u);
                            tc::mma_commit(&sm.emptyM[rm.i]);
                            tc::mma_commit(&sm.tfull[rt.i]);
                        }
                        __syncwarp();
                        rm.next(RM);
                        rt.next(RT);
                    }
                }
            }
            if (lane == 0 && issued) {   // every MMA of this CTA has completed before TMEM is freed
                tc::mma_commit(&sm.mma_done);
                tc::mbar_wait(&sm.mma_done, 0, kWaitLimitNs);
            }
            tc::tc_fence_before();
            __syncwarp();
        }
    } else if (warp < 4 + kConvWarps) {
        // ============================================================ B converters
        tc::setmaxnreg_dec<kRegsConv>();
        const int c = lane >> 3;                       // 8-position part of a 32-block
        const int rbase = 8 * (warp - 4) + (lane & 7); // rows rbase + 64k: a quarter-warp covers 8 consecutive rows
        Ring rb, rf, rm, rs;
        if constexpr (Q6) {   // the first super-block of the first tile
            if (blockIdx.x < units) {
                const Work w0 = work_of<Q6>(blockIdx.x, whole, splits, num_mt, S);
                q6_fetch(sm.braw[0], W, w0.n0, w0.sb0, N, wstride, wtotal, rbase, c);
            }
        }
        for (int u = blockIdx.x; u < units && !waborted(sm); u += gridDim.x) {
            const Work wk = work_of<Q6>(u, whole, splits, num_mt, S);
            const int n0 = wk.n0;
            for (int sb = wk.sb0; sb < wk.sb1 && !waborted(sm); ++sb) {
                if constexpr (Q6) {
                    // prefetch the next super-block into the other stage, then wait for this one
                    const int nu = (sb + 1 < wk.sb1) ? u : u + (int)gridDim.x;
                    if (nu < units) {
                        const Work nw = (nu == u) ? wk : work_of<Q6>(nu, whole, splits, num_mt, S);
                        q6_fetch(sm.braw[rb.i ^ 1], W, nw.n0, (nu == u) ? sb + 1 : nw.sb0, N, wstride, wtotal, rbase, c);
                    }
                    else tc::cp_async_commit();
                    tc::cp_async_wait<1>();
                    __syncwarp();
                } else {
                    if (!wwait(sm, &sm.fullB[rb.i], rb.ph)) break;
                }
                if (!wwait(sm, &sm.emptyS[rs.i], rs.ph ^ 1u)) break;
                if constexpr (!Q6) {
                    if (!wwait(sm, &sm.emptyM[rm.i], rm.ph ^ 1u)) break;
                }
                const uint8_t* stage = sm.braw[rb.i];
                // ---- per-row super-block scales
#pragma unroll
                for (int k = 0; k < kConvRows; ++k) {
                    const int r = 8 * kConvWarps * k + rbase, n = n0 + r;
                    const bool valid = n < N;
                    if constexpr (Q6) {
                        const int delta = (int)(((unsigned long long)n * wstride + (unsigned long long)sb * C::kSB) & 15ull);
                        if (c == 0)
                            sm.wd[rs.i][r] = valid ? __half2float(__ushort_as_half(
                                                         *reinterpret_cast<const unsigned short*>(stage + r * C::kBStride + delta + 208)))
                                                   : 0.0f;
                    } else {
                        uint4 hdr = make_uint4(0, 0, 0, 0);
                        if (valid) hdr = *reinterpret_cast<const uint4*>(stage + r * C::kBStride);
                        if (c == 0) {
                            sm.wd[rs.i][r] = __half2float(__ushort_as_half((unsigned short)(hdr.x & 0xffffu)));
                            sm.wdmin[rs.i][r] = __half2float(__ushort_as_half((unsigned short)(hdr.x >> 16)));
                        }
                        // part c decodes sub-blocks 2c, 2c+1: f16 {sc, sc}, {-1024 sc, -1024 sc}, and the mins
                        float mv[2];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int j = 2 * c + u;
                            int sc, mn;
                            if (j < 4) {
                                sc = (int)(byte_at(hdr.y, hdr.z, hdr.w, j) & 63u);
                                mn = (int)(byte_at(hdr.y, hdr.z, hdr.w, j + 4) & 63u);
                            } else {
                                const uint32_t b = byte_at(hdr.y, hdr.z, hdr.w, j + 4);
                                sc = (int)((b & 15u) | ((byte_at(hdr.y, hdr.z, hdr.w, j - 4) >> 6) << 4));
                                mn = (int)((b >> 4) | ((byte_at(hdr.y, hdr.z, hdr.w, j) >> 6) << 4));
                            }
                            sm.scpack[r][j] = make_uint2(h2_of_int(sc), h2_of_int(-1024 * sc));
                            mv[u] = (float)mn;
                        }
                        // B_ms row r: K' = j and 8 + j both hold m_j; part c writes K' 2c, 2c+1 and 8+2c, 9+2c
                        *reinterpret_cast<float2*>(sm.ms[rm.i] + kTile + tile_off(r, c >> 1) + 8 * (c & 1)) =
                            make_float2(mv[0], mv[1]);
                        *reinterpret_cast<float2*>(sm.ms[rm.i] + kTile + tile_off(r, 2 + (c >> 1)) + 8 * (c & 1)) =
                            make_float2(mv[0], mv[1]);
                    }
                }
                if constexpr (!Q6) tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tc::mbar_arrive(&sm.fullS[rs.i]);
                    if constexpr (!Q6) tc::mbar_arrive(&sm.fullM[rm.i]);
                }
                rs.next(RS);
                if constexpr (!Q6) rm.next(RM);

                // ---- operand tiles, two 32-blocks per step
#pragma unroll
                for (int P = 0; P < 4; ++P) {
                    const int f0 = rf.i;
                    if (!wwait(sm, &sm.emptyF[rf.i], rf.ph ^ 1u)) break;
                    rf.next(RF);
                    const int f1 = rf.i;
                    if (!wwait(sm, &sm.emptyF[rf.i], rf.ph ^ 1u)) break;
                    rf.next(RF);
                    uint8_t* b0 = sm.f16[f0] + kTile;
                    uint8_t* b1 = sm.f16[f1] + kTile;
                    // Rows >= N convert to zeros (q4_K: the copy zero-filled them, so their scales
                    // are 0; q6_K: their scale is taken as 0). For q6_K all shared-memory loads of
                    // the thread's rows come before any store: a store may alias a later load as
                    // far as the compiler knows, which would serialise the rows.
                    if constexpr (!Q6) {
                        // sub-blocks 2P (low nibbles) and 2P+1 (high nibbles), positions 8c .. 8c+7. (Here
                        // the per-row order measured faster than loads first: fewer live registers.)
#pragma unroll
                        for (int k = 0; k < kConvRows; ++k) {
                            const int r = 8 * kConvWarps * k + rbase;
                            const uint4 sp = *reinterpret_cast<const uint4*>(&sm.scpack[r][2 * P]);
                            const uint2 q = *reinterpret_cast<const uint2*>(stage + r * C::kBStride + 16 + 32 * P + 8 * c);
                            const uint32_t m4 = 0x0F0F0F0Fu;
                            uint4 o0, o1;
                            nib4_to_f16_1024(q.x & m4, sp.x, sp.y, o0.x, o0.y);
                            nib4_to_f16_1024(q.y & m4, sp.x, sp.y, o0.z, o0.w);
                            nib4_to_f16_1024((q.x >> 4) & m4, sp.z, sp.w, o1.x, o1.y);
                            nib4_to_f16_1024((q.y >> 4) & m4, sp.z, sp.w, o1.z, o1.w);
                            *reinterpret_cast<uint4*>(b0 + tile_off(r, c)) = o0;
                            *reinterpret_cast<uint4*>(b1 + tile_off(r, c)) = o1;
                        }
                    } else {
                        // blocks 2P, 2P+1: half h, quarters tq0 = 2(P&1), tq0+1
                        const int h = P >> 1, tq0 = 2 * (P & 1), nsh = (P & 1) ? 4 : 0;
                        uint32_t l0a[kConvRows], l0b[kConvRows], l1a[kConvRows], l1b[kConvRows], qa[kConvRows],
                            qb[kConvRows];
                        int sc0[kConvRows], sc1[kConvRows];
#pragma unroll
                        for (int k = 0; k < kConvRows; ++k) {
                            const int r = 8 * kConvWarps * k + rbase, n = n0 + r;
                            const int delta = (int)(((unsigned long long)n * wstride + (unsigned long long)sb * C::kSB) & 15ull);
                            const uint8_t* blk = stage + r * C::kBStride + delta;
                            lds8_unaligned(blk + 64 * h + 8 * c, l0a[k], l0b[k]);
                            lds8_unaligned(blk + 64 * h + 32 + 8 * c, l1a[k], l1b[k]);
                            lds8_unaligned(blk + 128 + 32 * h + 8 * c, qa[k], qb[k]);
                            sc0[k] = (n < N) ? (int)(int8_t)blk[192 + 4 * P + (c >> 1)] : 0;
                            sc1[k] = (n < N) ? (int)(int8_t)blk[192 + 4 * P + 2 + (c >> 1)] : 0;
                        }
#pragma unroll
                        for (int k = 0; k < kConvRows; ++k) {
                            const int r = 8 * kConvWarps * k + rbase;
                            const uint32_t m0 = h2_of_int(16 * sc0[k]), a0 = h2_of_int(-16 * sc0[k]);
                            const uint32_t m1 = h2_of_int(16 * sc1[k]), a1 = h2_of_int(-16 * sc1[k]);
                            const uint32_t hm0 = h2_of_int(256 * sc0[k]), ha0 = h2_of_int(-288 * sc0[k]);
                            const uint32_t hm1 = h2_of_int(256 * sc1[k]), ha1 = h2_of_int(-288 * sc1[k]);
                            const uint32_t m4 = 0x0F0F0F0Fu, m2 = 0x03030303u;
                            uint4 o0, o1, o2, o3;
                            // block 2P: B1 = sc*lo -> o0, B2 = 16 sc (hi - 2) -> o1
                            nib4_to_f16_one((l0a[k] >> nsh) & m4, m0, a0, o0.x, o0.y);
                            nib4_to_f16_one((l0b[k] >> nsh) & m4, m0, a0, o0.z, o0.w);
                            nib4_to_f16_one((qa[k] >> (2 * tq0)) & m2, hm0, ha0, o1.x, o1.y);
                            nib4_to_f16_one((qb[k] >> (2 * tq0)) & m2, hm0, ha0, o1.z, o1.w);
                            // block 2P+1 -> o2, o3
                            nib4_to_f16_one((l1a[k] >> nsh) & m4, m1, a1, o2.x, o2.y);
                            nib4_to_f16_one((l1b[k] >> nsh) & m4, m1, a1, o2.z, o2.w);
                            nib4_to_f16_one((qa[k] >> (2 * tq0 + 2)) & m2, hm1, ha1, o3.x, o3.y);
                            nib4_to_f16_one((qb[k] >> (2 * tq0 + 2)) & m2, hm1, ha1, o3.z, o3.w);
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
                if constexpr (!Q6) {
                    if (lane == 0) tc::mbar_arrive(&sm.emptyB[rb.i]);
                }
                rb.next(RB);
            }
        }
        if constexpr (Q6) tc::cp_async_wait<0>();   // no copy of this CTA is left in flight
    } else {
        // ============================================================ epilogue
        tc::setmaxnreg_inc<kRegsEpi>();
        const int ew = warp - 4 - kConvWarps;
        const int q = warp & 3;                 // TMEM lane quarter (warp % 4)
        const int cq = ew >> 2;                 // column half: 64 * cq .. 64 * cq + 63
        const int rloc = 32 * q + lane;
        const uint32_t lane_bits = (uint32_t)(32 * q) << 16;
        Ring rd, rt, rs, rm;
        for (int u = blockIdx.x; u < units && !waborted(sm); u += gridDim.x) {
            const Work wk = work_of<Q6>(u, whole, splits, num_mt, S);
            const bool add = Q6 ? (u >= whole && splits > 1) : (splits > 1);   // partial sums of a split tile
            const int m0 = wk.m0, n0 = wk.n0;
            const int m = m0 + rloc;
            for (int sb = wk.sb0; sb < wk.sb1 && !waborted(sm); ++sb) {
                if (!wwait(sm, &sm.fullD[rd.i], rd.ph)) break;
                float da[8];
                {
                    const float4* dp = reinterpret_cast<const float4*>(sm.draw[rd.i] + rloc * 32);
                    const float4 x0 = dp[0], x1 = dp[1];
                    da[0] = x0.x; da[1] = x0.y; da[2] = x0.z; da[3] = x0.w;
                    da[4] = x1.x; da[5] = x1.y; da[6] = x1.z; da[7] = x1.w;
                }
                if constexpr (!Q6) {
                    if (cq == 0) {
                        // min-term activation operand, row rloc: K' = j (hi part of d_a,j * s_j), 8 + j (lo part)
                        if (!wwait(sm, &sm.emptyM[rm.i], rm.ph ^ 1u)) break;
                        const int4* sp = reinterpret_cast<const int4*>(sm.draw[rd.i] + kDRaw + rloc * 32);
                        const int4 s0 = sp[0], s1 = sp[1];
                        const int sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
                        float hi[8], lo[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float beta = da[j] * (float)sv[j];
                            hi[j] = __uint_as_float(__float_as_uint(beta) & 0xFFFFE000u);
                            lo[j] = beta - hi[j];
                        }
                        uint8_t* tile = sm.ms[rm.i];
                        *reinterpret_cast<float4*>(tile + tile_off(rloc, 0)) = make_float4(hi[0], hi[1], hi[2], hi[3]);
                        *reinterpret_cast<float4*>(tile + tile_off(rloc, 1)) = make_float4(hi[4], hi[5], hi[6], hi[7]);
                        *reinterpret_cast<float4*>(tile + tile_off(rloc, 2)) = make_float4(lo[0], lo[1], lo[2], lo[3]);
                        *reinterpret_cast<float4*>(tile + tile_off(rloc, 3)) = make_float4(lo[4], lo[5], lo[6], lo[7]);
                        tc::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&sm.fullM[rm.i]);
                    }
                    rm.next(RM);
                }
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&sm.emptyD[rd.i]);
                rd.next(RD);

                // per 32-block: acc += d_a * I (exact integer block dot from the MMA)
                float2 acc[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) acc[c] = make_float2(0.0f, 0.0f);
                bool ok = true;
#pragma unroll 1
                for (int j = 0; j < 8; ++j) {
                    if (!wwait(sm, &sm.tfull[rt.i], rt.ph)) { ok = false; break; }
                    tc::tc_fence_after();
                    uint32_t I0[32], I1[32];
                    const uint32_t ta = tbase + lane_bits + kSlotCol0 + 128u * rt.i + 64u * cq;
                    tc::tmem_ld32(ta, I0);
                    tc::tmem_ld32(ta + 32, I1);
                    tc::tmem_ld_wait();
                    tc::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&sm.tempty[rt.i]);
                    rt.next(RT);
                    // d_a of block j picked by selects: a dynamically indexed array would live in local memory
                    float dj = da[0];
#pragma unroll
                    for (int u = 1; u < 8; ++u) dj = (j == u) ? da[u] : dj;
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        tc::ffma2(acc[c].x, acc[c].y, dj, dj, __uint_as_float(I0[2 * c]), __uint_as_float(I0[2 * c + 1]));
                        tc::ffma2(acc[16 + c].x, acc[16 + c].y, dj, dj, __uint_as_float(I1[2 * c]), __uint_as_float(I1[2 * c + 1]));
                    }
                }
                if (!ok) break;
                // per super-block: out += d * acc (- dmin * MS for q4_K)
                uint32_t ms_slot = 0;
                if constexpr (!Q6) {
                    if (!wwait(sm, &sm.tfull[rt.i], rt.ph)) break;
                    tc::tc_fence_after();
                    ms_slot = kSlotCol0 + 128u * rt.i;
                }
                if (!wwait(sm, &sm.fullS[rs.i], rs.ph)) break;
                const bool first = (sb == wk.sb0), last = (sb == wk.sb1 - 1);
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const int col = 64 * cq + 16 * h;
                    uint32_t o[16], mv[16];
                    if (!first) tc::tmem_ld16(tbase + lane_bits + kOutCol + col, o);
                    if constexpr (!Q6) tc::tmem_ld16(tbase + lane_bits + ms_slot + col, mv);
                    tc::tmem_ld_wait();
                    const float4* wdp = reinterpret_cast<const float4*>(&sm.wd[rs.i][col]);
                    const float4* wmp = reinterpret_cast<const float4*>(&sm.wdmin[rs.i][col]);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float4 wv = wdp[u];
                        const float w4[4] = {wv.x, wv.y, wv.z, wv.w};
                        float m4v[4] = {0.f, 0.f, 0.f, 0.f};
                        if constexpr (!Q6) {
                            const float4 mm = wmp[u];
                            m4v[0] = mm.x; m4v[1] = mm.y; m4v[2] = mm.z; m4v[3] = mm.w;
                        }
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int cc = 4 * u + e;                 // 0..15 within the chunk
                            const int ai = 8 * h + (cc >> 1);         // float2 index in acc
                            const float av = (cc & 1) ? acc[ai].y : acc[ai].x;
                            float v = first ? 0.0f : __uint_as_float(o[cc]);
                            v = fmaf(w4[e], av, v);
                            if constexpr (!Q6) v = fmaf(-m4v[e], __uint_as_float(mv[cc]), v);
                            o[cc] = __float_as_uint(v);               // the result overwrites the loaded value
                        }
                    }
                    if (last) {
                        if (m < M) {
                            float* orow = out + (size_t)m * N + n0 + col;
                            // split-K: partial sums are added into the zeroed output
                            if (n0 + col + 16 <= N && (N & 3) == 0) {
#pragma unroll
                                for (int x = 0; x < 4; ++x) {
                                    const float4 v4 = make_float4(__uint_as_float(o[4 * x]), __uint_as_float(o[4 * x + 1]),
                                                                  __uint_as_float(o[4 * x + 2]), __uint_as_float(o[4 * x + 3]));
                                    if (add) atomicAdd(reinterpret_cast<float4*>(orow) + x, v4);
                                    else reinterpret_cast<float4*>(orow)[x] = v4;
                                }
                            } else {
                                for (int x = 0; x < 16; ++x) {
                                    if (n0 + col + x < N) {
                                        if (add) atomicAdd(orow + x, __uint_as_float(o[x]));
                                        else orow[x] = __uint_as_float(o[x]);
                                    }
                                }
                            }
                        }
                    } else {
                        tc::tmem_st16(tbase + lane_bits + kOutCol + col, o);
                    }
                }
                tc::tmem_st_wait();
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    tc::mbar_arrive(&sm.emptyS[rs.i]);
                    if constexpr (!Q6) tc::mbar_arrive(&sm.tempty[rt.i]);
                }
                rs.next(RS);
                if constexpr (!Q6) rt.next(RT);
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
              uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
              CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_NONE) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Split-K for the tiles of the last, partial wave (all tiles when there are fewer
// than SMs): each such tile's super-blocks are divided among `splits` work units
// (at least 2 super-blocks each), chosen to minimise the number of unit waves per
// split plus a small per-split cost.
int choose_splits(long long tiles, int S, int sms) {
    if (tiles >= sms) return 1;
    int best = 1;
    double best_cost = 1e30;
    for (int s = 1; s <= 32 && 2 * s <= S; ++s) {
        const long long waves = (tiles * s + sms - 1) / sms;
        const double cost = (double)waves / s + 0.01 * s;
        if (cost < best_cost) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
}

int check_gemm(const mq_q8_plane* a, const void* w, int N, const float* out) {
    if (!a) return MQ_ERR_NULL;
    if (N < 0 || a->M < 0 || !mq::valid_k(a->K)) return MQ_ERR_SHAPE;
    int rc = mq::check_plane(a, a->M, a->K);
    if (rc != MQ_OK || N == 0 || a->M == 0) return rc;
    if (!a->qh || !w || !out) return MQ_ERR_NULL;
    if (!mq::aligned16(w) || !mq::aligned16(out)) return MQ_ERR_ALIGN;
    return mq::check_arch();
}

template <bool Q6>
int launch_gemm(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream) {
    int rc = check_gemm(a, w, N, out);
    if (rc != MQ_OK || N == 0 || a->M == 0) return rc;
    const int M = a->M, K = a->K;
    // Once per process: the register split between warpgroups assumes the launch
    // register count, and the kernel's shared-memory size is set. Later calls make
    // no attribute calls, so a sequence of entry points can be captured in a graph.
    const size_t smem = sizeof(Smem<Q6>) + 1024;
    static int ready = -1;
    if (ready < 0) {
        cudaFuncAttributes fa;
        ready = (cudaFuncGetAttributes(&fa, gemm_kernel<Q6>) == cudaSuccess && fa.numRegs == kLaunchRegs &&
                 cudaFuncSetAttribute(gemm_kernel<Q6>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) ==
                     cudaSuccess)
                    ? 1
                    : 0;
    }
    if (!ready) return MQ_ERR_LAUNCH;
    const unsigned long long row = (unsigned long long)(K / mq::QK_K) * Cfg<Q6>::kSB;
    CUtensorMap tmA, tmD, tmS, tmW;
    if (Q6) {
        tmW = CUtensorMap{};   // unused: q6_K rows are not 16-byte aligned for a tensor map
    } else if (!make_map(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, row, (uint64_t)N, row, mq::Q4K_BYTES, BN)) {
        return MQ_ERR_LAUNCH;
    }
    if (!make_map(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a->qh, (uint64_t)K, (uint64_t)M, (uint64_t)K * 2, 32, BM,
                  CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map(&tmD, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a->d, (uint64_t)K / 32, (uint64_t)M, (uint64_t)K / 8, 8, BM) ||
        !make_map(&tmS, CU_TENSOR_MAP_DATA_TYPE_INT32, a->s, (uint64_t)K / 32, (uint64_t)M, (uint64_t)K / 8, 8, BM))
        return MQ_ERR_LAUNCH;
    const long long num_mt = (M + BM - 1) / BM, tiles = num_mt * ((N + BN - 1) / BN);
    const int sms = mq::num_sms();
    // q6_K: full waves of whole tiles, and the tiles of the last, partial wave split along
    // K. q4_K: split only when there are fewer tiles than SMs (then every tile is).
    const long long whole = Q6 ? (tiles / sms) * sms : 0;
    const int splits = tiles > whole ? choose_splits(tiles - whole, K / mq::QK_K, sms) : 1;
    if (splits > 1) {
        // The split tiles are the last ones in m-fastest order: they lie in the tile columns
        // from the one holding tile `whole` on. Zero those columns (whole tiles among them
        // overwrite the zeros with plain stores).
        const size_t col0 = (size_t)(whole / num_mt) * BN;
        if (cudaMemset2DAsync(out + col0, (size_t)N * sizeof(float), 0, ((size_t)N - col0) * sizeof(float),
                              (size_t)M, stream) != cudaSuccess)
            return MQ_ERR_LAUNCH;
    }
    const long long units = whole + (tiles - whole) * splits;
    const int grid = (int)(units < sms ? units : sms);
    gemm_kernel<Q6><<<grid, kThreads, smem, stream>>>(tmA, tmD, tmS, tmW, static_cast<const uint8_t*>(w), out, M, N, K,
                                                      (int)whole, splits, row, row * (unsigned long long)N);
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
