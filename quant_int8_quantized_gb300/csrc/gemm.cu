// Prefill GEMM: activation operand form x q4_K / q6_K super-block weights -> f32.
//
// "64 · r60 — the coronation", §3.1-§3.2: for nt >= 16 tokens the matmul runs as
// block dot products of quantized activations with the weight quants, rescaled
// per block; q6_K runs its 32-wide chunks as two 16-element halves, each with
// its own int8 scale.
//
// sm_103a has no int8 tcgen05 MMA, and GB300's int8 rate is far below its f16
// rate, so the products run on the f16 tensor pipe with f32 accumulation. One
// accumulation covers a whole 256-wide super-block; the epilogue rescales once
// per super-block:
//   activations (B operand, smem, TMA, 128-byte swizzle): the plane's operand
//       form ah = f16(2^e * d_a * q_a), one power of two e per row and
//       super-block, so 2^-e * ah = d_a * q_a within 2^-11;
//   weights (A operand, tensor memory, written by converter warps):
//       q4_K  sc * q * 2^-k, exact in f16 (sc <= 63, q <= 15; k below);
//       q6_K  sc * (q - 32) as two exact parts sc * lo and 16 * sc * (hi - 2)
//             (q = lo + 16 hi), two MMAs per K step into the same accumulator.
//   q4_K min term: -dmin * sum_j m_j * sum_{k in block j} a_k is folded into the
//       same accumulator by two more K = 16 MMAs per super-block: A (shared memory)
//       = the exact hi + lo binary16 parts of -(dmin / (d 2^k)) m_j, B = the
//       plane's exact block sums of ah as hi + lo parts. k >= 0 is the least power of two with
//       |d| 2^k >= |dmin|, so the ratio is at most 1 (d = 0: the main operand
//       is 0 and the ratio 1).
//   epilogue: out[tok][n] += (c_n * 2^-e_tok) * S[n][tok], c = d 2^k (q4_K; dmin
//       when d = 0) or d (q6_K).
// The error is at most 2^-11 * sum_k |a||w| from the activation rounding plus
// f32 accumulation and 2^-21-relative terms of the min-term ratio.
//
// Tile: 128 weight rows (MMA M, TMEM lanes) x 192 tokens (MMA N): at N = 192 an
// M = 128, K = 16 MMA with A in tensor memory keeps the tensor pipe ~92% busy
// (N = 128: 67%; A from shared memory: at most 80%). With fewer than 192 tokens the
// tile is the token count rounded up to 16 (a small batch, M in [2, 16), takes
// N = 16): boxes, MMA and epilogue shrink with it, and the weight stream bounds.
// Tensor memory (512 columns): two 192-column super-block accumulators (the
// epilogue drains one while the MMAs fill the other), the weight operand slots
// (4 slots of 32 columns: q4_K one K = 64 chunk each, q6_K one K = 32 quarter with
// both parts each).
//
// One persistent CTA per SM, 640 threads:
//   warp 0      TMA producer: activation slots (K = 64 x 192 tokens), the block-sum
//               record and 2^-e row of each super-block, weight rows;
//   warp 1      MMA issuer (warps 0 and 1 run their loops as whole warps, one
//               elected lane issuing each copy, MMA and commit);
//   warp 2      TMEM allocator;
//   warp 3      (ordered split only) waits for the tile's previous K slice, see Order;
//   warps 4-11  weight converters, thread = weight row, two warps per TMEM lane
//               quarter, each half of a super-block's K;
//   warps 12-19 epilogue, thread = weight row, two warps per lane quarter, 96
//               token columns each, accumulators in registers across the
//               super-blocks of a work unit.
// Every mbarrier wait is bounded; on timeout the kernel records an error, stops,
// drains its own copies and MMAs, frees TMEM and returns.
// Launches are programmatic dependent launches (set-up overlaps the previous kernel). A q6_K
// call whose tiles leave the grid's last round partly idle makes a second, dependent launch
// that runs those tiles as K slices added into the output in a fixed order (Order).

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <mutex>

#include "mq_internal.cuh"
#include "tc.cuh"

namespace {

__device__ unsigned int g_gemm_error;   // bit 0: a bounded wait gave up
// Flags of ordered split launches (see Order): a ring shared by the launches of a device,
// each taking its own range; every flag is back at 0 when its launch ends.
constexpr int kOrderRing = 1 << 16;
__device__ unsigned int g_order_flags[kOrderRing];

constexpr int BW = 128;                 // weight rows per tile (MMA M)
constexpr int BT = 192;                 // tokens per tile (MMA N)
constexpr int KS = 64;                  // K per activation slot and weight-operand slot
constexpr int RA = 5;                   // activation slots (q6_K; q4_K: one per K chunk, see Cfg)
constexpr int RX = 3;                   // per-super-block stages (block sums, 2^-e, weight scales c)
constexpr int kAxBytes = BT * 32;       // 16 binary16 block-sum parts per token
#ifndef MQ_WAIT_LIMIT_NS
#define MQ_WAIT_LIMIT_NS 2000000000ull   // test builds may shorten it
#endif
constexpr uint64_t kWaitLimitNs = MQ_WAIT_LIMIT_NS;
#ifdef MQ_TEST_INJECT
// Test builds only: when set, CTA 0's TMA producer skips its first activation copy, so that
// chunk's barrier never completes and the kernel's bounded waits run out (abort path).
__device__ int g_test_skip_first_act;
// Test builds only: when set, the first K slice of each tile of an ordered split never passes
// its flag on, so the later slices' bounded waits for it run out (abort path).
__device__ int g_test_skip_release;
#endif
constexpr uint32_t kTmemCols = 512;
constexpr int kShortTok = 64;           // token tiles up to this take the short-tile form (q4_K)
constexpr int kMTile = BW * 16 * 2;     // q4_K min-term operand: 128 rows x K 16, f16

// Weight types of the GEMM.
enum : int { kQ4K = 0, kQ6K = 1, kQ40 = 2, kQ41 = 3 };

template <int WT, bool SH = false>
struct Cfg {
    // q4_K: one exact binary16 operand per weight, K chunks of 64 (slot j = chunk j).
    // q6_K, q4_0, q4_1: two exact binary16 parts per weight, 32-wide quarters, two MMAs
    // per K = 16 step. q4_K and q4_1 add the min-term MMAs.
    static constexpr bool kQuarters = WT != kQ4K;
    static constexpr bool kMin = WT == kQ4K || WT == kQ41;
    // Bytes per 256 weights in global memory, and staged bytes per weight row (the TMA
    // box). q4_K, q4_0: raw 144-byte super-blocks (8 x 18 B for q4_0). q6_K: the 224-byte
    // prepacked form (mq.h), staged with a 240-byte pitch (the box reads 16 bytes past the
    // block) so that one 16-byte load per thread and row hits 8 distinct bank groups per 8
    // rows; q4_1: 8 x 20 B, staged with a 176-byte pitch for the same reason.
    static constexpr int kSB = WT == kQ6K ? mq::Q6K_PACKED_BYTES : WT == kQ41 ? 160 : mq::Q4K_BYTES;
    static constexpr int kRowBytes = WT == kQ6K ? 240 : WT == kQ41 ? 176 : 144;
    static constexpr int kStage = BW * kRowBytes;
    static constexpr int kRB = kQuarters ? 2 : 3;      // weight stages
    // Weight-operand slots in tensor memory, 32 columns each. q4_K: slot j holds K chunk j
    // (64 wide) of every super-block and is written by one converter half only. q6_K: slot
    // t holds quarter t of a super-block half (32 wide, both exact parts), written
    // alternately by the two halves, each waiting on its own "empty" barrier: every waiter
    // then waits for consecutive phases of its barrier, which a parity wait tells apart.
    static constexpr int kRF = 4;
    static constexpr uint32_t kFCols = 32;
    // q4_K: activation slot j and weight-operand slot j both hold K chunk j, so one
    // barrier pair per chunk covers both (the TMA and the 4 converter warps of its half
    // arrive on "full", the MMAs' commit on "empty"), and the min-term operand joins
    // the per-super-block block-sum stage the same way: half the issuer's waits.
    static constexpr bool kJoint = !kQuarters;
    static constexpr int kRA = WT == kQ4K ? 4 : RA;
    // Tensor memory: two accumulators of kTok columns, then the weight-operand slots (32
    // columns each, one K = 64 chunk of q4_K). A full tile (192 tokens) leaves room for one
    // super-block's 4 slots: each chunk's operand is rewritten only after the previous
    // super-block's MMAs of that chunk have completed. A short tile (SH, q4_K, at most 64
    // tokens) keeps the operands of kD = 3 super-blocks and the activation ring as many (12
    // slots of 64 tokens), so that the converters and the copies run up to three
    // super-blocks ahead of the MMAs. There every K = 16 MMA costs a fixed ~96 cycles
    // whatever its N (measured for N = 16 to 128, A from tensor or shared memory, one or
    // several accumulators), so the MMAs, not the weight stream, set the pace; keeping them
    // fed is what the deeper rings do. Activation slot a and operand slot a both hold K chunk
    // a % 4 of a super-block, under one barrier pair.
    static constexpr int kD = SH ? 3 : 1;
    static constexpr int kNA = SH ? 4 * kD : kRA;      // activation slots
    static constexpr int kTok = SH ? kShortTok : BT;   // tokens per tile at most
    static constexpr int kActSlot = kTok * KS * 2;     // bytes per activation slot
    static constexpr uint32_t kSCol1 = kTok, kACol = 2 * kTok;
    // Warps: 4 (TMA producer, MMA issuer, TMEM allocator, idle), 8 weight converters (two per
    // TMEM lane quarter, one K half each), 8 epilogue warps (two per lane quarter, kEpiCols
    // token columns each). Registers: the launch's share per thread, redistributed by setmaxnreg.
    static constexpr int kConvWarps = 8;
    static constexpr int kEpiWarps = 8;
    static constexpr int kThreads = 128 + 32 * (kConvWarps + kEpiWarps);
    static constexpr int kLaunchRegs = 96;             // 65536 / kThreads, rounded down to 8
    // q4_K: 56 / 72 / 136 (its converters spilled at 64; 1.4 % faster, 5 % on 64-token tiles);
    // the two-part types keep 64 / 64 / 144 (q6_K spills nothing there and ran 1.5 % slower
    // with the q4_K split).
    static constexpr int kRegsWG0 = WT == kQ4K ? 56 : 64, kRegsConv = WT == kQ4K ? 72 : 64,
                         kRegsEpi = WT == kQ4K ? 136 : 144;
    static_assert(128 * kRegsWG0 + 32 * kConvWarps * kRegsConv + 32 * kEpiWarps * kRegsEpi <= kThreads * kLaunchRegs,
                  "register split");
    static constexpr int kMinWarps = 4;                // warps writing the q4_K / q4_1 min-term operand
    static constexpr int kEpiCols = kTok / 2;          // accumulator columns per epilogue thread
    static_assert(!SH || WT == kQ4K, "short tiles: q4_K");
    static_assert(kACol + kFCols * kRF * kD <= kTmemCols, "tensor memory");
};

template <int WT, bool SH = false>
struct Smem {
    using C = Cfg<WT, SH>;
    static constexpr bool kMin = C::kMin;
    alignas(1024) uint8_t act[C::kNA][C::kActSlot];
    alignas(256) uint8_t ax[RX][kAxBytes];
    alignas(16) float af[RX][BT];
    float cvec[RX][BW];
    alignas(128) uint8_t braw[C::kRB][C::kStage];
    alignas(128) uint8_t mop[kMin ? RX : 1][kMin ? 2 * kMTile : 16];   // min-term operand (hi, lo) per stage
    uint64_t act_full[C::kNA], act_empty[C::kNA], ax_full[RX], ax_empty[RX], c_full[RX], c_empty[RX];
    uint64_t b_full[C::kRB], b_empty[C::kRB];
    uint64_t a_full[C::kRF], a_empty[C::kRF][2];
    uint64_t t_full[2], t_empty[2], mma_done;
    uint64_t ord_go;   // ordered split: the tile's previous slice is in the output
    uint32_t tmem;
    int abort;
};

// A work unit: one output tile (token tile fastest) and a slice sp, [sb0, sb1), of its
// super-blocks. A launch covers tiles tile0 .. tile0 + ntiles - 1, each as `splits` units;
// r is the tile's index within the launch. Units that share a tile add their partial sums
// into the output: in any order for split-K (the host zeroed the output beforehand), in slice
// order for an ordered launch (see Order).
struct Work {
    int m0, n0, sb0, sb1, sp, r;
    int pb;   // paired launch: which of the two problems (0: out / N / tmW, 1: Pair)
};
// nfast: weight-row tiles fastest (when the activation operand is the larger one, so
// that each token tile's activations are read from memory once).
__device__ __forceinline__ Work work_of(int u, int splits, int num_mt, int num_nt, bool nfast, int S, int bt,
                                        int tile0) {
    const int r = u / splits, sp = u - r * splits, t = tile0 + r;
    const int mt = nfast ? t / num_nt : t % num_mt, nt = nfast ? t % num_nt : t / num_mt;
    return Work{mt * bt, nt * BW, (sp * S) / splits, ((sp + 1) * S) / splits, sp, r, 0};
}

// Paired launch (mq_gemm_q4k_pair): two q4_K problems that read the same activation plane (the
// same M and K, e.g. attn_q and attn_k, or ffn_gate and ffn_up) in one persistent launch, whole
// tiles only. Units 0 .. tiles0 - 1 are the first problem's tiles (out, N, tmW), the rest the
// second's (Pair::out, Pair::N, tmW2): the second problem's tiles fill the rounds the first
// leaves idle, and the pair pays one launch's fixed cost instead of two.
struct Pair {
    float* out;   // the second problem's output
    int N;        // its weight rows
    int tiles0;   // the first problem's tiles
};

// Ordered split. A persistent grid of G CTAs takes the output tiles G at a time; when their
// count T is not a multiple of G, the last round would leave SMs idle for a whole tile's
// time. The host then launches the first T - T mod G tiles whole, and the last T mod G tiles
// in a second launch, cut along K into `splits` slices each that run side by side (the second
// launch may start as the first one's CTAs retire). Slice sp adds its partial sums into the
// output only after slice sp - 1 has stored or added its own: one flag per tile, tagged with
// the launch's epoch, which warp 3 of each CTA waits for and passes on (the epilogue warps
// wait on shared-memory barriers only), so the order of the additions, and the result, do
// not depend on timing. The last slice resets the flag to 0 for the next launch on the range.
struct Order {
    int on;           // 0: split-K units add in any order (or no split)
    unsigned epoch;   // this launch's tag, in the high bits of each flag value
    unsigned base;    // this launch's first flag in g_order_flags
    unsigned* flags;  // the flags in place of g_order_flags (instances with SF set: mq_gemm_q6k_static)
};

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded wait for an ordered-split flag to reach `want`.
__device__ bool wait_flag(const unsigned* fl, unsigned want) {
    const uint64_t t0 = tc::globaltimer();
    for (unsigned spin = 0;; ++spin) {
        if (ld_acquire_u32(fl) == want) return true;
        if ((spin & 63u) == 63u && tc::globaltimer() - t0 > kWaitLimitNs) return false;
    }
}

// Non-suspending test of a phase (acquire semantics, like the waits).
__device__ __forceinline__ bool mbar_ready(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok)
                 : "r"(tc::smem_u32(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

template <class SM>
__device__ __forceinline__ bool wait1(SM& sm, uint64_t* bar, uint32_t parity) {
    if (mbar_ready(bar, parity) || tc::mbar_wait(bar, parity, kWaitLimitNs)) return true;
    atomicOr(&g_gemm_error, 1u);
    *(volatile int*)&sm.abort = 1;
    return false;
}

template <class SM>
__device__ __forceinline__ bool aborted(SM& sm) {
    return *(volatile int*)&sm.abort != 0;
}

// Whole-warp variants: every lane waits, and the outcome is made warp-uniform so
// that the warp never diverges in front of a warp-collective operation.
template <class SM>
__device__ __forceinline__ bool wwait(SM& sm, uint64_t* bar, uint32_t parity) {
    const bool ok = __all_sync(0xffffffffu, mbar_ready(bar, parity) || tc::mbar_wait(bar, parity, kWaitLimitNs));
    if (!ok) {
        if ((threadIdx.x & 31) == 0) atomicOr(&g_gemm_error, 1u);
        *(volatile int*)&sm.abort = 1;
    }
    return ok;
}

template <class SM>
__device__ __forceinline__ bool waborted(SM& sm) {
    return __any_sync(0xffffffffu, aborted(sm));
}

// f16 bit pattern of a value exactly representable in binary16, in both halves.
__device__ __forceinline__ uint32_t h2_of(float v) {
    const uint32_t h = (uint32_t)__half_as_ushort(__float2half_rn(v));
    return h | (h << 16);
}
__device__ __forceinline__ uint32_t h2_pack(float lo, float hi) {
    return (uint32_t)__half_as_ushort(__float2half_rn(lo)) | ((uint32_t)__half_as_ushort(__float2half_rn(hi)) << 16);
}

// Four 4-bit values in the low nibble of each byte of `x` (byte i = K position i)
// -> f16 pairs (0, 1), (2, 3) of mul * v. The value is placed in the mantissa of
// 1024 (1024 + v); with add = -1024 * mul the fused multiply-add gives mul * v
// exactly (q4_K: mul = sc * 2^-k, |1024 * mul| <= 64512).
__device__ __forceinline__ void nib4_1024(uint32_t x, uint32_t mul2, uint32_t add2, uint32_t& p01, uint32_t& p23) {
    p01 = tc::hfma2(tc::prmt(x, 0x64u, 0x4140u), mul2, add2);
    p23 = tc::hfma2(tc::prmt(x, 0x64u, 0x4342u), mul2, add2);
}

// Same for q6_K, where the multipliers reach 256 * 128: v (0..15) is placed as
// 1 + v/16 and mul16 = 16 * mul, add = -16 * mul + offset stay inside f16.
__device__ __forceinline__ void nib4_one(uint32_t x, uint32_t mul16, uint32_t add2, uint32_t& p01, uint32_t& p23) {
    const uint32_t t01 = (tc::prmt(x, 0u, 0x4140u) << 6) | 0x3C003C00u;
    const uint32_t t23 = (tc::prmt(x, 0u, 0x4342u) << 6) | 0x3C003C00u;
    p01 = tc::hfma2(t01, mul16, add2);
    p23 = tc::hfma2(t23, mul16, add2);
}

__device__ __forceinline__ uint32_t byte_of(uint32_t y, uint32_t z, uint32_t w, int i) {
    const uint32_t v = (i < 4) ? y : (i < 8 ? z : w);
    return (v >> (8 * (i & 3))) & 0xffu;
}

// A binary16 bit pattern as m * 2^E with m its integer significand (< 2048, 0 for zero).
__device__ __forceinline__ void f16_split(uint32_t hb, int& m, int& E) {
    const int e = (int)((hb >> 10) & 31u);
    m = e ? (int)(1024u | (hb & 1023u)) : (int)(hb & 1023u);
    E = (e ? e : 1) - 25;
}

// q4_K super-block header (the word holding f16 d and dmin): k, the least power of two in
// [0, 24] with |d| 2^k >= |dmin| (0 when d or dmin is 0; from the exponents and the
// significands, as the doubling loop it replaces would find it), sk = 2^-k, c = d 2^k (dmin
// when d = 0; exact) and rr = dmin / c.
struct Q4KHead {
    float d, c, rr, sk;
};
__device__ __forceinline__ Q4KHead q4k_head(uint32_t w) {
    Q4KHead h;
    h.d = __half2float(__ushort_as_half((unsigned short)(w & 0xffffu)));
    const float dmin = __half2float(__ushort_as_half((unsigned short)(w >> 16)));
    int k = 0;
    h.c = dmin;
    h.rr = 1.0f;
    if (h.d != 0.0f) {
        const uint32_t bd = __float_as_uint(h.d) & 0x7fffffffu, bm = __float_as_uint(dmin) & 0x7fffffffu;
        if (bm != 0u) {   // both normal in f32 (binary16 inputs): compare exponents, then significands
            const int kk = (int)(bm >> 23) - (int)(bd >> 23) + ((bm & 0x7fffffu) > (bd & 0x7fffffu) ? 1 : 0);
            k = min(24, max(0, kk));
        }
        h.c = __int_as_float(__float_as_int(h.d) + (k << 23));
        h.rr = __fdiv_rn(dmin, h.c);
    }
    h.sk = __int_as_float((127 - k) << 23);
    return h;
}

// A 32-bit word from a 2-byte-aligned shared-memory address.
__device__ __forceinline__ uint32_t ld_u32_a2(const uint8_t* p) {
    return (uint32_t)*reinterpret_cast<const uint16_t*>(p) | ((uint32_t)*reinterpret_cast<const uint16_t*>(p + 2) << 16);
}

template <int WT, bool SH, bool ORD = false, bool SF = false, bool PAIR = false>
__global__ void __launch_bounds__(Cfg<WT, SH>::kThreads, 1) gemm_kernel(const __grid_constant__ CUtensorMap tmAct,
                                                           const __grid_constant__ CUtensorMap tmAx,
                                                           const __grid_constant__ CUtensorMap tmAf,
                                                           const __grid_constant__ CUtensorMap tmW,
                                                           const __grid_constant__ CUtensorMap tmW2,
                                                           float* __restrict__ out, int M, int N, int K, int splits,
                                                           int nfast, int bt, int tile0, int ntiles, const Order ord,
                                                           const Pair pair) {
    using C = Cfg<WT, SH>;
    constexpr int kRB = C::kRB, kRF = C::kRF;
    extern __shared__ uint8_t smem_raw[];
    Smem<WT, SH>& sm = *reinterpret_cast<Smem<WT, SH>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = K / mq::QK_K;
    const int num_mt = (M + bt - 1) / bt, num_nt = (N + BW - 1) / BW;
    // the ordered split (Order) is compiled into its own instance, used only for the second
    // launch of an ordered split: compiled into the instances every other launch uses, it made
    // them up to 27 % slower
    constexpr bool kOrd = ORD;
    // q6_K launches may cover part of the tiles (the first launch of an ordered split)
    int units = WT == kQ6K ? ntiles * splits : num_mt * num_nt * splits;
    if constexpr (PAIR) units = pair.tiles0 + num_mt * ((pair.N + BW - 1) / BW);   // whole tiles (splits = 1)
    // the work unit u: its tile and super-block range, and for a paired launch its problem
    auto unit = [&](int u) -> Work {
        if constexpr (PAIR) {
            if (u >= pair.tiles0) {
                Work w = work_of(u - pair.tiles0, 1, num_mt, (pair.N + BW - 1) / BW, nfast, S, bt, 0);
                w.pb = 1;
                return w;
            }
            return work_of(u, 1, num_mt, num_nt, nfast, S, bt, 0);
        } else {
            return work_of(u, splits, num_mt, num_nt, nfast, S, bt, kOrd ? tile0 : 0);
        }
    };

    if (tid == 0) {
        tc::prefetch_tensormap(&tmW);
        if constexpr (PAIR) tc::prefetch_tensormap(&tmW2);
        tc::prefetch_tensormap(&tmAct);
        tc::prefetch_tensormap(&tmAx);
        tc::prefetch_tensormap(&tmAf);
        for (int i = 0; i < C::kNA; ++i) {
            tc::mbar_init(&sm.act_full[i], C::kJoint ? 5 : 1);
            tc::mbar_init(&sm.act_empty[i], 1);
        }
        for (int i = 0; i < RX; ++i) {
            tc::mbar_init(&sm.ax_full[i], C::kMin ? 1 + C::kMinWarps : 1);   // + the warps writing the min operand
            tc::mbar_init(&sm.ax_empty[i], 1 + C::kEpiWarps);   // the MMAs (block sums) and the epilogue (2^-e)
            tc::mbar_init(&sm.c_full[i], 4);
            tc::mbar_init(&sm.c_empty[i], C::kEpiWarps);
        }
        for (int i = 0; i < kRB; ++i) {
            tc::mbar_init(&sm.b_full[i], 1);
            tc::mbar_init(&sm.b_empty[i], C::kConvWarps);
        }
        for (int i = 0; i < kRF; ++i) {
            tc::mbar_init(&sm.a_full[i], 4);
            tc::mbar_init(&sm.a_empty[i][0], 1);
            tc::mbar_init(&sm.a_empty[i][1], 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&sm.t_full[i], 1);
            tc::mbar_init(&sm.t_empty[i], C::kEpiWarps);
        }
        tc::mbar_init(&sm.mma_done, 1);
        tc::mbar_init(&sm.ord_go, 1);
        sm.abort = 0;
        tc::fence_mbar_init();
    }
    if (warp == 2) tc::tmem_alloc(&sm.tmem, kTmemCols);
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tbase = sm.tmem;
    // Launched as a programmatic dependent launch, the set-up above overlaps the previous
    // kernel's tail; nothing in global memory is read or written before this wait. The next
    // launch may start only once every CTA has passed it, so the second launch of an ordered
    // split (which reads nothing the first one writes) needs no wait of its own here: by then
    // the kernels before the first launch have completed.
    if constexpr (!ORD) mq_grid_wait();
    mq_grid_release();

    if (warp < 4) {
        // ============================================================ warpgroup 0
        tc::setmaxnreg_dec<C::kRegsWG0>();
        if (warp == 0) {
            // ---------------------------------------------------- TMA producer
            // As the issuer: the whole warp runs the loop and waits, one elected lane issues
            // the copies (warp-uniform coordinates and addresses; the q6_K GEMM gained 7 %).
            const bool leader = tc::elect_one();
            uint32_t issA = 0, phA = 0, issX = 0, phX = 0, issB = 0, phB = 0;   // copies in flight (for an abort)
            int sbc = 0, ga = 0;
            for (int u = blockIdx.x; u < units && !waborted(sm); u += gridDim.x) {
                const Work wk = unit(u);
                for (int sb = wk.sb0; sb < wk.sb1 && !waborted(sm); ++sb, ++sbc) {
                    const int x = sbc % RX;
                    if (!wwait(sm, &sm.ax_empty[x], ((sbc / RX) & 1) ^ 1)) break;
                    if (leader) tc::mbar_arrive_expect_tx(&sm.ax_full[x], (uint32_t)bt * (32 + 4));
                    if (leader) tc::tma_load_2d(sm.ax[x], &tmAx, 16 * sb, wk.m0, &sm.ax_full[x]);
                    if (leader) tc::tma_load_2d(sm.af[x], &tmAf, wk.m0, sb, &sm.ax_full[x]);
                    issX |= 1u << x;
                    phX = (phX & ~(1u << x)) | (((sbc / RX) & 1) << x);
                    {
                        const int b = sbc % kRB;
                        if (!wwait(sm, &sm.b_empty[b], ((sbc / kRB) & 1) ^ 1)) break;
                        if (leader) tc::mbar_arrive_expect_tx(&sm.b_full[b], C::kStage);
                        if (leader) tc::tma_load_2d(sm.braw[b], PAIR && wk.pb ? &tmW2 : &tmW, sb * C::kSB, wk.n0, &sm.b_full[b]);
                        issB |= 1u << b;
                        phB = (phB & ~(1u << b)) | (((sbc / kRB) & 1) << b);
                    }
                    bool ok = true;
                    for (int j = 0; j < 4; ++j, ++ga) {
                        const int a = ga % C::kNA;
                        const uint32_t pa = (ga / C::kNA) & 1;
                        if (!wwait(sm, &sm.act_empty[a], pa ^ 1)) { ok = false; break; }
#ifdef MQ_TEST_INJECT
                        if (g_test_skip_first_act && blockIdx.x == 0 && ga == 0) continue;
#endif
                        if (leader) tc::mbar_arrive_expect_tx(&sm.act_full[a], (uint32_t)bt * KS * 2);
                        if (leader) tc::tma_load_2d(sm.act[a], &tmAct, sb * 256 + KS * j, wk.m0, &sm.act_full[a]);
                        issA |= 1u << a;
                        phA = (phA & ~(1u << a)) | (pa << a);
                    }
                    if (!ok) break;
                }
            }
            if (waborted(sm)) {   // let every copy already issued land before the CTA exits
                for (int i = 0; i < C::kNA; ++i) if (issA >> i & 1u) tc::mbar_wait(&sm.act_full[i], phA >> i & 1u, kWaitLimitNs);
                for (int i = 0; i < RX; ++i) if (issX >> i & 1u) tc::mbar_wait(&sm.ax_full[i], phX >> i & 1u, kWaitLimitNs);
                for (int i = 0; i < kRB; ++i) if (issB >> i & 1u) tc::mbar_wait(&sm.b_full[i], phB >> i & 1u, kWaitLimitNs);
            }
        } else if (warp == 1) {
            // ---------------------------------------------------- MMA issuer
            // The whole warp runs the issue loop (its waits are whole-warp waits) and one
            // elected lane issues each MMA and commit: the descriptors and tensor-memory
            // addresses are then warp-uniform values, which the MMA takes without per-issue
            // register moves. Issued from a lone thread, a K = 16 MMA of a 16-token tile took
            // ~120-150 cycles of issue; this way the q6_K GEMM runs 8 % faster and a 16-token
            // q4_K tile 13 %.
            // The tensor pipe queues only a few MMAs, so every wait between MMA groups that
            // finds the pipe empty leaves it idle. The issuer therefore tests the barriers of
            // the next group in the middle of the current one, with MMAs still queued: group
            // (sbc, j) for j = 0..3 is K chunk j of super-block sbc; after chunk 3 come the
            // super-block's q4_K min-term MMAs and the next super-block's accumulator slot.
            const bool leader = tc::elect_one();
            const uint32_t idesc = tc::instr_desc(BW, (uint32_t)bt, 0);
            int total = 0;   // super-blocks this CTA accumulates (the issuer needs no tile positions)
            for (int u = blockIdx.x; u < units; u += gridDim.x) {
                const Work wk = unit(u);
                total += wk.sb1 - wk.sb0;
            }
            // readiness of chunk j of super-block sbc, whose activation slot is ga
            // q4_K: chunk j is ready when its joint barrier completes; q6_K: its activation
            // slot and its first quarter's operand (the second quarter is waited for between
            // the first quarter's MMAs)
            auto chunk_ready = [&](int sbc_, int j_, int ga_) {
                if constexpr (C::kJoint) return wwait(sm, &sm.act_full[ga_ % C::kNA], (ga_ / C::kNA) & 1);
                return wwait(sm, &sm.act_full[ga_ % C::kNA], (ga_ / C::kNA) & 1) &&
                       wwait(sm, &sm.a_full[(2 * j_) & 3], (uint32_t)(j_ >> 1));
            };
            auto sb_ready = [&](int sbc_, int ga_) {   // accumulator slot free, first chunk ready
                return wwait(sm, &sm.t_empty[sbc_ & 1], ((sbc_ >> 1) & 1) ^ 1) && chunk_ready(sbc_, 0, ga_);
            };
            bool ok = total > 0 && sb_ready(0, 0);
            tc::tc_fence_after();
            int ga = 0;
            for (int sbc = 0; sbc < total && ok; ++sbc) {
                const int s = sbc & 1, x = sbc % RX;
                const uint32_t dcol = tbase + (s ? C::kSCol1 : 0u);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int a = (ga + j) % C::kNA;
                    const uint32_t sa = tc::smem_u32(sm.act[a]);
                    if constexpr (!C::kQuarters) {
                        const uint32_t fa = tbase + C::kACol + C::kFCols * a;   // operand slot a
#pragma unroll
                        for (int k = 0; k < 2; ++k)
                            if (leader) tc::mma_f16_ts(dcol, fa + 8 * k, tc::smem_desc_sw128(sa + 32 * k), idesc, (j | k) ? 1u : 0u);
                        // while those run: the next group's barriers
                        ok = j < 3 ? chunk_ready(sbc, j + 1, ga + j + 1) : wwait(sm, &sm.ax_full[x], (sbc / RX) & 1);
                        if (!ok) break;
                        tc::tc_fence_after();
#pragma unroll
                        for (int k = 2; k < 4; ++k)
                            if (leader) tc::mma_f16_ts(dcol, fa + 8 * k, tc::smem_desc_sw128(sa + 32 * k), idesc, 1u);
                        if (leader) tc::mma_commit(&sm.act_empty[a]);
                    } else {
                        // quarters q = 2j, 2j + 1 (operand slot q & 3, written by half j >> 1); each
                        // K = 16 step is two MMAs, the parts sc*lo and 16*sc*(hi - 2)
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            const int qq = (2 * j + i) & 3;
                            const uint32_t fa = tbase + C::kACol + C::kFCols * qq;
#pragma unroll
                            for (int k = 0; k < 2; ++k) {
                                const uint64_t bd = tc::smem_desc_sw128(sa + 64 * i + 32 * k);
                                if (leader) tc::mma_f16_ts(dcol, fa + 8 * k, bd, idesc, (j | i | k) ? 1u : 0u);
                                if (leader) tc::mma_f16_ts(dcol, fa + 16 + 8 * k, bd, idesc, 1u);
                            }
                            if (leader) tc::mma_commit(&sm.a_empty[qq][1 - (j >> 1)]);   // the next writer is the other half
                            // while those run: the next quarter (and at the chunk's end the next chunk)
                            if (i == 0) ok = wwait(sm, &sm.a_full[qq + 1], (uint32_t)(j >> 1));
                            else if (j < 3) ok = chunk_ready(sbc, j + 1, ga + j + 1);
                            if (!ok) break;
                            tc::tc_fence_after();
                        }
                        if (!ok) break;
                        if (leader) tc::mma_commit(&sm.act_empty[a]);
                    }
                }
                if (!ok) break;
                ga += 4;
                if constexpr (C::kMin) {
                    if constexpr (C::kQuarters) {   // q4_1: the block sums and the min operand (q4_K waited at chunk 3)
                        if (!wwait(sm, &sm.ax_full[x], (sbc / RX) & 1)) break;
                        tc::tc_fence_after();
                    }
                    const uint64_t bd = tc::smem_desc_sw32(tc::smem_u32(sm.ax[x]));
                    const uint32_t ma = tc::smem_u32(sm.mop[x]);
                    if (leader) tc::mma_f16(dcol, tc::smem_desc_noswizzle(ma, 128, 256), bd, idesc, 1u);
                    if (leader) tc::mma_f16(dcol, tc::smem_desc_noswizzle(ma + kMTile, 128, 256), bd, idesc, 1u);
                }
                if (leader) tc::mma_commit(&sm.ax_empty[x]);   // q6_K, q4_0: a token arrival (the block sums are the epilogue's)
                if (leader) tc::mma_commit(&sm.t_full[s]);
                if (sbc + 1 < total) {
                    ok = sb_ready(sbc + 1, ga);
                    tc::tc_fence_after();
                }
            }
            if (total > 0) {   // every MMA of this CTA has completed before TMEM is freed
                if (leader) tc::mma_commit(&sm.mma_done);
                tc::mbar_wait(&sm.mma_done, 0, kWaitLimitNs);
            }
            tc::tc_fence_before();
        } else if (kOrd && warp == 3 && ord.on) {
            // ---------------------------------------------------- ordered split: let the
            // epilogue add once the tile's previous slice (another CTA) is in; the flag is passed
            // on at the end of the kernel. An ordered launch gives each CTA at most one unit (the
            // host keeps its units within the grid).
            const int u = blockIdx.x;
            if (u < units) {
                const Work wk = unit(u);
                if (wk.sp > 0) {
                    const bool got =
                        lane == 0 ? wait_flag((SF ? ord.flags : g_order_flags) + ord.base + wk.r, (ord.epoch << 4) | (unsigned)wk.sp) : true;
                    if (__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
                        if (lane == 0) tc::mbar_arrive(&sm.ord_go);
                    } else {
                        if (lane == 0) atomicOr(&g_gemm_error, 1u);
                        *(volatile int*)&sm.abort = 1;
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp < 4 + C::kConvWarps) {
        // ============================================================ weight converters
        tc::setmaxnreg_dec<C::kRegsConv>();
        const int q = warp & 3, h = (warp - 4) >> 2;
        const int r = 32 * q + lane;                            // weight row within the tile
        const uint32_t lane_bits = (uint32_t)(32 * q) << 16;
        int sbc = 0;
        for (int u = blockIdx.x; u < units && !waborted(sm); u += gridDim.x) {
            const Work wk = unit(u);
            const int n = wk.n0 + r;
            for (int sb = wk.sb0; sb < wk.sb1 && !waborted(sm); ++sb, ++sbc) {
                const int b = sbc % kRB, x = sbc % RX;
                if (!wwait(sm, &sm.b_full[b], (sbc / kRB) & 1)) break;
                const uint8_t* row = sm.braw[b] + r * C::kRowBytes;
                if constexpr (WT == kQ4K) {
                    // ---- q4_K: scales and the power of two k; the main operand of chunks 2h, 2h + 1,
                    //      then (h == 0) the min-term operand and the epilogue's scale c
                    const uint4 hdr = *reinterpret_cast<const uint4*>(row);
                    const Q4KHead hd = q4k_head(hdr.x);
                    // chunk j of super-block sbc: operand (and activation) slot f, written by this
                    // half only, once the MMAs of its previous use (kD super-blocks ago) completed
                    auto main_chunk = [&](int j) -> bool {
                        const int f = 4 * (sbc % C::kD) + j;
                        if (!wwait(sm, &sm.act_empty[f], ((sbc / C::kD) & 1) ^ 1)) return false;
                        tc::tc_fence_after();   // the stores below come after the MMAs that read the slot
                        const int s0 = j < 2 ? (int)(byte_of(hdr.y, hdr.z, hdr.w, 2 * j) & 63u)
                                             : (int)((byte_of(hdr.y, hdr.z, hdr.w, 2 * j + 4) & 15u) |
                                                     ((byte_of(hdr.y, hdr.z, hdr.w, 2 * j - 4) >> 6) << 4));
                        const int s1 = j < 2 ? (int)(byte_of(hdr.y, hdr.z, hdr.w, 2 * j + 1) & 63u)
                                             : (int)((byte_of(hdr.y, hdr.z, hdr.w, 2 * j + 5) & 15u) |
                                                     ((byte_of(hdr.y, hdr.z, hdr.w, 2 * j - 3) >> 6) << 4));
                        const float m0f = hd.d != 0.0f ? (float)s0 * hd.sk : 0.0f;   // sc 2^-k, exact
                        const float m1f = hd.d != 0.0f ? (float)s1 * hd.sk : 0.0f;
                        const uint32_t mul0 = h2_of(m0f), add0 = h2_of(-1024.0f * m0f);
                        const uint32_t mul1 = h2_of(m1f), add1 = h2_of(-1024.0f * m1f);
                        const uint4 qa = *reinterpret_cast<const uint4*>(row + 16 + 32 * j);
                        const uint4 qb = *reinterpret_cast<const uint4*>(row + 32 + 32 * j);
                        const uint32_t wv[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
                        uint32_t o[32];
#pragma unroll
                        for (int w = 0; w < 8; ++w) {
                            nib4_1024(wv[w] & 0x0F0F0F0Fu, mul0, add0, o[2 * w], o[2 * w + 1]);
                            nib4_1024((wv[w] >> 4) & 0x0F0F0F0Fu, mul1, add1, o[16 + 2 * w], o[16 + 2 * w + 1]);
                        }
                        tc::tmem_st32(tbase + lane_bits + C::kACol + C::kFCols * f, o);
                        tc::tmem_st_wait();
                        tc::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&sm.act_full[f]);
                        return true;
                    };
                    // min-term operand of sub-blocks 2i, 2i + 1: -(dmin / c) m as exact hi + lo
                    // binary16 parts, packed in pairs
                    auto min_pair = [&](int i, uint32_t& hi, uint32_t& lo) {
                        float v[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int jj = 2 * i + e;
                            const uint32_t mn = jj < 4 ? (byte_of(hdr.y, hdr.z, hdr.w, jj + 4) & 63u)
                                                       : ((byte_of(hdr.y, hdr.z, hdr.w, jj + 4) >> 4) |
                                                          ((byte_of(hdr.y, hdr.z, hdr.w, jj) >> 6) << 4));
                            v[e] = -__fmul_rn(hd.rr, (float)mn);
                        }
                        const float hi0 = __half2float(__float2half_rn(v[0])), hi1 = __half2float(__float2half_rn(v[1]));
                        hi = h2_pack(v[0], v[1]);
                        lo = h2_pack(__fsub_rn(v[0], hi0), __fsub_rn(v[1], hi1));
                    };
                    // row r of the hi tile [hi_0..hi_7, hi_0..hi_7] and of the lo tile, K-major
                    // without swizzle: core matrices of 8 rows x 16 B, K-adjacent ones 128 B apart
                    uint8_t* mt = sm.mop[x] + (r >> 3) * 256 + (r & 7) * 16;
                    bool ok = true;
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj)
                        if (!main_chunk(2 * h + jj)) { ok = false; break; }
                    if (!ok) break;
                    if (h == 0) {
                        if (!wwait(sm, &sm.ax_empty[x], ((sbc / RX) & 1) ^ 1)) break;
                        uint32_t mh[8];
#pragma unroll
                        for (int i = 0; i < 4; ++i) min_pair(i, mh[i], mh[4 + i]);
                        const uint4 vh = make_uint4(mh[0], mh[1], mh[2], mh[3]), vl = make_uint4(mh[4], mh[5], mh[6], mh[7]);
                        *reinterpret_cast<uint4*>(mt) = vh;
                        *reinterpret_cast<uint4*>(mt + 128) = vh;
                        *reinterpret_cast<uint4*>(mt + kMTile) = vl;
                        *reinterpret_cast<uint4*>(mt + kMTile + 128) = vl;
                        tc::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&sm.ax_full[x]);
                        if (!wwait(sm, &sm.c_empty[x], ((sbc / RX) & 1) ^ 1)) break;
                        sm.cvec[x][r] = n < (PAIR && wk.pb ? pair.N : N) ? hd.c : 0.0f;
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&sm.c_full[x]);
                    }
                } else if constexpr (WT == kQ6K) {
                    // ---- q6_K (prepacked): half h of the block is 112 bytes at 112 h: ql (64), qh (32),
                    //      the half's 8 scales, d. Slot j = 2h + jj covers quarters t = 2jj + i, i = 0, 1:
                    //      low bits from ql bytes 32i.. (high nibble when jj = 1), high bits from qh
                    //      bits 2t, scale of element l = byte 2t + (l >= 16).
                    const uint8_t* half = row + 112 * h;
                    const uint4 c6 = *reinterpret_cast<const uint4*>(half + 96);
                    const uint4 h0 = *reinterpret_cast<const uint4*>(half + 64);
                    const uint4 h1 = *reinterpret_cast<const uint4*>(half + 80);
                    const uint32_t qh[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
                    bool ok = true;
                    // quarter t of this half -> operand slot t, written alternately by the halves:
                    // half 0 waits for the previous super-block's half-1 use to be read, half 1 for
                    // this super-block's half-0 use
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        if (!wwait(sm, &sm.a_empty[t][h], h ? (sbc & 1) : ((sbc & 1) ^ 1))) { ok = false; break; }
                        tc::tc_fence_after();   // the stores below come after the MMAs that read the slot
                        const uint32_t fa = tbase + lane_bits + C::kACol + C::kFCols * t;
                        const uint32_t scw = (t < 2) ? c6.x : c6.y;     // scale bytes 2t, 2t + 1 of the half
                        const uint4 l0 = *reinterpret_cast<const uint4*>(half + 32 * (t & 1));
                        const uint4 l1 = *reinterpret_cast<const uint4*>(half + 32 * (t & 1) + 16);
                        const uint32_t ql[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
                        const int nsh = (t >> 1) * 4, hsh = 2 * t;
                        uint32_t p1[16], p2[16];
#pragma unroll
                        for (int w = 0; w < 8; ++w) {
                            const float sc = (float)(int)(int8_t)(scw >> (8 * (2 * (t & 1) + (w >> 2))));
                            nib4_one((ql[w] >> nsh) & 0x0F0F0F0Fu, h2_of(16.0f * sc), h2_of(-16.0f * sc), p1[2 * w],
                                     p1[2 * w + 1]);
                            nib4_one((qh[w] >> hsh) & 0x03030303u, h2_of(256.0f * sc), h2_of(-288.0f * sc), p2[2 * w],
                                     p2[2 * w + 1]);
                        }
                        tc::tmem_st16(fa, p1);
                        tc::tmem_st16(fa + 16, p2);
                        tc::tmem_st_wait();
                        tc::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&sm.a_full[t]);
                    }
                    if (!ok) break;
                    if (h == 0) {
                        if (!wwait(sm, &sm.c_empty[x], ((sbc / RX) & 1) ^ 1)) break;
                        sm.cvec[x][r] = n < N ? __half2float(__ushort_as_half((unsigned short)(c6.z & 0xffffu))) : 0.0f;
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&sm.c_full[x]);
                    }
                } else {
                    // ---- q4_0 / q4_1: eight 32-blocks of kB bytes. Block b's scale is d_b = g_b 2^E_b
                    //      (g_b its 11-bit integer significand) and g_b = 64 Dh + Dl (Dh < 32, Dl < 64),
                    //      so that with c = 2^Ec a power of two per row and super-block,
                    //          d_b (q - o) / c = (q - o) Dh 2^(E_b + 6 - Ec) + (q - o) Dl 2^(E_b - Ec),
                    //      two parts of at most 9 and 10 significant bits: exact in binary16 (o = 8 for
                    //      q4_0, 0 for q4_1). Ec is the largest E_b (and, q4_1, large enough that every
                    //      m_b / c stays below 2^15), so the parts stay below 2^14 and are exact while the
                    //      super-block's block scales lie within 2^24 of each other. Quarter t of half h
                    //      is block 4h + t, in operand slot t (both parts), as q6_K's quarters.
                    constexpr bool Q41 = WT == kQ41;
                    constexpr int kB = Q41 ? 20 : 18;
                    int ec = -1000;
                    uint32_t dm[8];   // bit patterns: d_b (low half), q4_1: m_b (high half)
#pragma unroll
                    for (int bb = 0; bb < 8; ++bb) {
                        dm[bb] = Q41 ? *reinterpret_cast<const uint32_t*>(row + kB * bb)
                                     : (uint32_t)*reinterpret_cast<const uint16_t*>(row + kB * bb);
                        int g, E;
                        f16_split(dm[bb] & 0xffffu, g, E);
                        if (g) ec = max(ec, E);
                        if (Q41) {
                            f16_split(dm[bb] >> 16, g, E);
                            if (g) ec = max(ec, E - 4);   // |m_b| < 2^(E + 11) <= 2^15 c
                        }
                    }
                    if (ec == -1000) ec = 0;
                    bool ok = true;
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        if (!wwait(sm, &sm.a_empty[t][h], h ? (sbc & 1) : ((sbc & 1) ^ 1))) { ok = false; break; }
                        tc::tc_fence_after();   // the stores below come after the MMAs that read the slot
                        const int bb = 4 * h + t;
                        const uint8_t* blk = row + kB * bb;
                        int g, E;
                        f16_split(dm[bb] & 0xffffu, g, E);
                        const float sgn = (dm[bb] & 0x8000u) ? -1.0f : 1.0f;
                        const float m1 = sgn * ldexpf((float)(g >> 6), E + 6 - ec);
                        const float m2 = sgn * ldexpf((float)(g & 63), E - ec);
                        const float off = Q41 ? 16.0f : 24.0f;   // (1 + v/16) 16 mul - off mul = (v - o) mul
                        const uint32_t mul1 = h2_of(16.0f * m1), add1 = h2_of(-off * m1);
                        const uint32_t mul2 = h2_of(16.0f * m2), add2 = h2_of(-off * m2);
                        uint32_t qw[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            qw[i] = Q41 ? *reinterpret_cast<const uint32_t*>(blk + 4 + 4 * i) : ld_u32_a2(blk + 2 + 4 * i);
                        uint32_t p1[16], p2[16];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint32_t lo = qw[i] & 0x0F0F0F0Fu, hi = (qw[i] >> 4) & 0x0F0F0F0Fu;
                            nib4_one(lo, mul1, add1, p1[2 * i], p1[2 * i + 1]);          // K 4i .. 4i + 3
                            nib4_one(hi, mul1, add1, p1[8 + 2 * i], p1[9 + 2 * i]);      // K 16 + 4i ..
                            nib4_one(lo, mul2, add2, p2[2 * i], p2[2 * i + 1]);
                            nib4_one(hi, mul2, add2, p2[8 + 2 * i], p2[9 + 2 * i]);
                        }
                        const uint32_t fa = tbase + lane_bits + C::kACol + C::kFCols * t;
                        tc::tmem_st16(fa, p1);
                        tc::tmem_st16(fa + 16, p2);
                        tc::tmem_st_wait();
                        tc::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&sm.a_full[t]);
                    }
                    if (!ok) break;
                    if (h == 0) {
                        if constexpr (Q41) {   // the min operand: m_b / c as hi + lo binary16 parts
                            if (!wwait(sm, &sm.ax_empty[x], ((sbc / RX) & 1) ^ 1)) break;
                            uint32_t mh[8];
#pragma unroll
                            for (int j = 0; j < 8; j += 2) {
                                float v[2];
#pragma unroll
                                for (int e = 0; e < 2; ++e) {
                                    const float mb = __half2float(__ushort_as_half((unsigned short)(dm[j + e] >> 16)));
                                    v[e] = ldexpf(mb, -ec);
                                }
                                const float hi0 = __half2float(__float2half_rn(v[0]));
                                const float hi1 = __half2float(__float2half_rn(v[1]));
                                mh[j / 2] = h2_pack(v[0], v[1]);
                                mh[4 + j / 2] = h2_pack(__fsub_rn(v[0], hi0), __fsub_rn(v[1], hi1));
                            }
                            uint8_t* mt = sm.mop[x] + (r >> 3) * 256 + (r & 7) * 16;
                            const uint4 vh = make_uint4(mh[0], mh[1], mh[2], mh[3]), vl = make_uint4(mh[4], mh[5], mh[6], mh[7]);
                            *reinterpret_cast<uint4*>(mt) = vh;
                            *reinterpret_cast<uint4*>(mt + 128) = vh;
                            *reinterpret_cast<uint4*>(mt + kMTile) = vl;
                            *reinterpret_cast<uint4*>(mt + kMTile + 128) = vl;
                            tc::fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) tc::mbar_arrive(&sm.ax_full[x]);
                        }
                        if (!wwait(sm, &sm.c_empty[x], ((sbc / RX) & 1) ^ 1)) break;
                        sm.cvec[x][r] = n < N ? ldexpf(1.0f, ec) : 0.0f;
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&sm.c_full[x]);
                    }
                }
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&sm.b_empty[b]);
            }
        }
    } else {
        // ============================================================ epilogue
        tc::setmaxnreg_inc<C::kRegsEpi>();
        const int ew = warp - 4 - C::kConvWarps;
        const int q = warp & 3, ch = ew >> 2;         // lane quarter, column half (kEpiCols tokens)
        const int r = 32 * q + lane;
        const uint32_t lane_bits = (uint32_t)(32 * q) << 16;
        int sbc = 0;
        for (int u = blockIdx.x; u < units && !waborted(sm); u += gridDim.x) {
            const Work wk = unit(u);
            float acc[C::kEpiCols];
#pragma unroll
            for (int i = 0; i < C::kEpiCols; ++i) acc[i] = 0.0f;
            bool ok = true;
            for (int sb = wk.sb0; sb < wk.sb1; ++sb, ++sbc) {
                const int s = sbc & 1, x = sbc % RX;
                if (!wwait(sm, &sm.c_full[x], (sbc / RX) & 1) || !wwait(sm, &sm.ax_full[x], (sbc / RX) & 1) ||
                    !wwait(sm, &sm.t_full[s], (sbc >> 1) & 1)) {
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
                const float c = sm.cvec[x][r];
                const uint32_t ta = tbase + lane_bits + (s ? C::kSCol1 : 0u) + C::kEpiCols * ch;
                // 16 columns at a time (32 at a time, the accumulators no longer all fit in registers)
#pragma unroll
                for (int cc = 0; cc < C::kEpiCols / 16; ++cc) {
                    if (C::kEpiCols * ch + 16 * cc >= bt) break;   // no token of the tile in these columns
                    uint32_t v[16];
                    tc::tmem_ld16(ta + 16 * cc, v);
                    tc::tmem_ld_wait();
                    const float4* fp = reinterpret_cast<const float4*>(&sm.af[x][C::kEpiCols * ch + 16 * cc]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float4 f4 = fp[i];
                        float g0, g1, g2, g3;
                        tc::fmul2(g0, g1, c, c, f4.x, f4.y);
                        tc::fmul2(g2, g3, c, c, f4.z, f4.w);
                        float* a = &acc[16 * cc + 4 * i];
                        tc::ffma2(a[0], a[1], g0, g1, __uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]));
                        tc::ffma2(a[2], a[3], g2, g3, __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
                    }
                }
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    tc::mbar_arrive(&sm.t_empty[s]);
                    tc::mbar_arrive(&sm.ax_empty[x]);
                    tc::mbar_arrive(&sm.c_empty[x]);
                }
            }
            if (!ok) break;
            // ordered split: slice sp > 0 adds once warp 3 has seen slice sp - 1 in (the same
            // reduction as split-K, in a fixed order)
            bool add;
            if constexpr (kOrd) {
                const int usp = u % splits;   // the unit's slice (recomputed: fewer live registers)
                if (ord.on && usp > 0 && !wwait(sm, &sm.ord_go, 0)) break;   // (one unit per CTA)
                add = splits > 1 && !(ord.on && usp == 0);
            } else {
                add = splits > 1;
            }
            const int n = wk.n0 + r;
            const int NN = PAIR && wk.pb ? pair.N : N;
            if (n < NN) {
                const int t0 = wk.m0 + C::kEpiCols * ch;
                float* op = (PAIR && wk.pb ? pair.out : out) + (size_t)t0 * NN + n;
#pragma unroll
                for (int i = 0; i < C::kEpiCols; ++i) {
                    if (t0 + i < M) {
                        if (add) atomicAdd(op + (size_t)i * NN, acc[i]);
                        else op[(size_t)i * NN] = acc[i];
                    }
                }
            }
        }
    }

    __syncthreads();
    if (warp == 2) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tbase, kTmemCols);
    }
    if (kOrd && ord.on && warp == 3 && lane == 0 && blockIdx.x < units && !aborted(sm)) {
        // every store and addition of this CTA came before the block barrier above; the release
        // at GPU scope passes the tile to its next slice, or frees the flag after the last one
        const int sp = blockIdx.x % splits, r0 = blockIdx.x / splits;
        unsigned* fl = (SF ? ord.flags : g_order_flags) + ord.base + r0;
#ifdef MQ_TEST_INJECT
        if (g_test_skip_release && sp == 0) fl = nullptr;
#endif
        if (fl && sp < splits - 1) st_release_u32(fl, (ord.epoch << 4) | (unsigned)(sp + 1));
        else if (fl) *fl = 0u;
    }
    // the second launch of an ordered split ends after the first one (otherwise the wait has
    // returned already), so that what follows on the stream sees both
    mq_grid_wait();
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

// Split-K when there are fewer tiles than SMs: each tile's super-blocks are divided
// among `splits` work units (at least 2 super-blocks each), chosen to minimise the
// number of unit waves per split plus a small per-split cost.
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

// Slices per tile for the tiles of an incomplete last round (Order), or 1: at most as many
// as fit the grid (and 15, the flag's slice field), chosen to minimise that round's length
// in super-blocks: ceil(S / ts), plus kChainCost for each hand-over between slices (a flag and
// the additions, ~2-3 us) and kLaunchCost for the second launch (its pipeline fills and drains
// again: ~20 us, measured on the q6_K kernel at ~2.2 us a super-block). No split if nothing is
// gained.
constexpr int kChainCost = 2, kLaunchCost = 10;
int order_slices(long long tiles, int S, int sms) {
    if (tiles <= sms) return 1;   // fewer tiles than SMs: split-K instead
    const long long rest = tiles % sms;
    if (rest == 0) return 1;
    const long long cap = sms / rest < 15 ? sms / rest : 15;
    int best = 1, best_cost = S;
    for (int ts = 2; ts <= cap; ++ts) {
        const int cost = (S + ts - 1) / ts + kChainCost * (ts - 1) + kLaunchCost;
        if (cost < best_cost) {
            best_cost = cost;
            best = ts;
        }
    }
    return best;
}

// The epoch and flag range of an ordered launch, per device. Launches take consecutive
// ranges of the ring, so launches in flight together never share a flag.
bool order_range(int need, unsigned* epoch, unsigned* base) {
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static unsigned ep[kMaxDevices], next[kMaxDevices];
    int dev = 0;
    if (need > kOrderRing || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lk(mu);
    if (next[dev] + (unsigned)need > (unsigned)kOrderRing) next[dev] = 0;
    *base = next[dev];
    next[dev] += (unsigned)need;
    ep[dev] = (ep[dev] + 1u) & 0x0fffffffu;   // 28 bits
    if (ep[dev] == 0u) ep[dev] = 1u;
    *epoch = ep[dev];
    return true;
}

// The host-side checks of one GEMM call's arguments (check_gemm adds the architecture).
int check_gemm_args(const mq_q8_plane* a, const void* w, int N, const float* out) {
    if (!a) return MQ_ERR_NULL;
    if (N < 0 || a->M < 0 || !mq::valid_k(a->K)) return MQ_ERR_SHAPE;
    int rc = mq::check_plane(a, a->M, a->K);
    if (rc != MQ_OK || N == 0 || a->M == 0) return rc;
    if (!mq::has_op(a) || !w || !out) return MQ_ERR_NULL;
    if (!mq::aligned16(w) || !mq::aligned16(out)) return MQ_ERR_ALIGN;
    return MQ_OK;
}

int check_gemm(const mq_q8_plane* a, const void* w, int N, const float* out) {
    const int rc = check_gemm_args(a, w, N, out);
    if (rc != MQ_OK || N == 0 || a->M == 0) return rc;
    return mq::check_arch();
}

// Once per device: the register split between warpgroups assumes the launch register
// count, and the kernel's shared-memory size is set. Later calls make no attribute
// calls, so a sequence of entry points can be captured in a graph.
template <int WT, bool SH, bool ORD = false, bool SF = false, bool PAIR = false>
bool gemm_ready(size_t smem) {
    constexpr int kMaxDevices = 64;
    static int state[kMaxDevices];   // 0 unknown, 1 ready, 2 failed
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    int v = __atomic_load_n(&state[dev], __ATOMIC_ACQUIRE);
    if (v == 0) {
        std::lock_guard<std::mutex> lk(mu);
        v = state[dev];
        if (v == 0) {
            cudaFuncAttributes fa;
            v = (cudaFuncGetAttributes(&fa, gemm_kernel<WT, SH, ORD, SF, PAIR>) == cudaSuccess &&
                 fa.numRegs == Cfg<WT, SH>::kLaunchRegs &&
                 cudaFuncSetAttribute(gemm_kernel<WT, SH, ORD, SF, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)smem) ==
                     cudaSuccess)
                    ? 1
                    : 2;
            __atomic_store_n(&state[dev], v, __ATOMIC_RELEASE);
        }
    }
    return v == 1;
}

// Token-tile height: 192 tokens, or for fewer tokens the count rounded up to the
// MMA's N granule of 16. A small batch (M in [2, 16) and beyond) then moves, multiplies
// and reads back only the columns it has: the activation boxes, the MMA's N and the
// epilogue's TMEM loads all shrink with it, and the kernel becomes bound by the
// weight stream and its conversion rather than by work on empty columns.
int token_tile(int M) { return M >= BT ? BT : ((M + 15) / 16) * 16; }

// static_flags: mq_gemm_q6k_static's fixed flag array (device address), else nullptr
constexpr int kStaticFlags = 1024;   // tiles an ordered split of mq_gemm_q6k_static may cut, at most

// Tensor maps of the plane's operand arrays for token tiles of bt.
bool act_maps(const mq_q8_plane* a, int bt, CUtensorMap* tmAct, CUtensorMap* tmAx, CUtensorMap* tmAf) {
    const int M = a->M, K = a->K, S = K / mq::QK_K, mp = mq::af_stride(M);
    return make_map(tmAct, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a->ah, (uint64_t)K, (uint64_t)M, (uint64_t)K * 2, KS, bt,
                    CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_map(tmAx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a->ax, (uint64_t)S * 16, (uint64_t)M, (uint64_t)S * 32, 16, bt,
                    CU_TENSOR_MAP_SWIZZLE_32B) &&
           make_map(tmAf, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a->af, (uint64_t)mp, (uint64_t)S, (uint64_t)mp * 4, bt, 1);
}

template <int WT>
int launch_gemm(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream,
                unsigned* static_flags = nullptr) {
    int rc = check_gemm(a, w, N, out);
    if (rc != MQ_OK || N == 0 || a->M == 0) return rc;
    const int M = a->M, K = a->K, S = K / mq::QK_K;
    const int bt = token_tile(M);
    constexpr bool kS = WT == kQ4K;   // the short-tile form exists for q4_K
    const bool sh = kS && bt <= kShortTok;
    const size_t smem = sh ? sizeof(Smem<WT, kS>) + 1024 : sizeof(Smem<WT, false>) + 1024;
    if (!(sh ? gemm_ready<WT, kS>(smem) : gemm_ready<WT, false>(smem))) return MQ_ERR_LAUNCH;
    const unsigned long long row = (unsigned long long)S * Cfg<WT>::kSB;
    CUtensorMap tmAct, tmAx, tmAf, tmW;
    if (!make_map(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, row, (uint64_t)N, row, Cfg<WT>::kRowBytes, BW))
        return MQ_ERR_LAUNCH;
    if (!act_maps(a, bt, &tmAct, &tmAx, &tmAf)) return MQ_ERR_LAUNCH;
    const long long tiles = (long long)((M + bt - 1) / bt) * ((N + BW - 1) / BW);
    const int sms = mq::num_sms();
    const int splits = choose_splits(tiles, S, sms);
    if (splits > 1 && cudaMemsetAsync(out, 0, (size_t)M * N * sizeof(float), stream) != cudaSuccess)
        return MQ_ERR_LAUNCH;
    // weight-row tiles fastest when the activations outweigh the weights
    const int nfast = (double)M * K * 2 > (double)N * row ? 1 : 0;
    // one launch of tiles [tile0, tile0 + ntiles), each as `sp` units
    const Order none{0, 0u, 0u};
    auto plain = [&](int tile0, int ntiles, int sp) -> int {
        const long long units = (long long)ntiles * sp;
        const int grid = (int)(units < sms ? units : sms);
        if (sh)
            return mq::launch_pdl(gemm_kernel<WT, kS>, dim3(grid), dim3(Cfg<WT, kS>::kThreads), smem, stream, tmAct,
                                  tmAx, tmAf, tmW, tmW, out, M, N, K, sp, nfast, bt, tile0, ntiles, none, Pair{});
        return mq::launch_pdl(gemm_kernel<WT, false>, dim3(grid), dim3(Cfg<WT, false>::kThreads), smem, stream, tmAct,
                              tmAx, tmAf, tmW, tmW, out, M, N, K, sp, nfast, bt, tile0, ntiles, none, Pair{});
    };
    const int ts = WT == kQ6K && !sh && splits == 1 ? order_slices(tiles, S, sms) : 1;
    if (ts == 1) return plain(0, (int)tiles, splits);
    if constexpr (WT == kQ6K) {
        // ordered split: whole tiles for the complete rounds, then the rest in ts slices each, in
        // a dependent launch of the ordered instance (at most one unit per CTA: rest * ts <= sms)
        const int full = (int)(tiles - tiles % sms), rest = (int)(tiles - full);
        if (static_flags) {
            // mq_gemm_q6k_static: its own flags, cleared on the stream, used from 0 with one epoch
            if (rest > kStaticFlags) return MQ_ERR_SCRATCH;
            if (!gemm_ready<WT, false, true, true>(smem)) return MQ_ERR_LAUNCH;
            if (cudaMemsetAsync(static_flags, 0, (size_t)rest * sizeof(unsigned), stream) != cudaSuccess)
                return MQ_ERR_LAUNCH;
            rc = plain(0, full, 1);
            if (rc != MQ_OK) return rc;
            return mq::launch_pdl(gemm_kernel<WT, false, true, true>, dim3(rest * ts), dim3(Cfg<WT, false>::kThreads), smem,
                                  stream, tmAct, tmAx, tmAf, tmW, tmW, out, M, N, K, ts, nfast, bt, full, rest,
                                  Order{1, 1u, 0u, static_flags}, Pair{});
        }
        if (!gemm_ready<WT, false, true>(smem)) return MQ_ERR_LAUNCH;
        Order ord{1, 0u, 0u};
        if (!order_range(rest, &ord.epoch, &ord.base)) return MQ_ERR_LAUNCH;
        rc = plain(0, full, 1);
        if (rc != MQ_OK) return rc;
        return mq::launch_pdl(gemm_kernel<WT, false, true>, dim3(rest * ts), dim3(Cfg<WT, false>::kThreads), smem, stream,
                              tmAct, tmAx, tmAf, tmW, tmW, out, M, N, K, ts, nfast, bt, full, rest, ord, Pair{});
    }
    return MQ_ERR_LAUNCH;
}

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return na && nb && x < y + nb && y < x + na;
}

// Two q4_K problems on one plane (Pair): one launch when both have whole 192-token tiles and
// together fill at least one round of the grid, else two ordinary calls.
int launch_gemm_q4k_pair(const mq_q8_plane* a, const void* w0, int N0, float* out0, const void* w1, int N1,
                         float* out1, cudaStream_t stream) {
    int rc = check_gemm_args(a, w0, N0, out0);
    if (rc == MQ_OK) rc = check_gemm_args(a, w1, N1, out1);
    if (rc != MQ_OK) return rc;
    if (a->M == 0 || (N0 == 0 && N1 == 0)) return MQ_OK;
    rc = mq::check_arch();
    if (rc != MQ_OK) return rc;
    const int M = a->M, K = a->K, S = K / mq::QK_K;
    if (ranges_overlap(out0, (size_t)M * N0 * sizeof(float), out1, (size_t)M * N1 * sizeof(float))) return MQ_ERR_SHAPE;
    const int bt = token_tile(M), sms = mq::num_sms();
    const long long num_mt = (M + bt - 1) / bt;
    const long long tiles0 = num_mt * ((N0 + BW - 1) / BW), tiles1 = num_mt * ((N1 + BW - 1) / BW);
    if (N0 == 0 || N1 == 0 || bt != BT || tiles0 + tiles1 < sms) {
        rc = launch_gemm<kQ4K>(a, w0, N0, out0, stream);
        return rc != MQ_OK ? rc : launch_gemm<kQ4K>(a, w1, N1, out1, stream);
    }
    using C = Cfg<kQ4K, false>;
    const size_t smem = sizeof(Smem<kQ4K, false>) + 1024;
    if (!gemm_ready<kQ4K, false, false, false, true>(smem)) return MQ_ERR_LAUNCH;
    const unsigned long long row = (unsigned long long)S * C::kSB;
    CUtensorMap tmAct, tmAx, tmAf, tmW0, tmW1;
    if (!make_map(&tmW0, CU_TENSOR_MAP_DATA_TYPE_UINT8, w0, row, (uint64_t)N0, row, C::kRowBytes, BW) ||
        !make_map(&tmW1, CU_TENSOR_MAP_DATA_TYPE_UINT8, w1, row, (uint64_t)N1, row, C::kRowBytes, BW) ||
        !act_maps(a, bt, &tmAct, &tmAx, &tmAf))
        return MQ_ERR_LAUNCH;
    const int nfast = (double)M * K * 2 > (double)(N0 + N1) * row ? 1 : 0;
    const long long units = tiles0 + tiles1;
    const int grid = (int)(units < sms ? units : sms);
    return mq::launch_pdl(gemm_kernel<kQ4K, false, false, false, true>, dim3(grid), dim3(C::kThreads), smem, stream,
                          tmAct, tmAx, tmAf, tmW0, tmW1, out0, M, N0, K, 1, nfast, bt, 0, (int)tiles0, Order{},
                          Pair{out1, N1, (int)tiles0});
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
        // a launch that gave up may have left ordered-split flags set
        void* flags = nullptr;
        if (cudaGetSymbolAddress(&flags, g_order_flags) != cudaSuccess ||
            cudaMemset(flags, 0, sizeof(unsigned) * kOrderRing) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
            return MQ_ERR_LAUNCH;
    }
    *code = v;
    return MQ_OK;
}
}  // namespace mq

#ifdef MQ_TEST_INJECT
// Test builds only: switch the injected failures on or off (bit 0: the missing copy, bit 1:
// the missing flag release of an ordered split).
extern "C" int mq_test_inject(int on) {
    const int act = on & 1, rel = (on >> 1) & 1;
    return cudaMemcpyToSymbol(g_test_skip_first_act, &act, sizeof(act)) == cudaSuccess &&
                   cudaMemcpyToSymbol(g_test_skip_release, &rel, sizeof(rel)) == cudaSuccess
               ? MQ_OK
               : MQ_ERR_LAUNCH;
}
#endif

extern "C" int mq_gemm_q4k(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream) {
    return launch_gemm<kQ4K>(a, w, N, out, stream);
}

extern "C" int mq_gemm_q6k(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream) {
    return launch_gemm<kQ6K>(a, w, N, out, stream);
}

extern "C" int mq_gemm_q4k_pair(const mq_q8_plane* a, const void* w0, int N0, float* out0, const void* w1, int N1,
                                float* out1, cudaStream_t stream) {
    return launch_gemm_q4k_pair(a, w0, N0, out0, w1, N1, out1, stream);
}

// The scratch of mq_gemm_q6k_static: one flag per tile of an ordered split's second launch
// (4 KB, held by every GPU that loads the library until the process exits). Host code must
// not pass the name itself to a kernel: on the host it stands for a host-side shadow, not the
// device memory. static_flags_ptr looks the device address up, once per device.
static __device__ __align__(256) unsigned int g_static_flags[kStaticFlags];

namespace {
unsigned* static_flags_ptr() {
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static unsigned* ptr[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_flags) != cudaSuccess || !p) return nullptr;
        ptr[dev] = static_cast<unsigned*>(p);
    }
    return ptr[dev];
}
}  // namespace

extern "C" int mq_gemm_q6k_static(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream) {
    const int rc = check_gemm(a, w, N, out);
    if (rc != MQ_OK || N == 0 || a->M == 0) return rc;
    unsigned* flags = static_flags_ptr();
    if (!flags) return MQ_ERR_LAUNCH;
    return launch_gemm<kQ6K>(a, w, N, out, stream, flags);
}

extern "C" int mq_gemm_q4_0(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream) {
    return launch_gemm<kQ40>(a, w, N, out, stream);
}

extern "C" int mq_gemm_q4_1(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream) {
    return launch_gemm<kQ41>(a, w, N, out, stream);
}
