// Helpers shared by the decode / small-batch GEMV translation units.
#pragma once

#include "mq_internal.cuh"

namespace gemv {

constexpr int kThreads = 128;                  // 4 warps a block
constexpr int kWarpsPerBlock = kThreads / 32;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// dp4a of unsigned bytes (a) with signed bytes (b).
__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Checks shared by every GEMV entry point: 1 <= M <= MQ_GEMV_MAX_ROWS, K a multiple
// of 256, the plane's q8 arrays present, weights and output 16-byte aligned.
inline int check(const mq_q8_plane* a, const void* w, int N, const float* out) {
    if (!a) return MQ_ERR_NULL;
    if (N < 0 || a->M < 1 || a->M > MQ_GEMV_MAX_ROWS || !mq::valid_k(a->K)) return MQ_ERR_SHAPE;
    int rc = mq::check_plane(a, a->M, a->K);
    if (rc != MQ_OK || N == 0) return rc;
    if (!mq::has_q8(a) || !w || !out) return MQ_ERR_NULL;
    if (!mq::aligned16(w) || !mq::aligned16(out)) return MQ_ERR_ALIGN;
    return mq::check_arch();
}

// Persistent grid for a kernel of kThreads-thread blocks whose warps take `units`
// units of work grid-stride: as many blocks as are resident at once, never more than
// the work needs.
template <typename Kern>
int grid_for(long long units, Kern kern) {
    const int b = mq::resident_blocks(reinterpret_cast<const void*>(kern), kThreads, 0);
    const long long need = (units + kWarpsPerBlock - 1) / kWarpsPerBlock;
    const long long cap = (long long)mq::num_sms() * b;
    return (int)(need < cap ? need : cap);
}

}  // namespace gemv
