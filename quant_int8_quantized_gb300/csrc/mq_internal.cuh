// Internal helpers shared by the libmq CUDA translation units.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "mq.h"

namespace mq {

constexpr int QK = 32;          // activation block
constexpr int QK_K = 256;       // weight super-block
constexpr int Q4K_BYTES = 144;
constexpr int Q6K_BYTES = 210;
constexpr int Q6K_PACKED_BYTES = 224;   // prepacked q6_K super-block (mq_prepack_q6k)

// Host-side validation helpers ------------------------------------------------

int check_arch();   // MQ_OK if the current device is compute capability 10.3

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool has_q8(const mq_q8_plane* p) { return p->qs || p->d || p->s; }
inline bool has_op(const mq_q8_plane* p) { return p->ah || p->ax || p->af; }

// Shape and pointers of a plane: each array group (q8: qs, d, s; operand: ah, ax, af)
// is all present or all absent, at least one is present, and every array is 16-byte
// aligned.
inline int check_plane(const mq_q8_plane* p, int M, int K) {
    if (!p) return MQ_ERR_NULL;
    if (p->M != M || p->K != K) return MQ_ERR_SHAPE;
    if (M == 0) return MQ_OK;
    const bool q8 = has_q8(p), op = has_op(p);
    if (!q8 && !op) return MQ_ERR_NULL;
    if (q8 && (!p->qs || !p->d || !p->s)) return MQ_ERR_NULL;
    if (op && (!p->ah || !p->ax || !p->af)) return MQ_ERR_NULL;
    if (q8 && (!aligned16(p->qs) || !aligned16(p->d) || !aligned16(p->s))) return MQ_ERR_ALIGN;
    if (op && (!aligned16(p->ah) || !aligned16(p->ax) || !aligned16(p->af))) return MQ_ERR_ALIGN;
    return MQ_OK;
}

// Row stride (elements) of the operand array af: M rounded up to a multiple of 4.
inline int af_stride(int M) { return (M + 3) & ~3; }

inline bool valid_k(int K) { return K > 0 && (K % QK_K) == 0; }

inline int launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? MQ_OK : MQ_ERR_LAUNCH;
}

int num_sms();      // SM count of the current device (cached)

// Blocks of `kern` (launched with `threads` threads and `smem` bytes of dynamic shared
// memory) resident per SM on the current device; queried once per kernel, device and
// launch shape, then cached. At least 1.
int resident_blocks(const void* kern, int threads, size_t smem);

// Launch with programmatic stream serialization: the kernel may start while the
// previous kernel on the stream is finishing. Kernels launched this way call
// mq_grid_wait() before reading anything an earlier kernel writes and before
// writing anything, and mq_grid_release() so that their own dependents can start.
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, Args... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
    return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? MQ_OK : MQ_ERR_LAUNCH;
}

// Ordinary launch (no overlap with the previous kernel) through the same interface.
template <typename... KArgs, typename... Args>
int launch_plain(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
    return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? MQ_OK : MQ_ERR_LAUNCH;
}

// Device-side failure record (bounded waits) -----------------------------------
// Each translation unit with bounded waits owns one word; these read and clear it.
int take_gemm_device_error(cudaStream_t stream, unsigned* code);
int take_gemv_device_error(cudaStream_t stream, unsigned* code);

}  // namespace mq

// Device helpers -----------------------------------------------------------------

// Wait until the kernels this one depends on (programmatic launch) have completed
// and their writes are visible; a no-op for an ordinary launch.
__device__ __forceinline__ void mq_grid_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Let the next kernel on the stream be scheduled once every block of this one has
// called this (or exited).
__device__ __forceinline__ void mq_grid_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Loads of data that an earlier kernel on the stream writes (activation planes, producer
// inputs), made after mq_grid_wait(). A kernel launched with launch_pdl may start while
// that kernel is still running, so the data is not read-only for this kernel's lifetime
// and must not be read through the non-coherent path (ld.global.nc, __ldg): a replayed
// graph then read a stale plane. These are coherent loads that may be cached in L1.
// Weights, which no kernel in flight writes, may use __ldg; so may a kernel launched
// with launch_plain, which starts only after the previous kernel has completed.
__device__ __forceinline__ int4 mq_ld_dep(const int4* p) { return __ldca(p); }
__device__ __forceinline__ int2 mq_ld_dep(const int2* p) { return __ldca(p); }
__device__ __forceinline__ float2 mq_ld_dep(const float2* p) { return __ldca(p); }
__device__ __forceinline__ float4 mq_ld_dep(const float4* p) { return __ldca(p); }
__device__ __forceinline__ float mq_ld_dep(const float* p) { return __ldca(p); }

__device__ __forceinline__ float mq_f16_to_f32(uint16_t h) {
    float f;
    asm("{ .reg .f16 t; mov.b16 t, %1; cvt.f32.f16 %0, t; }" : "=f"(f) : "h"(h));
    return f;
}

// Packed pairs of f32 operations (the f32x2 instructions of sm_100 and later: one issue slot
// for two results). Each half is the correctly rounded result of the scalar operation, so
// packing changes no bit of any result; the compiler does not pair these by itself.
__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{ .reg .b64 ra, rb, rc, rd;\n\t mov.b64 ra, {%2, %3};\n\t mov.b64 rb, {%4, %5};\n\t mov.b64 rc, {%6, %7};\n\t"
        " fma.rn.f32x2 rd, ra, rb, rc;\n\t mov.b64 {%0, %1}, rd; }"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 f2_mul(float2 a, float2 b) {
    float2 d;
    asm("{ .reg .b64 ra, rb, rd;\n\t mov.b64 ra, {%2, %3};\n\t mov.b64 rb, {%4, %5};\n\t"
        " mul.rn.f32x2 rd, ra, rb;\n\t mov.b64 {%0, %1}, rd; }"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 f2_add(float2 a, float2 b) {
    float2 d;
    asm("{ .reg .b64 ra, rb, rd;\n\t mov.b64 ra, {%2, %3};\n\t mov.b64 rb, {%4, %5};\n\t"
        " add.rn.f32x2 rd, ra, rb;\n\t mov.b64 {%0, %1}, rd; }"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 f2_dup(float v) { return make_float2(v, v); }

// rint(v / d) with v / d the correctly rounded f32 quotient, computed as
// rint(v * inv) with inv an approximate 1/d (rcp.approx: at most 1 ulp off)
// unless that product lies within 6.2e-5 of a rounding boundary (n + 1/2), where
// the exact quotient is taken instead. For |v / d| <= 128 the product is within
// 128 * (2^-23 + 2^-24 + 2^-24) = 3.1e-5 of the rounded quotient (the reciprocal's
// error, the product's rounding and the quotient's), so both round to the same
// integer outside that band.
__device__ __forceinline__ int mq_rint_div(float v, float d, float inv) {
    const float t = v * inv;
    const float r = rintf(t);
    if (0.5f - fabsf(t - r) > 6.2e-5f) return (int)r;
    return __float2int_rn(__fdiv_rn(v, d));
}

// Quantize four f32 values that belong to one 32-block whose 8 owners are the
// lanes of one aligned 8-lane group. amax and the int sum are combined with xor
// shuffles at offsets 4, 2, 1 (max and integer sums are exact in any order).
// q = rint(v / d) with the correctly rounded quotient (see mq_rint_div).
// Returns the packed int8 quants; d and s are valid in every lane of the group.
// The band test is one warp vote for the warp's 128 values: the whole warp must call it together.
__device__ __forceinline__ uint32_t mq_quant4_group8(float v0, float v1, float v2, float v3,
                                                     float& d_out, int& s_out, int (&q)[4]) {
    float am = fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3)));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 4));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
    const float d = __fdiv_rn(am, 127.0f);
    float inv;
    asm("rcp.approx.f32 %0, %1;" : "=f"(inv) : "f"(d));
    int q0 = 0, q1 = 0, q2 = 0, q3 = 0;
    // Common case, one warp-uniform test for all four values of every lane: each product lies
    // outside the band around n + 1/2 (or the block is all zero), so rint of the product is
    // rint of the quotient (see mq_rint_div). Otherwise the lanes take the per-value path.
    const float2 t01 = f2_mul(make_float2(v0, v1), f2_dup(inv)), t23 = f2_mul(make_float2(v2, v3), f2_dup(inv));
    const float r0 = rintf(t01.x), r1 = rintf(t01.y), r2 = rintf(t23.x), r3 = rintf(t23.y);
    // t - r, exact (r is the integer nearest t)
    const float2 e01 = f2_fma(make_float2(r0, r1), f2_dup(-1.0f), t01);
    const float2 e23 = f2_fma(make_float2(r2, r3), f2_dup(-1.0f), t23);
    constexpr float kIn = 0.5f - 6.2e-5f;
    const bool clear = fabsf(e01.x) < kIn && fabsf(e01.y) < kIn && fabsf(e23.x) < kIn && fabsf(e23.y) < kIn;
    if (__all_sync(0xffffffffu, d == 0.0f || (isfinite(inv) && clear))) {
        // no clamp needed: |v| <= amax and d = amax / 127 rounded, so |t| stays within
        // 127 (1 + 2^-21) and its nearest integer within [-127, 127]
        if (d != 0.0f) {
            q0 = (int)r0;
            q1 = (int)r1;
            q2 = (int)r2;
            q3 = (int)r3;
        }
    } else if (d != 0.0f) {
        if (isfinite(inv)) {
            q0 = mq_rint_div(v0, d, inv);
            q1 = mq_rint_div(v1, d, inv);
            q2 = mq_rint_div(v2, d, inv);
            q3 = mq_rint_div(v3, d, inv);
        } else {   // d subnormal: 1/d overflows (rcp.approx keeps subnormal inputs)
            q0 = __float2int_rn(__fdiv_rn(v0, d));
            q1 = __float2int_rn(__fdiv_rn(v1, d));
            q2 = __float2int_rn(__fdiv_rn(v2, d));
            q3 = __float2int_rn(__fdiv_rn(v3, d));
        }
        q0 = max(-127, min(127, q0));
        q1 = max(-127, min(127, q1));
        q2 = max(-127, min(127, q2));
        q3 = max(-127, min(127, q3));
    }
    const uint32_t packed = (uint32_t)(q0 & 0xff) | ((uint32_t)(q1 & 0xff) << 8) | ((uint32_t)(q2 & 0xff) << 16) |
                            ((uint32_t)(q3 & 0xff) << 24);
    int s = __dp4a((int)packed, 0x01010101, 0);   // q0 + q1 + q2 + q3 from the signed bytes
    s += __shfl_xor_sync(0xffffffffu, s, 4);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    d_out = d;
    s_out = s;
    q[0] = q0;
    q[1] = q1;
    q[2] = q2;
    q[3] = q3;
    return packed;
}
