/*
 * mq.h — C ABI of the GB300 (sm_103a) block-quantized matmul library (libmq.so).
 *
 * The library computes the hot path of GGML-style quantized LLM inference:
 * activations quantized to int8 blocks of 32 (a "q8 plane"), produced either
 * standalone or fused into RMSNorm / SwiGLU, multiplied against q4_K / q6_K
 * weight super-blocks (prefill GEMM, decode GEMV).
 *
 * Sources (engineering write-ups of the "minfer" inference engine):
 *   [r60]  "64 · r60 — the coronation: flipping the verified gate set to default-on"
 *   [r52]  "55 · r52 — skip-write mode 2: skipping the f32 intermediate write-out"
 *   [D3-7] "72 · D3-7 — attn_v-q6K MMVQ routing (2b) + rms wide-block / positions memo (2c)"
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Dimensions: M = tokens (activation rows), K = input features (the
 *    reduction axis, "id" on the pages), N = output features ("od").
 *  - Every pointer argument that names tensor data is a DEVICE pointer on the
 *    current CUDA device. The caller allocates and owns every buffer. The
 *    library never allocates, frees or synchronizes; it only enqueues kernels
 *    (and, for a split GEMM, a memset of part of its output) asynchronously on
 *    `stream` (0 = legacy default stream).
 *  - Inputs are read only. Outputs (planes, out) are overwritten, never
 *    accumulated into.
 *  - Stream order holds as for any CUDA work: a call's memory accesses come after
 *    the work enqueued before it on `stream` and before the work enqueued after
 *    it. The producers and the prefill GEMMs are programmatic dependent launches:
 *    their set-up may overlap the end of the previous kernel on the stream, but
 *    they touch no global memory before that kernel has completed.
 *  - K must be a positive multiple of 256 (one weight super-block; it also
 *    gives the producers whole 8-lane groups, [r52] §3.2). M == 0 or N == 0 is
 *    a no-op returning MQ_OK.
 *  - Alignment: every device pointer must be 16-byte aligned.
 *  - Return value: MQ_OK, or an MQ_ERR_* code from host-side validation,
 *    returned before anything is launched, or MQ_ERR_LAUNCH when the launch
 *    itself failed. There is no fallback path. Kernel faults surface, as with
 *    any CUDA work, at the next synchronizing call.
 */
#ifndef MQ_H
#define MQ_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    MQ_OK = 0,
    MQ_ERR_NULL = 1,    /* a required pointer is NULL */
    MQ_ERR_SHAPE = 2,   /* K not a positive multiple of 256, negative M/N, plane dims mismatch, GEMV M outside [1, 8] */
    MQ_ERR_ALIGN = 3,   /* a pointer is not 16-byte aligned */
    MQ_ERR_ARCH = 4,    /* the current device is not a compute capability 10.3 (GB300) GPU */
    MQ_ERR_LAUNCH = 5,  /* the CUDA launch (or tensor-map encoding) failed */
    MQ_ERR_DEVICE = 6,  /* a kernel gave up on a bounded wait (reported by mq_device_status) */
    MQ_ERR_SCRATCH = 7  /* mq_gemm_q6k_static: the call needs more than its fixed scratch array holds */
};

/* Most activation rows one mq_gemv_q4k / mq_gemv_q6k call takes. */
#define MQ_GEMV_MAX_ROWS 8

/*
 * q8 activation plane ([r52] §2.2; [D3-7] Excerpt C): for each row m and each
 * block b of 32 consecutive elements, int8 quants qs, an f32 scale d and the
 * int32 sum of the block's quants s:
 *     qs : int8     [M][K]      row-major, row stride K bytes
 *     d  : float    [M][K/32]   row-major
 *     s  : int32_t  [M][K/32]   row-major
 * The prefill GEMM multiplies on the f16 tensor pipe and reads the activations
 * in an operand form derived from the same quants (the library's reading; the
 * pages' GEMM reads the int8 plane). Per row m and super-block t of 256
 * (blocks 8t .. 8t+7), with D = the largest of the 8 block scales and
 * e = 3 - E where D = f * 2^E, f in [1/2, 1) (so D * 2^e lies in [4, 8); e is
 * clamped to [-126, 126], and e = 0 when D == 0):
 *     ah : uint16_t [M][K]        binary16 bit patterns of f16(f32(d * q) * 2^e)
 *                                 (|ah| < 1016);
 *     ax : uint16_t [M][K/256][16] binary16: for block j of the super-block,
 *                                 slot j = f16(sigma_j) and slot 8+j =
 *                                 f16(sigma_j - slot j), sigma_j the exact f32
 *                                 sum of the block's 32 ah values;
 *     af : float    [K/256][Mp]   2^-e, Mp = M rounded up to a multiple of 4
 *                                 (entries of rows >= M are not written).
 * 2^-e * ah equals d * q to within 2^-11 relative (binary16 normal range).
 * A plane holds the q8 arrays (qs, d, s), the operand arrays (ah, ax, af), or
 * both; each group is all present or all NULL. Producers write every array
 * that is present. The GEMV reads the q8 arrays, the GEMM the operand arrays.
 * The plane is a pure function of the f32 values it quantizes, so one plane
 * may feed several GEMMs (Q/K/V, gate/up). The library reads only rows < M.
 * The struct lives in host memory; only its pointers are device pointers.
 */
typedef struct mq_q8_plane {
    int8_t*   qs;
    float*    d;
    int32_t*  s;
    uint16_t* ah;
    uint16_t* ax;
    float*    af;
    int M;
    int K;
} mq_q8_plane;

/* Bytes of each plane array for an M x K activation (any output pointer may be
 * NULL). Returns the sum of all six. Pure host helper. */
size_t mq_plane_bytes(int M, int K, size_t* qs_bytes, size_t* d_bytes, size_t* s_bytes,
                      size_t* ah_bytes, size_t* ax_bytes, size_t* af_bytes);

/*
 * Bytes of one weight row (K/256 super-blocks):
 *   q4_K super-block, 144 B: f16 d, f16 dmin, 12 B of packed 6-bit scales and
 *     mins for eight 32-element sub-blocks, 128 B of 4-bit quants;
 *   q6_K super-block, 210 B: 128 B low 4 bits, 64 B high 2 bits, 16 int8
 *     scales (one per 16 elements), f16 d.
 * ([r60] §3.2 names the types; the byte order is the library's documented
 * reading, the public GGUF order.) Weights are N rows x K/256 super-blocks, row-major,
 * rows packed back to back (row stride = the value returned here).
 */
size_t mq_q4k_row_bytes(int K);
size_t mq_q6k_row_bytes(int K);

/*
 * Prepacked q6_K (the prefill GEMM's weight form): the same super-blocks re-laid
 * out once, at weight registration ([r60] §1 and §3.2, registration-time layouts;
 * [D3-7] Excerpt A, padded q6_K blocks), into 224-byte blocks, so that every
 * block starts on a 16-byte boundary and each half of it is contiguous. Half h
 * (h = 0, 1) of a packed block, at byte 112*h:
 *     64 bytes  raw ql[64h .. 64h+63]   (low 4 bits)
 *     32 bytes  raw qh[32h .. 32h+31]   (high 2 bits)
 *      8 bytes  raw scales[8h .. 8h+7]  (int8)
 *      2 bytes  d (f16), then 6 zero bytes.
 * mq_q6k_packed_row_bytes(K) = K/256 * 224. mq_prepack_q6k reads N raw rows (w,
 * 2-byte aligned, N*K/256*210 bytes) and writes N packed rows (packed, 16-byte
 * aligned, caller-owned) on `stream`. Returns MQ_ERR_SHAPE for K not a positive
 * multiple of 256 or N < 0.
 */
size_t mq_q6k_packed_row_bytes(int K);
int mq_prepack_q6k(const void* w, int N, int K, void* packed, cudaStream_t stream);

/*
 * mq_quantize_q8 — standalone activation quantization ([r52] §2.2; [D3-7]
 * Excerpt C, the per-32-block epilogue; [D3-7] Excerpt A2, the decode
 * quantize). x: f32 [M][K] row-major. For every block of 32:
 *     amax = max|v|; d = amax / 127 (f32); q = rint(v / d) (IEEE f32 divide,
 *     ties to even) clamped to [-127, 127]; s = sum q; an all-zero block gives
 *     d = 0, q = 0, s = 0.
 * Every producer writes whichever of the plane's array groups are present
 * (the q8 arrays, the operand arrays, or both).
 * out->M, out->K must equal M, K. Input values must be finite.
 */
int mq_quantize_q8(const float* x, int M, int K, const mq_q8_plane* out, cudaStream_t stream);

/*
 * mq_rms_quant — fused RMSNorm -> q8 plane that never writes the f32
 * normalized rows ([r52] §3.2, the mode-2 rms kernel; [D3-7] §2c(i) and
 * Excerpt C for the single-row decode shape). x: f32 [M][K], w: f32 [K].
 *     ss = sum x^2 in a fixed order (32 lane partials over float4 l, l+32, ...;
 *          each float4 adds ((x0*x0 + x1*x1) + x2*x2) + x3*x3; xor butterfly),
 *     scale = 1 / sqrt(ss / K + eps) (correctly rounded f32 ops),
 *     v = (x * scale) * w, then the mq_quantize_q8 block rule on v.
 * The result is bit-identical to quantizing the f32 RMSNorm output computed in
 * that order.
 */
int mq_rms_quant(const float* x, const float* w, int M, int K, float eps,
                 const mq_q8_plane* out, cudaStream_t stream);

/*
 * mq_swiglu_quant — fused SwiGLU -> q8 plane that never writes the f32
 * product ([r52] §3.2, the mode-2 swiglu kernel). g, u: f32 [M][K].
 *     v = (g / (1 + exp(-g))) * u, then the mq_quantize_q8 block rule on v.
 * The division is IEEE f32. exp is fixed bit for bit, since an f32 exp has no
 * single correct result: Cody-Waite range reduction (n = rint(x log2 e),
 * r = (x - n ln2_hi) - n ln2_lo, as two fused multiply-adds) and the degree-7
 * Taylor series in Horner form (one fused multiply-add a step), each step one
 * correctly rounded f32 operation, scaled exactly by 2^n; 0 below x = -86,
 * +inf above x = 88; within 0.91 ulp of e^x. The plane is thus a function of g
 * and u alone, like the other producers' planes.
 */
int mq_swiglu_quant(const float* g, const float* u, int M, int K,
                    const mq_q8_plane* out, cudaStream_t stream);

/*
 * mq_gemm_q4k / mq_gemm_q6k — prefill matmul of a plane by super-block weights
 * ([r60] §3.1 and §3.2, the MMQ dispatch for nt >= 16; q6_K runs each 32-wide
 * chunk as two 16-element halves with their own int8 scales):
 *     out[m][n] = sum_k (d_a[m][k/32] * q_a[m][k]) * w[n][k]
 * with w the dequantized weight (q4_K: d*sc*q - dmin*m per 32; q6_K:
 * d*sc*(q-32) per 16). a: plane with a->M >= 1 rows, a->K = K and its operand
 * arrays (ah, ax, af; MQ_ERR_NULL otherwise); w: N rows of super-blocks, q4_K
 * in the raw layout above, q6_K in the prepacked layout (mq_prepack_q6k); out:
 * f32 [a->M][N] row-major, overwritten. Any M >= 1 is accepted (the kernel is
 * built for M >= 16).
 * Arithmetic: per 256-wide super-block, the f16 tensor pipe multiplies the
 * binary16 activations ah by the exact integer weight operands (q4_K sc*q,
 * q6_K sc*(q-32) in two parts) and, for q4_K, the min term's exact block sums
 * by -dmin/d*m in hi + lo parts, accumulating in f32; the result is scaled by
 * d * 2^-e. Accuracy: within 1e-3 * sum_k |a||w| per element (the binary16
 * activation contributes at most 2^-11 of it).
 * When the output has fewer 192-token x 128-row tiles than the GPU has SMs
 * (small M or N), the K axis is split across several thread blocks, `out` is
 * zeroed on `stream` and the partial sums are added with f32 atomics: the result
 * is then within the same bound, but its last bits may differ from run to run.
 * mq_gemm_q6k with more tiles than SMs but not a whole number of rounds of them
 * may make two launches: the tiles of the complete rounds whole, then (a
 * programmatic dependent launch on `stream`) the rest cut along K into slices
 * that add into `out` in a fixed order; the result is the same on every run (on
 * a GPU with the same SM count). The hand-over uses flags in the library's own
 * device memory and bounded waits (mq_device_status reports a wait given up).
 */
int mq_gemm_q4k(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream);
int mq_gemm_q6k(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream);

/*
 * mq_gemm_q4k_pair — two q4_K GEMMs that read the same activation plane (the same M and K,
 * e.g. attn_q and attn_k, or ffn_gate and ffn_up: [r52] §2.2's one plane feeding several
 * projections), out0 = a x w0 (N0 rows) and out1 = a x w1 (N1 rows), each exactly as
 * mq_gemm_q4k computes it (the same bits, for tiles that mq_gemm_q4k would not split along
 * K). When both have whole 192-token tiles (M >= 192) and together fill at least one round of
 * the GPU's SMs, they run in one launch, the second problem's tiles filling what the first
 * leaves idle and the pair paying one launch's fixed cost; otherwise the call makes two
 * mq_gemm_q4k calls. Arguments, accuracy and errors as for mq_gemm_q4k, for each problem;
 * MQ_ERR_SHAPE also if out0 and out1 overlap.
 */
int mq_gemm_q4k_pair(const mq_q8_plane* a, const void* w0, int N0, float* out0, const void* w1, int N1,
                     float* out1, cudaStream_t stream);

/*
 * mq_gemm_q6k_static — mq_gemm_q6k for callers that cannot have device memory allocated on
 * their behalf: a server that hands all device memory to its own pool at start-up, or code
 * that must not call cudaMalloc because it can synchronize the device and stall other work.
 * The pages have no counterpart; this is a property of this library's interface only.
 * Same arguments, result, accuracy and errors as mq_gemm_q6k. Where mq_gemm_q6k's ordered
 * split takes its flags from a ring shared by all its launches, this variant uses a fixed
 * array of its own of 1024 flags (4 KB of device memory, held by every GPU that loads the
 * library until the process exits; one flag per tile the split cuts). It clears the flags it
 * uses on `stream` at every call. A call that would need more than 1024 of them returns
 * MQ_ERR_SCRATCH before anything is enqueued. Calls share the array, so two calls that run
 * on the GPU at the same time (on different streams) race and may give wrong results. The
 * first call on a device looks the array's device address up (once per device); make that
 * first call before any stream capture. It calls no cudaMalloc or cudaFree.
 */
int mq_gemm_q6k_static(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream);

/*
 * mq_gemm_q4_0 / mq_gemm_q4_1 — the same prefill matmul for the Q4_0 / Q4_1 types
 * of the matmul dispatch list ([r60] §3.2), with w in the raw layouts given at
 * mq_gemv_q4_0 below (18 / 20 bytes per 32 weights, rows 16-byte aligned since K
 * is a multiple of 256). Arguments, output, split-K and errors as for mq_gemm_q4k.
 * Arithmetic: per 256-wide super-block and weight row, a power of two c; block b's
 * scale d_b = g_b 2^E_b (g_b its 11-bit integer significand) is split
 * g_b = 64 Dh + Dl, and each weight d_b (q - o) / c enters the f16 tensor pipe as
 * the two exact binary16 parts (q - o) Dh 2^(E_b+6) / c and (q - o) Dl 2^E_b / c
 * (o = 8 for q4_0, 0 for q4_1), two MMAs per K step; q4_1's m_b / c multiplies the
 * plane's exact block sums like q4_K's min term. The weight operand is exact
 * while a super-block's block scales lie within a factor 2^24 of each other;
 * accuracy within 1e-3 * sum_k |a||w| per element.
 */
int mq_gemm_q4_0(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream);
int mq_gemm_q4_1(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream);

/*
 * mq_gemv_q4k / mq_gemv_q6k — decode (M == 1) and small-batch
 * (1 <= M <= MQ_GEMV_MAX_ROWS) matrix products ([D3-7] §2 (2b) and Excerpt
 * A/A2, the MMVQ decode path): the same result as the GEMM, within the same
 * bound. Integer dp4a block dots on the plane's q8 arrays (qs, d, s must be
 * present; the operand arrays are not read). Each weight super-block is loaded
 * and decoded once and dotted with every activation row, so a call streams the
 * weights once whatever M is.
 *   w   : raw q4_K / q6_K rows, N * (K/256) * 144 or 210 bytes (the q6_K GEMV
 *         reads the raw layout, not mq_prepack_q6k's), 16-byte aligned.
 *   out : f32 [M][N] row-major, written (not accumulated).
 * Returns MQ_ERR_SHAPE if a->M is outside [1, MQ_GEMV_MAX_ROWS]. Between one row
 * and the GEMM's region the caller picks the faster call per M: the GEMV's cost
 * grows with M (its integer dot work), the GEMM's does not below 16 rows.
 *
 * Launch overlap: the three producers above are launched with programmatic
 * stream serialization, so each may start while the kernel enqueued before it
 * on `stream` is finishing. Each waits for that kernel to complete before it
 * reads its inputs (with coherent loads) and before it writes anything, so
 * chains of these calls keep stream order. The RMSNorm weight `w` is read
 * through the read-only path: it must not be written by a kernel still running
 * when mq_rms_quant's kernel starts (an event wait or a synchronization between
 * the two suffices; weights written by cudaMemcpy* or before the stream work
 * began are always safe). The GEMVs, the GEMMs and mq_prepack_q6k are ordinary
 * launches.
 */
int mq_gemv_q4k(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream);
int mq_gemv_q6k(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream);

/*
 * mq_gemv_q6k_packed — mq_gemv_q6k on prepacked rows: w is mq_prepack_q6k's output
 * (N * (K/256) * 224 bytes, 16-byte aligned), the weight form the q6_K GEMM reads, so
 * one registered copy of a q6_K matrix serves prefill and decode ([r60] §1, weights
 * re-laid out once at registration; [D3-7] §2 (2b) and Excerpt A, the q6_K decode
 * arm). Every super-block is 16-byte aligned, so the rows are read with aligned
 * 16-byte loads straight into registers. Same arguments, result bound and errors as
 * mq_gemv_q6k; the same products are summed in another order.
 */
int mq_gemv_q6k_packed(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream);

/*
 * mq_gemv_q5k / mq_gemv_q4_0 / mq_gemv_q4_1 — the same decode / small-batch
 * product for the other block types the pages dispatch: q5_K in the decode
 * arm ([D3-7] Excerpt B), Q4_0 / Q4_1 in the matmul dispatch list ([r60]
 * §3.2). The pages name these types but print no layout; the library reads the
 * GGUF blocks of those names:
 *   q5_K : 176 bytes per 256 elements — d (f16), dmin (f16), the 12-byte
 *          scale/min field packed as in q4_K, 32 bytes qh, 128 bytes of
 *          nibbles. Element 64j + l (l < 32) is the low nibble of byte 32j + l
 *          plus 16 * (bit 2j of qh[l]); element 64j + 32 + l the high nibble plus
 *          16 * (bit 2j + 1 of qh[l]). w = d * sc * q - dmin * m.
 *   q4_0 : 18 bytes per 32 elements — d (f16), 16 bytes; element l < 16 is the
 *          low nibble of byte l, element 16 + l its high nibble. w = d * (q - 8).
 *   q4_1 : 20 bytes per 32 elements — d (f16), m (f16), 16 bytes as q4_0.
 *          w = d * q + m.
 * Row bytes: mq_q5k_row_bytes(K) = K/256 * 176, mq_q4_0_row_bytes(K) = K/32 * 18,
 * mq_q4_1_row_bytes(K) = K/32 * 20. Arguments, errors and the 1..8 rows of `a`
 * as for mq_gemv_q4k; out f32 [M][N]; within the same bound.
 */
size_t mq_q5k_row_bytes(int K);
size_t mq_q4_0_row_bytes(int K);
size_t mq_q4_1_row_bytes(int K);
int mq_gemv_q5k(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream);
int mq_gemv_q4_0(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream);
int mq_gemv_q4_1(const mq_q8_plane* a, const void* w, int N, float* out, cudaStream_t stream);

/*
 * mq_device_status — synchronizes `stream`, then returns MQ_OK if no kernel of
 * this library launched so far on the current device has given up on a
 * bounded wait, else MQ_ERR_DEVICE, and clears the record. Returns
 * MQ_ERR_LAUNCH if the synchronization itself reports a CUDA error.
 */
int mq_device_status(cudaStream_t stream);

/* Human-readable name of a status code (static string, never NULL). */
const char* mq_status_str(int status);

#ifdef __cplusplus
}
#endif

#endif /* MQ_H */
