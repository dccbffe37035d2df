// Registration-time weight prepack: q6_K super-blocks re-laid out for the prefill GEMM.
//
// The pages re-lay their weights once at registration for their kernels ("64 · r60 —
// the coronation", §1 and §3.2; "72 · D3-7", Excerpt A's padded q6_K blocks with a
// padded block stride). A raw q6_K super-block is 210 bytes, so rows of them are only
// 2-byte aligned and cannot be staged by TMA. The packed block is 224 bytes (16-byte
// aligned) and keeps each half of the super-block together: at 112 h, half h holds
// its 64 low-bit bytes (raw ql[64h ..]), its 32 high-bit bytes (raw qh[32h ..]), its 8
// int8 scales (raw scales[8h ..]), the f16 d and 6 zero bytes. The element values and
// their order are unchanged; only the bytes move.

#include "mq_internal.cuh"

namespace {

constexpr int kChunks = mq::Q6K_PACKED_BYTES / 16;   // 14 output chunks of 16 bytes per block

// One thread per 16-byte output chunk. The raw block is 2-byte aligned: it is read in
// 16-bit pieces.
__global__ void prepack_q6k_kernel(const uint16_t* __restrict__ raw, uint4* __restrict__ out, long long blocks) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= blocks * kChunks) return;
    const long long blk = i / kChunks;
    const int c = (int)(i - blk * kChunks), h = c / 7, cc = c - 7 * h;
    const uint16_t* src = raw + blk * (mq::Q6K_BYTES / 2);   // 105 pieces per raw block
    uint32_t w[4] = {0, 0, 0, 0};
    auto pick = [&](int byte_off, int npieces) {               // npieces 16-bit pieces into w
        for (int k = 0; k < npieces; ++k) w[k >> 1] |= (uint32_t)__ldg(src + byte_off / 2 + k) << (16 * (k & 1));
    };
    if (cc < 4) pick(64 * h + 16 * cc, 8);                     // ql
    else if (cc < 6) pick(128 + 32 * h + 16 * (cc - 4), 8);    // qh
    else {
        pick(192 + 8 * h, 4);                                  // scales
        w[2] = __ldg(src + 104);                               // d (raw bytes 208, 209)
    }
    out[i] = make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace

extern "C" size_t mq_q6k_packed_row_bytes(int K) {
    return K > 0 ? (size_t)(K / mq::QK_K) * mq::Q6K_PACKED_BYTES : 0;
}

extern "C" int mq_prepack_q6k(const void* w, int N, int K, void* packed, cudaStream_t stream) {
    if (N < 0 || !mq::valid_k(K)) return MQ_ERR_SHAPE;
    if (N == 0) return MQ_OK;
    if (!w || !packed) return MQ_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(w) & 1u) || !mq::aligned16(packed)) return MQ_ERR_ALIGN;
    const int rc = mq::check_arch();
    if (rc != MQ_OK) return rc;
    const long long blocks = (long long)N * (K / mq::QK_K);
    const long long threads = blocks * kChunks;
    return mq::launch_plain(prepack_q6k_kernel, dim3((unsigned)((threads + 255) / 256)), dim3(256), 0, stream,
                            static_cast<const uint16_t*>(w), static_cast<uint4*>(packed), blocks);
}
