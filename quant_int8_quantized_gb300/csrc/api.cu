// Host-side helpers of the C ABI: sizes, status strings, architecture check,
// device-status query.

#include <map>
#include <mutex>
#include <tuple>

#include "mq_internal.cuh"

namespace mq {

namespace {
constexpr int kMaxDevices = 64;
int g_arch_ok[kMaxDevices];     // 0 unknown, 1 ok, 2 wrong arch
int g_sms[kMaxDevices];
std::mutex g_mu;
}  // namespace

int check_arch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MQ_ERR_ARCH;
    int v = __atomic_load_n(&g_arch_ok[dev], __ATOMIC_ACQUIRE);
    if (v == 0) {
        std::lock_guard<std::mutex> lk(g_mu);
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            return MQ_ERR_ARCH;
        }
        g_sms[dev] = sms;
        v = (major == 10 && minor == 3) ? 1 : 2;
        __atomic_store_n(&g_arch_ok[dev], v, __ATOMIC_RELEASE);
    }
    return v == 1 ? MQ_OK : MQ_ERR_ARCH;
}

int num_sms() {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= kMaxDevices) return 152;
    if (__atomic_load_n(&g_arch_ok[dev], __ATOMIC_ACQUIRE) == 0) check_arch();
    return g_sms[dev] > 0 ? g_sms[dev] : 152;
}

int resident_blocks(const void* kern, int threads, size_t smem) {
    static std::mutex mu;
    static std::map<std::tuple<const void*, int, int, size_t>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_tuple(kern, dev, threads, smem);
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, threads, smem) != cudaSuccess || b < 1) {
        cudaGetLastError();
        b = 1;
    }
    cache.emplace(key, b);
    return b;
}

}  // namespace mq

extern "C" size_t mq_plane_bytes(int M, int K, size_t* qs_bytes, size_t* d_bytes, size_t* s_bytes,
                                 size_t* ah_bytes, size_t* ax_bytes, size_t* af_bytes) {
    const size_t m = M > 0 ? (size_t)M : 0, k = K > 0 ? (size_t)K : 0;
    const size_t qs = m * k, d = m * (k / mq::QK) * sizeof(float), s = m * (k / mq::QK) * sizeof(int32_t);
    const size_t ah = m * k * sizeof(uint16_t), ax = m * (k / mq::QK_K) * 16 * sizeof(uint16_t);
    const size_t af = (k / mq::QK_K) * ((m + 3) & ~(size_t)3) * sizeof(float);
    if (qs_bytes) *qs_bytes = qs;
    if (d_bytes) *d_bytes = d;
    if (s_bytes) *s_bytes = s;
    if (ah_bytes) *ah_bytes = ah;
    if (ax_bytes) *ax_bytes = ax;
    if (af_bytes) *af_bytes = af;
    return qs + d + s + ah + ax + af;
}

extern "C" size_t mq_q4k_row_bytes(int K) { return K > 0 ? (size_t)(K / mq::QK_K) * mq::Q4K_BYTES : 0; }
extern "C" size_t mq_q6k_row_bytes(int K) { return K > 0 ? (size_t)(K / mq::QK_K) * mq::Q6K_BYTES : 0; }

extern "C" const char* mq_status_str(int status) {
    switch (status) {
        case MQ_OK: return "MQ_OK";
        case MQ_ERR_NULL: return "MQ_ERR_NULL: a required pointer is NULL";
        case MQ_ERR_SHAPE: return "MQ_ERR_SHAPE: invalid shape (K must be a positive multiple of 256; plane dims must match)";
        case MQ_ERR_ALIGN: return "MQ_ERR_ALIGN: a device pointer is not 16-byte aligned";
        case MQ_ERR_ARCH: return "MQ_ERR_ARCH: the current device is not a compute capability 10.3 GPU";
        case MQ_ERR_LAUNCH: return "MQ_ERR_LAUNCH: the CUDA launch failed";
        case MQ_ERR_DEVICE: return "MQ_ERR_DEVICE: a kernel gave up on a bounded wait";
        case MQ_ERR_SCRATCH: return "MQ_ERR_SCRATCH: the call needs more than the entry point's fixed scratch array holds";
        default: return "MQ_ERR_UNKNOWN";
    }
}

extern "C" int mq_device_status(cudaStream_t stream) {
    unsigned gemm = 0, gemv = 0;
    int rc = mq::take_gemm_device_error(stream, &gemm);
    if (rc == MQ_OK) rc = mq::take_gemv_device_error(stream, &gemv);
    if (rc != MQ_OK) return rc;
    return (gemm | gemv) ? MQ_ERR_DEVICE : MQ_OK;
}
