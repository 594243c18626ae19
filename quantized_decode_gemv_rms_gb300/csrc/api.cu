// api.cu -- process-wide state of the C ABI: device properties, options,
// launch counters, device flags, status strings and the block-sum test hook.
#include "common.cuh"

#include <atomic>
#include <map>
#include <mutex>
#include <utility>

namespace qdg {

static __device__ unsigned g_flags_api;

namespace {
std::mutex g_dev_mutex;
DeviceInfo g_dev_cache[64];
std::atomic<int> g_pdl{0};
std::atomic<int64_t> g_counts[15];
}  // namespace

DeviceInfo device_info() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return DeviceInfo{};
    }
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo& d = g_dev_cache[dev];
    if (d.device < 0) {
        int sms = 0, optin = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
            cudaGetLastError();
            return DeviceInfo{};
        }
        d.sms = sms;
        d.smem_optin = static_cast<size_t>(optin);
        d.device = dev;
    }
    return d;
}

// Waits on a barrier that nothing completes: the bounded wait must give up,
// set the timeout flag and return, leaving the context usable.
__global__ void timeout_probe_kernel() {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0)) atomicOr(&g_flags_api, FLAG_TIMEOUT);
}

unsigned flags_read_clear_api(cudaStream_t stream) {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_flags_api, sizeof(v), 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return ~0u;
    if (cudaMemcpyToSymbolAsync(g_flags_api, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream) !=
        cudaSuccess)
        return ~0u;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return ~0u;
    return v;
}

cudaError_t ensure_smem_limit(const void* func, size_t bytes) {
    static std::mutex mu;
    static std::map<std::pair<int, const void*>, size_t> done;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    size_t& have = done[std::make_pair(dev, func)];
    if (have >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e == cudaSuccess) have = bytes;
    return e;
}

bool pdl_enabled() { return g_pdl.load(std::memory_order_relaxed) != 0; }

void count_launch(int which) { g_counts[which].fetch_add(1, std::memory_order_relaxed); }

}  // namespace qdg

using namespace qdg;

extern "C" int qdg_set_option(int option, int64_t value) {
    if (option == QDG_OPT_PDL) {
        if (value != 0 && value != 1) return QDG_EINVAL;
        g_pdl.store(static_cast<int>(value));
        return QDG_OK;
    }
    return QDG_EINVAL;
}

extern "C" int64_t qdg_launch_count(int which) {
    if (which == -1) {
        int64_t t = 0;
        for (auto& c : g_counts) t += c.load();
        return t;
    }
    if (which < 0 || which >= 15) return -1;
    return g_counts[which].load();
}

extern "C" const char* qdg_status_string(int status) {
    switch (status) {
        case QDG_OK: return "ok";
        case QDG_EINVAL: return "invalid argument (null pointer, size or option)";
        case QDG_EALIGN: return "misaligned pointer or leading dimension";
        case QDG_ESHAPE: return "unsupported shape (K multiple or maximum size)";
        case QDG_ECUDA: return "CUDA runtime error";
        case QDG_ETIMEOUT: return "a bounded device-side wait gave up; output incomplete";
        case QDG_EOVERFLOW: return "a Q8_0 scale overflowed fp16";
        default: return "unknown status";
    }
}

extern "C" int qdg_device_status(qdg_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return QDG_ECUDA;
    }
    unsigned f = 0;
    const unsigned parts[] = {flags_read_clear_quantize(s), flags_read_clear_gemv(s), flags_read_clear_gemv_seg(s),
                              flags_read_clear_small_n(s), flags_read_clear_small_n_seg(s),
                              flags_read_clear_gemm(s), flags_read_clear_api(s),
                              flags_read_clear_chain(s), flags_read_clear_gemv_q4k(s),
                              flags_read_clear_gemv_segn(s)};
    for (unsigned p : parts) {
        if (p == ~0u) {
            cudaGetLastError();
            return QDG_ECUDA;
        }
        f |= p;
    }
    if (f & FLAG_TIMEOUT) return QDG_ETIMEOUT;
    if (f & FLAG_OVERFLOW) return QDG_EOVERFLOW;
    return QDG_OK;
}

extern "C" int qdg_debug_block_sums(const void* W, const void* xq, int32_t* isum, int64_t O, int64_t K, int64_t N,
                                    int path, qdg_stream_t stream) {
    if (!isum) return QDG_EINVAL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    switch (path) {
        case 0:
            if (N != 1) return QDG_EINVAL;
            return gemv_launch(W, xq, nullptr, O, K, s, isum);
        case 1:
            return small_n_launch(W, xq, nullptr, O, O, K, N, s, isum);
        case 2: {
            // test hook: its own workspace, released after the launches complete
            const int64_t bytes = gemm_workspace_bytes(K, N);
            if (bytes < 0) return static_cast<int>(bytes);
            void* ws = nullptr;
            if (cudaMalloc(&ws, static_cast<size_t>(bytes)) != cudaSuccess) return QDG_ECUDA;
            int rc = gemm_launch(W, xq, nullptr, O, O, K, N, ws, bytes, s, isum);
            if (cudaStreamSynchronize(s) != cudaSuccess && rc == QDG_OK) rc = QDG_ECUDA;
            cudaFree(ws);
            return rc;
        }
        case 3:
            if (N != 1) return QDG_EINVAL;
            return gemv_seg_launch(W, xq, nullptr, O, K, s, isum);
        case 4:
            if (N != 1) return QDG_EINVAL;
            return gemv_q8w_launch(W, xq, nullptr, O, K, s, isum);
        case 6:
            if (N != 1) return QDG_EINVAL;
            return gemv_q4k_launch(W, xq, nullptr, O, K, s, isum);
        case 7:
            if (N != 1) return QDG_EINVAL;
            return gemv_q5k_launch(W, xq, nullptr, O, K, s, isum);
        case 5:
            if (N == 1) return gemv_seg_launch(W, xq, nullptr, O, K, s, isum);
            if (N == 2) return gemv_seg2_launch(W, xq, nullptr, O, O, K, s, isum);
            if (gemv_segn_supported(K, N)) return gemv_segn_launch(W, xq, nullptr, O, O, K, N, s, isum);
            return small_n_seg_launch(W, xq, nullptr, O, O, K, N, s, isum);
        default:
            return QDG_EINVAL;
    }
}

extern "C" int qdg_debug_timeout_probe(qdg_stream_t stream) {
    timeout_probe_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>();
    return cudaGetLastError() == cudaSuccess ? QDG_OK : QDG_ECUDA;
}
