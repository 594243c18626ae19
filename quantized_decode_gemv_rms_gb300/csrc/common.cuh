// common.cuh -- shared device helpers of the sm_103a kernels: status flags,
// hand-written PTX for mbarriers, bulk asynchronous copies and programmatic
// dependent launch, and the host-side validation helpers of the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <cmath>

#include "../../include/qdg.h"

namespace qdg {

// Device flag bits (per translation unit; qdg_device_status gathers them).
enum : unsigned { FLAG_TIMEOUT = 1u, FLAG_OVERFLOW = 2u };

// A wait gives up after kWaitNs nanoseconds of the global timer, or after
// kSpinLimit polls, whichever comes first (legitimate waits take microseconds).
constexpr uint32_t kSpinLimit = 1u << 24;
constexpr uint64_t kWaitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the asynchronous (bulk copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// As mbar_try_wait, but the thread may stay suspended (issuing nothing) for
// up to kSuspendNs while the phase is incomplete; it resumes as soon as the
// phase completes.
constexpr uint32_t kSuspendNs = 1000000;
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for the phase of `parity` to complete.  False = gave up.
// Each try suspends the thread in hardware until the phase completes (or up
// to kSuspendNs), so waiting warps take no issue slots from working ones.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1; i < kSpinLimit; ++i) {
        if (mbar_try_wait_suspend(bar, parity)) return true;
        if (global_ns() - t0 > kWaitNs) return false;
    }
    return false;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 1-D bulk copy global -> shared (TMA engine), completion counted in bytes
// on `bar`.  dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// The same without a cache policy.
__device__ __forceinline__ void bulk_g2s_plain(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// 16-byte asynchronous copy global -> shared, cached in L2 only (so it reads
// what other CTAs wrote before a grid-wide synchronisation); completes at
// cp_async_wait_all of the same thread.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Programmatic dependent launch: wait for the preceding grid's memory, and
// allow the following grid to be scheduled.  No-ops without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ float half_bits_to_float(uint32_t bits16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xFFFFu)));
}

// Bytes 2..5 of the 8-byte little-endian pair (lo, hi).
__device__ __forceinline__ uint32_t bytes_2_to_5(uint32_t lo, uint32_t hi) { return __byte_perm(lo, hi, 0x5432); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int h = 16; h >= 1; h >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, h));
    return v;
}

// (a0, a1) += (s0, s1) * (v0, v1), one packed fp32x2 fused multiply-add.
__device__ __forceinline__ void ffma2(float& a0, float& a1, float s0, float s1, float v0, float v1) {
    asm("{\n\t.reg .b64 s, v, a;\n\t"
        "mov.b64 s, {%2, %3};\n\tmov.b64 v, {%4, %5};\n\tmov.b64 a, {%0, %1};\n\t"
        "fma.rn.f32x2 a, s, v, a;\n\tmov.b64 {%0, %1}, a;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(s0), "f"(s1), "f"(v0), "f"(v1));
}

// (d0, d1) = (a0, a1) * (b0, b1), packed fp32x2.
__device__ __forceinline__ void fmul2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 a, b, d;\n\t"
        "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// ---------------------------------------------------------------- host side
inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct DeviceInfo {
    int device = -1;
    int sms = 0;
    size_t smem_optin = 0;
};

// Per-device properties, cached (one GPU per process in practice).
DeviceInfo device_info();

bool pdl_enabled();
void count_launch(int which);

// Raise `func`'s dynamic shared-memory limit to at least `bytes` on the
// current device.  The attribute belongs to a (device, kernel) pair, so the
// record of what was set is kept per device; later calls that need no more
// than was set cost one map lookup.
cudaError_t ensure_smem_limit(const void* func, size_t bytes);

// Launch with the PDL attribute when enabled.
template <typename Kern, typename... Args>
cudaError_t launch(Kern kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool allow_pdl,
                   Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    cfg.attrs = attr;
    cfg.numAttrs = 0;
    if (allow_pdl && pdl_enabled()) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Launch as clusters of `cluster` CTAs along x (1 = no cluster attribute),
// with the PDL attribute when enabled.
template <typename Kern, typename... Args>
cudaError_t launch_cluster(Kern kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool allow_pdl,
                           int cluster, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    cfg.attrs = attr;
    cfg.numAttrs = 0;
    if (cluster > 1) {
        attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
        attr[cfg.numAttrs].val.clusterDim.x = static_cast<unsigned>(cluster);
        attr[cfg.numAttrs].val.clusterDim.y = 1;
        attr[cfg.numAttrs].val.clusterDim.z = 1;
        ++cfg.numAttrs;
    }
    if (allow_pdl && pdl_enabled()) {
        attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
        ++cfg.numAttrs;
    }
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Internal launchers shared with the debug hook (dbg != nullptr writes the
// exact per-block integer sums [N][O][K/32] as the kernel forms them).
int gemv_launch(const void* W, const void* xq, float* y, int64_t O, int64_t K, cudaStream_t stream,
                int32_t* dbg);
int gemv_q8w_launch(const void* W, const void* xq, float* y, int64_t O, int64_t K, cudaStream_t stream,
                    int32_t* dbg);
int gemv_q4k_launch(const void* W, const void* xq, float* y, int64_t O, int64_t K, cudaStream_t stream,
                    int32_t* dbg);
int gemv_q5k_launch(const void* W, const void* xq, float* y, int64_t O, int64_t K, cudaStream_t stream,
                    int32_t* dbg);
int gemv_seg2_launch(const void* W, const void* xq, float* y, int64_t ldy, int64_t O, int64_t K,
                     cudaStream_t stream, int32_t* dbg);
int gemv_seg_launch(const void* W, const void* xq, float* y, int64_t O, int64_t K, cudaStream_t stream,
                    int32_t* dbg);
int small_n_launch(const void* W, const void* xq, float* y, int64_t ldy, int64_t O, int64_t K, int64_t N,
                   cudaStream_t stream, int32_t* dbg);
int small_n_seg_launch(const void* W, const void* xq, float* y, int64_t ldy, int64_t O, int64_t K, int64_t N,
                       cudaStream_t stream, int32_t* dbg);
// three or four vectors on the segment layout by dp4a (one block a lane), K <= 16384
bool gemv_segn_supported(int64_t K, int64_t N);
int gemv_segn_launch(const void* W, const void* xq, float* y, int64_t ldy, int64_t O, int64_t K, int64_t N,
                     cudaStream_t stream, int32_t* dbg);
int64_t gemm_workspace_bytes(int64_t K, int64_t T);
int chain_launch(const qdg_chain_stage* stages, int nstages, float eps, void* sync, cudaStream_t stream);
int gemm_launch(const void* W, const void* xq, float* y, int64_t ldy, int64_t O, int64_t K, int64_t T, void* ws,
                int64_t ws_bytes, cudaStream_t stream, int32_t* dbg);

// Per-translation-unit device flags: read and clear (synchronises stream).
unsigned flags_read_clear_quantize(cudaStream_t stream);
unsigned flags_read_clear_gemv(cudaStream_t stream);
unsigned flags_read_clear_gemv_seg(cudaStream_t stream);
unsigned flags_read_clear_small_n(cudaStream_t stream);
unsigned flags_read_clear_small_n_seg(cudaStream_t stream);
unsigned flags_read_clear_gemm(cudaStream_t stream);
unsigned flags_read_clear_api(cudaStream_t stream);
unsigned flags_read_clear_chain(cudaStream_t stream);
unsigned flags_read_clear_gemv_q4k(cudaStream_t stream);
unsigned flags_read_clear_gemv_segn(cudaStream_t stream);

}  // namespace qdg
