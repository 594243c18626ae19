// stage.cu -- host <-> device staging of a decode step's vectors by a kernel.
//
// On a Grace-Blackwell node, pinned host memory is mapped into the GPU's
// address space and reachable from kernels over the coherent chip-to-chip
// link.  Moving a step's input vectors in (and its outputs out) with a
// kernel keeps that move inside the chain of programmatically dependent
// launches; a copy-engine transfer between two kernels ends the chain, and
// the kernel after it pays a full launch latency.
//
// The copy kernel triggers its dependents at once (they launch and wait for
// it to complete) and waits for the preceding grid before it reads or writes
// anything, so the staged data are ordered after everything before it on the
// stream, as with a stream-ordered copy.
#include "common.cuh"

#include <algorithm>

namespace qdg {
namespace {

constexpr int kStageThreads = 256;

__global__ void __launch_bounds__(kStageThreads) stage_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src,
                                                              int64_t n16) {
    pdl_trigger();
    pdl_wait();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kStageThreads;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kStageThreads + threadIdx.x; i < n16; i += stride)
        dst[i] = src[i];
}

// The address under which the current device reaches p: p itself for device
// or managed memory, the mapped address for pinned host memory, nullptr for
// memory the device cannot reach (pageable host memory, unknown pointers).
void* device_view(const void* p) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    switch (at.type) {
        case cudaMemoryTypeDevice:
        case cudaMemoryTypeManaged:
            return const_cast<void*>(p);
        case cudaMemoryTypeHost:
            return at.devicePointer;
        default:
            return nullptr;
    }
}

}  // namespace
}  // namespace qdg

using namespace qdg;

extern "C" int qdg_stage_copy(void* dst, const void* src, int64_t bytes, qdg_stream_t stream) {
    if (!dst || !src || bytes < 0) return QDG_EINVAL;
    if (bytes == 0) return QDG_OK;
    if (!aligned(dst, 16) || !aligned(src, 16) || bytes % 16 != 0) return QDG_EALIGN;
    void* d = device_view(dst);
    const void* s = device_view(src);
    if (!d || !s) return QDG_EINVAL;
    const char* dc = static_cast<const char*>(d);
    const char* sc = static_cast<const char*>(s);
    if (dc < sc + bytes && sc < dc + bytes) return QDG_EINVAL;   // overlapping ranges
    const DeviceInfo dev = device_info();
    if (dev.sms <= 0) return QDG_ECUDA;
    const int64_t n16 = bytes / 16;
    const int64_t want = (n16 + kStageThreads - 1) / kStageThreads;
    const int grid = static_cast<int>(std::min<int64_t>(want, 4LL * dev.sms));
    const cudaError_t e = launch(stage_kernel, dim3(grid), dim3(kStageThreads), 0,
                                 reinterpret_cast<cudaStream_t>(stream), true, static_cast<uint4*>(d),
                                 static_cast<const uint4*>(s), n16);
    if (e != cudaSuccess) return QDG_ECUDA;
    count_launch(10);
    return QDG_OK;
}
