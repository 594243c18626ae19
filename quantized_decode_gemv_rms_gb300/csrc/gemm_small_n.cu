// gemm_small_n.cu -- Q4_0 x Q8_0 product for 1..8 activation vectors that
// share one pass over W (speculative / parallel decode: the "vector case" of
// the quantized matrix-vector route [GGML: Backend abstraction and hardware
// acceleration, section "CUDA: mmvq, mmq, cublas -- three matrix paths"]).
//
// Still bound by the weight stream, but N dot products per weight make the
// integer work N times larger than at N = 1, so the exact per-block sums are
// formed with the integer tensor-core MMA m16n8k32 (u8 weights x s8
// activations -> s32): one instruction covers 16 rows x 8 columns x one
// 32-element block.  The Q4_0 nibble order lines up with its A fragment: a
// lane's 32-bit word c of a block holds elements 4c..4c+3 in its low nibbles
// and 16+4c..16+4c+3 in its high nibbles, exactly the lane's two A registers
// for that row.  The "-8" of Q4_0 enters as the accumulator input
// -8 * sum(q_x), itself one MMA with an all(-8) A operand.
//
// Staging: each CTA owns a contiguous row range, processed in tiles of 32
// rows; a producer warp copies, per stage, the tile's rows for 4 groups of 8
// blocks plus the N activation chunks of those blocks with 1-D bulk copies
// (TMA engine) into padded shared-memory rows (row strides = 16 mod 32 bytes,
// so fragment loads are free of bank conflicts).  Eight consumer warps split
// the stage's blocks, accumulate fp32 partials per (row, column) and reduce
// across warps in a fixed order at the end of each tile.
#include "common.cuh"

#include <algorithm>
#include <mutex>

namespace qdg {

static __device__ unsigned g_flags_small_n;

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr int kTileRows = 32;                 // two 16-row MMA slabs
constexpr int kGroupsPerStage = 4;            // 4 groups of 8 blocks = 1024 elements of K per stage
constexpr int kBlocksPerStage = kGroupsPerStage * 8;
constexpr int kWStride = kGroupsPerStage * 144 + 16;   // 592 = 16 mod 32
constexpr int kXStride = kBlocksPerStage * 34 + 16;    // 1104 = 16 mod 32
constexpr int kStageBytes = kTileRows * kWStride + 8 * kXStride;
constexpr int kStages = 6;
constexpr int kRedBytes = kConsumerWarps * 2 * 128 * 4;
constexpr size_t kSmem = static_cast<size_t>(kStages) * kStageBytes + kRedBytes + 2 * kStages * 8 + 16;
constexpr uint32_t kNibbles = 0x0F0F0F0Fu;

static_assert(kWStride % 32 == 16 && kXStride % 32 == 16, "padded strides");
static_assert(kStageBytes % 16 == 0, "stage alignment");

__device__ __forceinline__ void mma_u8s8(int& d0, int& d1, int& d2, int& d3, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1, int c0, int c1, int c2, int c3) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.u8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3)
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "r"(c0), "r"(c1), "r"(c2), "r"(c3));
}

__device__ __forceinline__ void mma_s8s8(int& d0, int& d1, int& d2, int& d3, uint32_t a, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%4,%4,%4}, {%5,%6}, "
        "{%7,%7,%7,%7};"
        : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3)
        : "r"(a), "r"(b0), "r"(b1), "r"(0));
}

// 32-bit word starting at a 2-byte aligned shared-memory address.
__device__ __forceinline__ uint32_t lds_u32_a2(const uint8_t* p) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    if ((a & 3u) == 0) return *reinterpret_cast<const uint32_t*>(p);
    const uint32_t lo = *reinterpret_cast<const uint32_t*>(p - 2);
    const uint32_t hi = *reinterpret_cast<const uint32_t*>(p + 2);
    return bytes_2_to_5(lo, hi);
}

struct Args {
    const uint8_t* W;
    const uint8_t* xq;
    float* y;
    int32_t* dbg;
    int64_t ldy;
    int64_t O;
    int rowbytes;   // K/32 * 18
    int xrow;       // K/32 * 34
    int nb;         // K/32
    int groups;     // K/256
    int N;
};

template <bool kDebug>
__global__ void __launch_bounds__(kThreads, 1) small_n_kernel(Args a) {
    extern __shared__ __align__(128) uint8_t smem[];
    float* red = reinterpret_cast<float*>(smem + static_cast<size_t>(kStages) * kStageBytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(kStages) * kStageBytes + kRedBytes);
    uint64_t* empty = full + kStages;
    // Set by a consumer warp whose wait gave up: the others stop computing but
    // still reach every tile-end barrier, so no warp is left waiting.
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kStages);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * a.O / gridDim.x;
    const int64_t r1 = static_cast<int64_t>(blockIdx.x + 1) * a.O / gridDim.x;
    const int nrows = static_cast<int>(r1 - r0);
    const int ntiles = (nrows + kTileRows - 1) / kTileRows;
    const int nchunks = (a.groups + kGroupsPerStage - 1) / kGroupsPerStage;
    const int nst = ntiles * nchunks;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        fence_barrier_init();
        *abort_flag = 0;
    }
    __syncthreads();
    pdl_trigger();
    pdl_wait();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        const uint64_t policy = l2_policy_evict_first();
        bool ok = true;
        int issued = 0;
        for (int k = 0; k < nst; ++k) {
            const int s = k % kStages;
            if (k >= kStages) {
                ok = __all_sync(0xffffffffu, mbar_wait(&empty[s], ((k / kStages) - 1) & 1));
                if (!ok) break;
            }
            const int t = k / nchunks;
            const int ck = k - t * nchunks;
            const int64_t rt = r0 + static_cast<int64_t>(t) * kTileRows;
            const int rows = static_cast<int>((r1 - rt) < kTileRows ? (r1 - rt) : kTileRows);
            const int g0 = ck * kGroupsPerStage;
            const int vg = (a.groups - g0) < kGroupsPerStage ? (a.groups - g0) : kGroupsPerStage;
            const uint32_t wbytes = static_cast<uint32_t>(vg) * 144;
            const uint32_t xbytes = static_cast<uint32_t>(vg) * 272;
            uint8_t* st = smem + static_cast<size_t>(s) * kStageBytes;
            if (lane == 0) mbar_arrive_expect_tx(&full[s], rows * wbytes + a.N * xbytes);
            __syncwarp();
            for (int i = lane; i < rows + a.N; i += 32) {
                if (i < rows) {
                    bulk_g2s(st + i * kWStride, a.W + (rt + i) * a.rowbytes + static_cast<int64_t>(g0) * 144, wbytes,
                             &full[s], policy);
                } else {
                    const int n = i - rows;
                    bulk_g2s(st + kTileRows * kWStride + n * kXStride,
                             a.xq + static_cast<int64_t>(n) * a.xrow + static_cast<int64_t>(g0) * 272, xbytes,
                             &full[s], policy);
                }
            }
            __syncwarp();
            issued = k + 1;
        }
        if (!ok) {
            if (lane == 0) atomicOr(&g_flags_small_n, FLAG_TIMEOUT);
            for (int k = (issued - kStages > 0 ? issued - kStages : 0); k < issued; ++k)
                mbar_wait(&full[k % kStages], (k / kStages) & 1);
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int cw = warp - 1;
    const int g = lane >> 2;
    const int c = lane & 3;
    const bool colg = g < a.N;
    const bool col0 = 2 * c < a.N;
    const bool col1 = 2 * c + 1 < a.N;
    float acc[2][4];
#pragma unroll
    for (int sl = 0; sl < 2; ++sl)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[sl][i] = 0.0f;

    for (int k = 0; k < nst; ++k) {
        const int s = k % kStages;
        bool ok = *abort_flag == 0;
        if (ok) {
            ok = __all_sync(0xffffffffu, mbar_wait(&full[s], (k / kStages) & 1));
            if (!ok && lane == 0) {
                atomicOr(&g_flags_small_n, FLAG_TIMEOUT);
                *abort_flag = 1;
            }
        }
        const int t = k / nchunks;
        const int ck = k - t * nchunks;
        const int64_t rt = r0 + static_cast<int64_t>(t) * kTileRows;
        const int g0 = ck * kGroupsPerStage;
        const int vg = (a.groups - g0) < kGroupsPerStage ? (a.groups - g0) : kGroupsPerStage;
        const int vblocks = ok ? vg * 8 : 0;
        const uint8_t* st = smem + static_cast<size_t>(s) * kStageBytes;
        const uint8_t* xs = st + kTileRows * kWStride;
        for (int bl = cw; bl < vblocks; bl += kConsumerWarps) {
            uint32_t b0 = 0, b1 = 0;
            if (colg) {
                const uint8_t* xb = xs + g * kXStride + bl * 34;
                b0 = lds_u32_a2(xb + 2 + 4 * c);
                b1 = lds_u32_a2(xb + 18 + 4 * c);
            }
            const float dx0 = col0 ? half_bits_to_float(*reinterpret_cast<const unsigned short*>(
                                         xs + (2 * c) * kXStride + bl * 34))
                                   : 0.0f;
            const float dx1 = col1 ? half_bits_to_float(*reinterpret_cast<const unsigned short*>(
                                         xs + (2 * c + 1) * kXStride + bl * 34))
                                   : 0.0f;
            int m0, m1, m2, m3;   // -8 * sum(q_x) for columns 2c, 2c+1
            mma_s8s8(m0, m1, m2, m3, 0xF8F8F8F8u, b0, b1);
#pragma unroll
            for (int sl = 0; sl < 2; ++sl) {
                const uint8_t* wr0 = st + (sl * 16 + g) * kWStride + bl * 18;
                const uint8_t* wr1 = wr0 + 8 * kWStride;
                const uint32_t w0 = lds_u32_a2(wr0 + 2 + 4 * c);
                const uint32_t w1 = lds_u32_a2(wr1 + 2 + 4 * c);
                const float dw0 = half_bits_to_float(*reinterpret_cast<const unsigned short*>(wr0));
                const float dw1 = half_bits_to_float(*reinterpret_cast<const unsigned short*>(wr1));
                int d0, d1, d2, d3;
                mma_u8s8(d0, d1, d2, d3, w0 & kNibbles, w1 & kNibbles, (w0 >> 4) & kNibbles, (w1 >> 4) & kNibbles,
                         b0, b1, m0, m1, m0, m1);
                acc[sl][0] = __fmaf_rn(__fmul_rn(dw0, dx0), static_cast<float>(d0), acc[sl][0]);
                acc[sl][1] = __fmaf_rn(__fmul_rn(dw0, dx1), static_cast<float>(d1), acc[sl][1]);
                acc[sl][2] = __fmaf_rn(__fmul_rn(dw1, dx0), static_cast<float>(d2), acc[sl][2]);
                acc[sl][3] = __fmaf_rn(__fmul_rn(dw1, dx1), static_cast<float>(d3), acc[sl][3]);
                if (kDebug) {
                    const int64_t row0 = rt + sl * 16 + g;
                    const int64_t b = static_cast<int64_t>(g0) * 8 + bl;
                    if (row0 < r1) {
                        if (col0) a.dbg[((2 * c) * a.O + row0) * a.nb + b] = d0;
                        if (col1) a.dbg[((2 * c + 1) * a.O + row0) * a.nb + b] = d1;
                    }
                    if (row0 + 8 < r1) {
                        if (col0) a.dbg[((2 * c) * a.O + row0 + 8) * a.nb + b] = d2;
                        if (col1) a.dbg[((2 * c + 1) * a.O + row0 + 8) * a.nb + b] = d3;
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);

        if (ck == nchunks - 1) {
            // End of a row tile: fixed-order reduction across the consumer warps.
            float* rw = red + cw * 256;
#pragma unroll
            for (int sl = 0; sl < 2; ++sl)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    rw[sl * 128 + lane * 4 + i] = acc[sl][i];
                    acc[sl][i] = 0.0f;
                }
            asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
            const int e = threadIdx.x - 32;             // 0..255
            const int sl = e >> 7;
            const int ln = (e >> 2) & 31;
            const int i = e & 3;
            const int row = sl * 16 + (ln >> 2) + 8 * (i >> 1);
            const int col = 2 * (ln & 3) + (i & 1);
            float v = red[e];
#pragma unroll
            for (int w = 1; w < kConsumerWarps; ++w) v = __fadd_rn(v, red[w * 256 + e]);
            if (a.y != nullptr && rt + row < r1 && col < a.N) a.y[col * a.ldy + rt + row] = v;
            asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
        }
    }
}

std::mutex g_attr_mutex;
bool g_attr_done[2] = {false, false};

template <bool kDebug>
cudaError_t ensure_smem() {
    std::lock_guard<std::mutex> lock(g_attr_mutex);
    if (g_attr_done[kDebug]) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(small_n_kernel<kDebug>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmem));
    if (e == cudaSuccess) g_attr_done[kDebug] = true;
    return e;
}

}  // namespace

int small_n_launch(const void* W, const void* xq, float* y, int64_t ldy, int64_t O, int64_t K, int64_t N,
                   cudaStream_t stream, int32_t* dbg) {
    if (!W || !xq || (!y && !dbg)) return QDG_EINVAL;
    if (O <= 0 || K <= 0 || N < 1 || N > 8) return QDG_EINVAL;
    if (!dbg && ldy < O) return QDG_EINVAL;
    if (K % 256 != 0 || K > 65536 || O >= (int64_t(1) << 31)) return QDG_ESHAPE;
    if (!aligned(W, 16) || !aligned(xq, 16) || (y && !aligned(y, 4))) return QDG_EALIGN;
    const DeviceInfo dev = device_info();
    if (dev.device < 0) return QDG_ECUDA;
    if (kSmem > dev.smem_optin) return QDG_ECUDA;
    Args a;
    a.W = static_cast<const uint8_t*>(W);
    a.xq = static_cast<const uint8_t*>(xq);
    a.y = y;
    a.dbg = dbg;
    a.ldy = ldy;
    a.O = O;
    a.nb = static_cast<int>(K / 32);
    a.rowbytes = a.nb * 18;
    a.xrow = a.nb * 34;
    a.groups = static_cast<int>(K / 256);
    a.N = static_cast<int>(N);
    const int grid = static_cast<int>(std::min<int64_t>(dev.sms, O));
    cudaError_t e;
    if (dbg) {
        e = ensure_smem<true>();
        if (e == cudaSuccess) e = launch(small_n_kernel<true>, dim3(grid), dim3(kThreads), kSmem, stream, false, a);
    } else {
        e = ensure_smem<false>();
        if (e == cudaSuccess) e = launch(small_n_kernel<false>, dim3(grid), dim3(kThreads), kSmem, stream, true, a);
    }
    if (e != cudaSuccess) return QDG_ECUDA;
    count_launch(2);
    return QDG_OK;
}

unsigned flags_read_clear_small_n(cudaStream_t stream) {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_flags_small_n, sizeof(v), 0, cudaMemcpyDeviceToHost, stream) !=
        cudaSuccess)
        return ~0u;
    if (cudaMemcpyToSymbolAsync(g_flags_small_n, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream) !=
        cudaSuccess)
        return ~0u;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return ~0u;
    return v;
}

}  // namespace qdg

extern "C" int q4_0_q8_0_gemm_small_n(const void* W, const void* xq, float* y, int64_t ldy, int64_t O, int64_t K,
                                      int64_t N, qdg_stream_t stream) {
    if (!y) return QDG_EINVAL;
    return qdg::small_n_launch(W, xq, y, ldy, O, K, N, reinterpret_cast<cudaStream_t>(stream), nullptr);
}
