// gemv.cu -- batch-1 Q4_0 x Q8_0 matrix-vector product (the "mmvq" route of
// batch-1 decode [GGML: Backend abstraction and hardware acceleration,
// section "CUDA: mmvq, mmq, cublas -- three matrix paths"]).
//
// The product is bound by the weight stream: 4.5 bits per weight read once
// from HBM, against a few integer operations per weight.  Design:
//   * One persistent CTA per SM owns a contiguous range of rows.  With
//     K % 256 == 0 a row is a multiple of 16 bytes, so the CTA's share of W is
//     one contiguous byte range, copied in stages of whole rows by 1-D bulk
//     asynchronous copies (TMA engine) into a ring of shared-memory buffers
//     guarded by mbarriers; one producer warp keeps the ring full.
//   * Consumer warps read W from shared memory in 36-byte block pairs (two
//     Q4_0 blocks, 4-byte aligned): lane l of segment s owns pair p = 32s + l
//     of every row, keeps the matching 64 Q8_0 activations in registers for
//     the whole kernel, unpacks nibbles and forms the exact block sums with
//     dp4a, then scales by d_w * d_x (exact in fp32) and reduces across the
//     warp with shuffles.  Rows with more than 32 pairs are split into
//     segments handled by different warps; the producer warp adds the
//     segment partials in a fixed order and stores y, so results are
//     deterministic.
//   * Programmatic dependent launch (optional): W is prefetched before the
//     kernel waits for the preceding grid; activations are read and y is
//     written only after the wait.
#include "common.cuh"

#include <algorithm>
#include <mutex>

namespace qdg {

static __device__ unsigned g_flags_gemv;

namespace {

constexpr int kMaxConsumerWarps = 16;
constexpr int kMaxThreads = 32 * (kMaxConsumerWarps + 1);
constexpr int kStageTarget = 20 * 1024;     // bytes of W per ring stage (whole rows)
constexpr int kRingBudget = 200 * 1024;     // shared memory for the ring
constexpr int kMaxStages = 12;
constexpr uint32_t kNibbles = 0x0F0F0F0Fu;

struct Plan {
    int rowbytes;     // K/32 * 18
    int nb;           // K/32
    int P;            // block pairs per row (K/64)
    int nseg;         // ceil(P / 32)
    int ncw;          // consumer warps, a multiple of nseg
    int nslots;       // rows processed concurrently = ncw / nseg
    int rps;          // rows per stage
    int stage_bytes;  // rps * rowbytes
    int stages;       // ring depth
    size_t smem;      // dynamic shared memory
};

Plan make_plan(int64_t K) {
    Plan p{};
    p.nb = static_cast<int>(K / 32);
    p.rowbytes = p.nb * 18;
    p.P = static_cast<int>(K / 64);
    p.nseg = (p.P + 31) / 32;
    p.ncw = p.nseg * (kMaxConsumerWarps / p.nseg);
    p.nslots = p.ncw / p.nseg;
    const int m = std::max(1, kStageTarget / (p.nslots * p.rowbytes));
    p.rps = p.nslots * m;
    p.stage_bytes = p.rps * p.rowbytes;
    p.stages = std::max(2, std::min(kMaxStages, kRingBudget / p.stage_bytes));
    const size_t part = static_cast<size_t>(p.stages) * p.rps * p.nseg * sizeof(float);
    p.smem = static_cast<size_t>(p.stages) * p.stage_bytes + ((part + 15) / 16) * 16 +
             2 * static_cast<size_t>(p.stages) * sizeof(uint64_t);
    return p;
}

__device__ __forceinline__ int block_dot(uint32_t q0, uint32_t q1, uint32_t q2, uint32_t q3, const uint32_t* x) {
    int acc = 0;
    acc = __dp4a(static_cast<int>(q0 & kNibbles), static_cast<int>(x[0]), acc);
    acc = __dp4a(static_cast<int>((q0 >> 4) & kNibbles), static_cast<int>(x[4]), acc);
    acc = __dp4a(static_cast<int>(q1 & kNibbles), static_cast<int>(x[1]), acc);
    acc = __dp4a(static_cast<int>((q1 >> 4) & kNibbles), static_cast<int>(x[5]), acc);
    acc = __dp4a(static_cast<int>(q2 & kNibbles), static_cast<int>(x[2]), acc);
    acc = __dp4a(static_cast<int>((q2 >> 4) & kNibbles), static_cast<int>(x[6]), acc);
    acc = __dp4a(static_cast<int>(q3 & kNibbles), static_cast<int>(x[3]), acc);
    acc = __dp4a(static_cast<int>((q3 >> 4) & kNibbles), static_cast<int>(x[7]), acc);
    return acc;
}

template <bool kDebug>
__global__ void __launch_bounds__(kMaxThreads, 1)
gemv_kernel(const uint8_t* __restrict__ W, const uint8_t* __restrict__ xq, float* __restrict__ y, int64_t O,
            Plan plan, int32_t* __restrict__ dbg) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int S = plan.stages;
    const int rps = plan.rps;
    const int nseg = plan.nseg;
    uint8_t* ring = smem;
    float* part = reinterpret_cast<float*>(smem + static_cast<size_t>(S) * plan.stage_bytes);
    const size_t part_bytes = ((static_cast<size_t>(S) * rps * nseg * sizeof(float) + 15) / 16) * 16;
    uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(part) + part_bytes);
    uint64_t* empty = full + S;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * O / gridDim.x;
    const int64_t r1 = static_cast<int64_t>(blockIdx.x + 1) * O / gridDim.x;
    const int nrows = static_cast<int>(r1 - r0);
    const int nst = (nrows + rps - 1) / rps;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], plan.ncw);
        }
        fence_barrier_init();
    }
    __syncthreads();
    pdl_trigger();

    if (warp == 0) {
        // ------------------------------------------------ producer + y writer
        const uint64_t policy = l2_policy_evict_first();
        bool ok = true;
        bool waited = false;
        int issued = 0;
        auto store_stage = [&](int k) {
            const int s = k % S;
            const int64_t rs = r0 + static_cast<int64_t>(k) * rps;
            const int rows = static_cast<int>((r1 - rs) < rps ? (r1 - rs) : rps);
            const float* ps = part + static_cast<size_t>(s) * rps * nseg;
            for (int i = lane; i < rows; i += 32) {
                float v = ps[i * nseg];
                for (int g = 1; g < nseg; ++g) v = __fadd_rn(v, ps[i * nseg + g]);
                if (!kDebug) y[rs + i] = v;   // the block-sum hook stores no y
            }
            __syncwarp();
        };
        for (int k = 0; k < nst; ++k) {
            const int s = k % S;
            if (k >= S) {
                ok = __all_sync(0xffffffffu, mbar_wait(&empty[s], ((k / S) - 1) & 1));
                if (!ok) break;
                if (!waited) {
                    pdl_wait();
                    waited = true;
                }
                store_stage(k - S);
            }
            if (lane == 0) {
                const int64_t rs = r0 + static_cast<int64_t>(k) * rps;
                const int rows = static_cast<int>((r1 - rs) < rps ? (r1 - rs) : rps);
                const uint32_t bytes = static_cast<uint32_t>(rows) * plan.rowbytes;
                mbar_arrive_expect_tx(&full[s], bytes);
                bulk_g2s(ring + static_cast<size_t>(s) * plan.stage_bytes, W + rs * plan.rowbytes, bytes, &full[s],
                         policy);
            }
            __syncwarp();
            issued = k + 1;
        }
        if (ok) {
            for (int k = (issued - S > 0 ? issued - S : 0); k < issued; ++k) {
                ok = __all_sync(0xffffffffu, mbar_wait(&empty[k % S], (k / S) & 1));
                if (!ok) break;
                if (!waited) {
                    pdl_wait();
                    waited = true;
                }
                store_stage(k);
            }
        }
        if (!ok) {
            if (lane == 0) atomicOr(&g_flags_gemv, FLAG_TIMEOUT);
            // Do not leave with copies still landing in this CTA's shared memory.
            for (int k = (issued - S > 0 ? issued - S : 0); k < issued; ++k) mbar_wait(&full[k % S], (k / S) & 1);
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int cw = warp - 1;
    const int seg = cw % nseg;
    const int slot = cw / nseg;
    const int p = seg * 32 + lane;
    const bool active = p < plan.P;

    pdl_wait();
    uint32_t xa[8], xb[8];
    float dxa = 0.0f, dxb = 0.0f;
    int sa = 0, sb = 0;
    if (active) {
        const uint32_t* xp = reinterpret_cast<const uint32_t*>(xq + static_cast<size_t>(p) * 68);
        uint32_t w[17];
#pragma unroll
        for (int i = 0; i < 17; ++i) w[i] = __ldg(xp + i);
        dxa = half_bits_to_float(w[0]);
#pragma unroll
        for (int i = 0; i < 8; ++i) xa[i] = bytes_2_to_5(w[i], w[i + 1]);
        dxb = half_bits_to_float(w[8] >> 16);
#pragma unroll
        for (int i = 0; i < 8; ++i) xb[i] = w[9 + i];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            sa = __dp4a(static_cast<int>(xa[i]), 0x01010101, sa);
            sb = __dp4a(static_cast<int>(xb[i]), 0x01010101, sb);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) xa[i] = xb[i] = 0u;
    }

    for (int k = 0; k < nst; ++k) {
        const int s = k % S;
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&full[s], (k / S) & 1));
        if (!ok) {
            if (lane == 0) atomicOr(&g_flags_gemv, FLAG_TIMEOUT);
            break;
        }
        const int64_t rs = r0 + static_cast<int64_t>(k) * rps;
        const int rows = static_cast<int>((r1 - rs) < rps ? (r1 - rs) : rps);
        const uint8_t* st = ring + static_cast<size_t>(s) * plan.stage_bytes;
        float* ps = part + static_cast<size_t>(s) * rps * nseg;
        for (int row = slot; row < rows; row += plan.nslots) {
            float acc = 0.0f;
            if (active) {
                const uint32_t* wp =
                    reinterpret_cast<const uint32_t*>(st + static_cast<size_t>(row) * plan.rowbytes + p * 36);
                uint32_t w[9];
#pragma unroll
                for (int i = 0; i < 9; ++i) w[i] = wp[i];
                const int ia = block_dot(bytes_2_to_5(w[0], w[1]), bytes_2_to_5(w[1], w[2]),
                                         bytes_2_to_5(w[2], w[3]), bytes_2_to_5(w[3], w[4]), xa) -
                               8 * sa;
                const int ib = block_dot(w[5], w[6], w[7], w[8], xb) - 8 * sb;
                const float dwa = half_bits_to_float(w[0]);
                const float dwb = half_bits_to_float(w[4] >> 16);
                acc = __fmul_rn(__fmul_rn(dwa, dxa), static_cast<float>(ia));
                acc = __fmaf_rn(__fmul_rn(dwb, dxb), static_cast<float>(ib), acc);
                if (kDebug) {
                    int32_t* d = dbg + (rs + row) * plan.nb + 2 * p;
                    d[0] = ia;
                    d[1] = ib;
                }
            }
            acc = warp_sum(acc);
            if (lane == 0) ps[row * nseg + seg] = acc;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
}

std::mutex g_attr_mutex;
size_t g_attr_smem[2] = {0, 0};

template <bool kDebug>
cudaError_t ensure_smem(size_t bytes) {
    std::lock_guard<std::mutex> lock(g_attr_mutex);
    if (g_attr_smem[kDebug] >= bytes) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel<kDebug>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(bytes));
    if (e == cudaSuccess) g_attr_smem[kDebug] = bytes;
    return e;
}

}  // namespace

int gemv_launch(const void* W, const void* xq, float* y, int64_t O, int64_t K, cudaStream_t stream, int32_t* dbg) {
    if (!W || !xq || (!y && !dbg)) return QDG_EINVAL;
    if (O <= 0 || K <= 0) return QDG_EINVAL;
    if (K % 256 != 0 || K > 32768 || O >= (int64_t(1) << 31)) return QDG_ESHAPE;
    if (!aligned(W, 16) || !aligned(xq, 4) || !aligned(y, 4) || !aligned(dbg, 4)) return QDG_EALIGN;
    const DeviceInfo dev = device_info();
    if (dev.device < 0) return QDG_ECUDA;
    const Plan plan = make_plan(K);
    if (plan.smem > dev.smem_optin) return QDG_ESHAPE;
    const int grid = static_cast<int>(std::min<int64_t>(dev.sms, O));
    cudaError_t e;
    if (dbg) {
        e = ensure_smem<true>(plan.smem);
        if (e == cudaSuccess)
            e = launch(gemv_kernel<true>, dim3(grid), dim3(32 * (plan.ncw + 1)), plan.smem, stream, false,
                       static_cast<const uint8_t*>(W), static_cast<const uint8_t*>(xq), y, O, plan, dbg);
    } else {
        e = ensure_smem<false>(plan.smem);
        if (e == cudaSuccess)
            e = launch(gemv_kernel<false>, dim3(grid), dim3(32 * (plan.ncw + 1)), plan.smem, stream, true,
                       static_cast<const uint8_t*>(W), static_cast<const uint8_t*>(xq), y, O, plan,
                       static_cast<int32_t*>(nullptr));
    }
    if (e != cudaSuccess) return QDG_ECUDA;
    count_launch(1);
    return QDG_OK;
}

unsigned flags_read_clear_gemv(cudaStream_t stream) {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_flags_gemv, sizeof(v), 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return ~0u;
    if (cudaMemcpyToSymbolAsync(g_flags_gemv, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream) !=
        cudaSuccess)
        return ~0u;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return ~0u;
    return v;
}

}  // namespace qdg

extern "C" int q4_0_q8_0_gemv(const void* W, const void* xq, float* y, int64_t O, int64_t K,
                              qdg_stream_t stream) {
    if (!y) return QDG_EINVAL;
    return qdg::gemv_launch(W, xq, y, O, K, reinterpret_cast<cudaStream_t>(stream), nullptr);
}
