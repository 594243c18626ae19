// gemv_segn.cu -- the small-N product for three or four activation vectors on
// weights in the segment layout: Y[n] = W * x[n], one pass over W.
//
// Several decode streams share one weight pass in the quantized vector path;
// GGML's CUDA back end keeps a batch of a few columns on that path rather than
// the matrix path [GGML: Backend abstraction and hardware acceleration,
// section "CUDA: mmvq, mmq, cublas -- three matrix paths"].
//
// Design: exact block sums by dp4a, as the one- and two-vector kernels, but
// with one weight block per lane instead of two, so that the activations of
// four vectors (32 words) still fit in registers beside an eight-deep ring:
//   * a segment (64 blocks, 1152 bytes; see gemv_seg.cu) is cut into two
//     halves of 32 blocks; a warp owns one half-segment h of segment s of
//     rows slot, slot + nslots, ...; lane l owns block 64s + 32h + l and
//     holds that block of every vector in registers for the whole kernel;
//   * per row-segment half the lane loads its 16 nibble bytes (a warp reads
//     512 contiguous bytes) and its scale word, eight rows ahead of use
//     (80 KB in flight per SM);
//   * per vector: the block sum sum((q - 8) q_x) by eight dp4a starting from
//     -8 sum(q_x), then (d_w d_x) isum in fp32;
//   * every four rows the 16 partials (four rows x four vectors) of a lane go
//     through one transposed warp butterfly, which leaves each total in two
//     lanes; half-segment partials are combined per row in a fixed order
//     (deterministic).
// A row needs 2 * nseg half-segments (one fewer when the last segment holds
// at most 32 blocks), so K <= 16384 gives every half-segment a warp.
#include "common.cuh"

#include <algorithm>

namespace qdg {

static __device__ unsigned g_flags_gemv_segn;

namespace {

constexpr int kWarps = 16;
constexpr int kThreads = 32 * kWarps;
constexpr int kDepth = 8;                   // row halves in flight per warp
constexpr int kSegStride = 1152;
constexpr int kPartFloats = 3072;
constexpr int kL2Prefetch = 96 * 1024;
constexpr uint32_t kNibbles = 0x0F0F0F0Fu;

struct PlanN {
    int rowbytes;   // bytes of one row in the segment layout
    int nb;         // K/32
    int nseg;       // ceil(nb / 64)
    int rlast;      // blocks in the last segment (8..64)
    int nhs;        // half-segments per row
    int nslots;     // rows in flight per CTA = kWarps / nhs
    int rch;        // rows per chunk of partial sums, a multiple of nslots
};

PlanN make_plan_n(int64_t K, int nv) {
    PlanN p{};
    p.nb = static_cast<int>(K / 32);
    p.nseg = (p.nb + 63) / 64;
    p.rlast = p.nb - 64 * (p.nseg - 1);
    p.rowbytes = kSegStride * (p.nseg - 1) + 16 * p.rlast + 128;
    p.nhs = 2 * (p.nseg - 1) + (p.rlast > 32 ? 2 : 1);
    p.nslots = kWarps / p.nhs;
    p.rch = p.nslots > 0 ? (kPartFloats / (p.nhs * nv)) / p.nslots * p.nslots : 0;
    return p;
}

struct ArgsN {
    const uint8_t* W;
    const uint8_t* xq;      // nv Q8_0 vectors of K/32 blocks, back to back
    int xq_bulk;            // xq is 16-byte aligned: one bulk copy into shared memory
    float* y;               // y[n][row] at y + n * ldy
    int64_t ldy;
    int32_t* dbg;           // [nv][O][K/32] exact block sums instead of y
    int64_t O;
};

__device__ __forceinline__ uint4 ldg_stream16(const uint8_t* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ldg_stream4(const uint8_t* p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// One lane's share of one row's half-segment: its block's 16 nibble bytes and
// the segment's scale word l (the lane's scale in half h).
struct EntryN {
    uint4 q;
    uint32_t sc;
};

template <int NV, bool kDebug>
__global__ void __launch_bounds__(kThreads, 1) gemv_segn_kernel(const __grid_constant__ ArgsN a,
                                                                const __grid_constant__ PlanN plan) {
    static_assert(NV == 3 || NV == 4, "three or four vectors: sixteen partials per butterfly");
    __shared__ float part[kPartFloats];
    __shared__ uint64_t xbar;
    extern __shared__ __align__(16) uint8_t xs[];   // the NV vectors when a.xq_bulk
    const int64_t O = a.O;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nhs = plan.nhs;
    const int hs = warp % nhs;
    const int slot = warp / nhs;
    const bool worker = slot < plan.nslots;
    const int seg = hs >> 1, half = hs & 1;
    const int r = (seg == plan.nseg - 1) ? plan.rlast : 64;     // blocks in this warp's segment
    const int blk = 32 * half + lane;                            // block within the segment
    const bool has = worker && blk < r;
    const int nib_off = seg * kSegStride + 16 * blk;
    const int sc_off = seg * kSegStride + 16 * r + 4 * lane;
    const int sc_shift = 16 * half;

    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * O / gridDim.x;
    const int64_t r1 = static_cast<int64_t>(blockIdx.x + 1) * O / gridDim.x;
    const int nrows = static_cast<int>(r1 - r0);

    if (threadIdx.x == 0) {
        mbar_init(&xbar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    pdl_trigger();

    EntryN pipe[kDepth] = {};
    auto load_at = [&](const uint8_t* rowp, EntryN& e) {
        if (has) e.q = ldg_stream16(rowp + nib_off);
        e.sc = ldg_stream4(rowp + sc_off);
    };
    auto load = [&](int64_t row, EntryN& e) { load_at(a.W + row * plan.rowbytes, e); };
    auto fill = [&](int64_t c0, int crows) {
#pragma unroll
        for (int d = 0; d < kDepth; ++d) {
            const int ri = slot + d * plan.nslots;
            if (ri < crows) load(c0 + ri, pipe[d]);
        }
    };
    if (worker) fill(r0, min(nrows, plan.rch));
    if (threadIdx.x == 0) {
        const int64_t first = r0 + static_cast<int64_t>(kDepth) * plan.nslots;
        const int64_t n = min(r1 - first, static_cast<int64_t>(kL2Prefetch / plan.rowbytes));
        if (n > 0)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a.W + first * plan.rowbytes),
                         "r"(static_cast<uint32_t>(n * plan.rowbytes))
                         : "memory");
    }

    pdl_wait();

    // the lane's block of every vector: codes as 8 words, fp32 scale, and
    // -8 sum(q_x) (the dp4a chains start from it, so they end at the exact
    // block sum of (q - 8) q_x)
    uint32_t xv[NV][8];
    float dx[NV];
    int base[NV];
    const int vec = plan.nb * 34;
    const int b = 64 * seg + blk;
    auto load_vec = [&](const uint8_t* src, bool shared) {
#pragma unroll
        for (int n = 0; n < NV; ++n) {
            const unsigned short* h = reinterpret_cast<const unsigned short*>(src + n * vec + b * 34);
            auto ld = [&](int i) -> uint32_t { return shared ? h[i] : __ldg(h + i); };
            dx[n] = half_bits_to_float(ld(0));
            int sum = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                xv[n][i] = ld(1 + 2 * i) | (ld(2 + 2 * i) << 16);
                sum = __dp4a(static_cast<int>(xv[n][i]), 0x01010101, sum);
            }
            base[n] = -8 * sum;
        }
    };
#pragma unroll
    for (int n = 0; n < NV; ++n) {
        dx[n] = 0.0f;
        base[n] = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) xv[n][i] = 0u;
    }
    if (a.xq_bulk) {
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(&xbar, static_cast<uint32_t>(NV * vec));
            bulk_g2s_plain(xs, a.xq, static_cast<uint32_t>(NV * vec), &xbar);
        }
        if (!mbar_wait(&xbar, 0)) atomicOr(&g_flags_gemv_segn, FLAG_TIMEOUT);
        if (has) load_vec(xs, true);
    } else if (has) {
        load_vec(a.xq, false);
    }

    // dot the entry with every vector, then refill it with the row kDepth
    // slots ahead; v[4 k + n] = the lane's partial for vector n.  Entries
    // are consumed in row order, so their refills are consecutive rows of
    // this warp's slot: one running pointer, advanced by a slot stride.
    const uint8_t* wnext = nullptr;
    const int64_t wstride = static_cast<int64_t>(plan.nslots) * plan.rowbytes;
    auto consume = [&](int64_t c0, int crows, int ri, EntryN& entry, float (&v)[16], int k) {
        const uint4 q = entry.q;
        const uint32_t lo[4] = {q.x & kNibbles, q.y & kNibbles, q.z & kNibbles, q.w & kNibbles};
        const uint32_t hi[4] = {(q.x >> 4) & kNibbles, (q.y >> 4) & kNibbles, (q.z >> 4) & kNibbles,
                                (q.w >> 4) & kNibbles};
        const float dw = half_bits_to_float(entry.sc >> sc_shift);
        float f[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int n = 0; n < NV; ++n) {
            int acc = base[n];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc = __dp4a(static_cast<int>(lo[i]), static_cast<int>(xv[n][i]), acc);
                acc = __dp4a(static_cast<int>(hi[i]), static_cast<int>(xv[n][4 + i]), acc);
            }
            f[n] = static_cast<float>(acc);
            if (kDebug && has) a.dbg[(n * O + c0 + ri) * plan.nb + b] = acc;
        }
        // (d_w d_x) isum, two vectors per packed multiply (same roundings)
        float s0, s1, s2, s3;
        fmul2(s0, s1, dw, dw, dx[0], dx[1]);
        fmul2(v[4 * k], v[4 * k + 1], s0, s1, f[0], f[1]);
        if (NV == 4) {
            fmul2(s2, s3, dw, dw, dx[2], dx[NV - 1]);
            fmul2(v[4 * k + 2], v[4 * k + 3], s2, s3, f[2], f[3]);
        } else {
            v[4 * k + 2] = __fmul_rn(__fmul_rn(dw, dx[2]), f[2]);
            v[4 * k + 3] = 0.0f;
        }
        const int ahead = ri + kDepth * plan.nslots;
        if (ahead < crows) {
            load_at(wnext, entry);
            wnext += wstride;
        }
    };

    // sixteen partials v[4 k + n] (row ri + k step, vector n) in one
    // butterfly: the xor-16, -8, -4 and -2 exchanges halve the values each
    // time and leave value 8 b16 + 4 b8 + 2 b4 + b2 in the lanes whose bits
    // 4, 3, 2, 1 are b16, b8, b4, b2; the xor-1 exchange completes the sum
    auto reduce16 = [&](int ri, int step, int crows, const float (&v)[16]) {
        const bool u16 = (lane & 16) != 0, u8 = (lane & 8) != 0, u4 = (lane & 4) != 0, u2 = (lane & 2) != 0;
        float w8[8], w4[4], w2[2];
#pragma unroll
        for (int q = 0; q < 8; ++q)
            w8[q] = __fadd_rn(u16 ? v[8 + q] : v[q], __shfl_xor_sync(0xffffffffu, u16 ? v[q] : v[8 + q], 16));
#pragma unroll
        for (int q = 0; q < 4; ++q)
            w4[q] = __fadd_rn(u8 ? w8[4 + q] : w8[q], __shfl_xor_sync(0xffffffffu, u8 ? w8[q] : w8[4 + q], 8));
#pragma unroll
        for (int q = 0; q < 2; ++q)
            w2[q] = __fadd_rn(u4 ? w4[2 + q] : w4[q], __shfl_xor_sync(0xffffffffu, u4 ? w4[q] : w4[2 + q], 4));
        float c = __fadd_rn(u2 ? w2[1] : w2[0], __shfl_xor_sync(0xffffffffu, u2 ? w2[0] : w2[1], 2));
        c = __fadd_rn(c, __shfl_xor_sync(0xffffffffu, c, 1));
        const int idx = lane >> 1;
        const int k = idx >> 2, n = idx & 3;
        const int row = ri + k * step;
        if ((lane & 1) == 0 && n < NV && row < crows) part[(row * nhs + hs) * NV + n] = c;
    };

    // four ring entries (pipe[o + k], rows ri + k step) into one butterfly
    auto group4 = [&](int64_t c0, int crows, int ri, int step, int o) {
        float v[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (ri + k * step < crows) {
                consume(c0, crows, ri + k * step, pipe[o + k], v, k);
            } else {
#pragma unroll
                for (int n = 0; n < 4; ++n) v[4 * k + n] = 0.0f;
            }
        }
        if (!kDebug) reduce16(ri, step, crows, v);
    };

    for (int64_t c0 = r0; c0 < r1; c0 += plan.rch) {
        const int crows = static_cast<int>((r1 - c0) < plan.rch ? (r1 - c0) : plan.rch);
        if (worker) {
            if (c0 != r0) fill(c0, crows);
            wnext = a.W + (c0 + slot + static_cast<int64_t>(kDepth) * plan.nslots) * plan.rowbytes;
            const int step = plan.nslots;
            for (int ri = slot; ri < crows; ri += kDepth * step) {
                group4(c0, crows, ri, step, 0);
                if (ri + 4 * step < crows) group4(c0, crows, ri + 4 * step, step, 4);
            }
        }
        __syncthreads();
        if (!kDebug) {
            for (int t = threadIdx.x; t < NV * crows; t += kThreads) {
                const int row = t / NV, n = t - row * NV;
                float v = part[row * nhs * NV + n];
                for (int g = 1; g < nhs; ++g) v = __fadd_rn(v, part[(row * nhs + g) * NV + n]);
                a.y[n * a.ldy + c0 + row] = v;
            }
        }
        __syncthreads();
    }
}

template <int NV>
int launch_nv(const ArgsN& a, const PlanN& plan, int grid, size_t smem, cudaStream_t stream, bool debug) {
    const void* k0 = reinterpret_cast<const void*>(gemv_segn_kernel<NV, false>);
    const void* k1 = reinterpret_cast<const void*>(gemv_segn_kernel<NV, true>);
    if (ensure_smem_limit(k0, smem) != cudaSuccess || ensure_smem_limit(k1, smem) != cudaSuccess) return QDG_ECUDA;
    cudaError_t e;
    if (debug)
        e = launch(gemv_segn_kernel<NV, true>, dim3(grid), dim3(kThreads), smem, stream, false, a, plan);
    else
        e = launch(gemv_segn_kernel<NV, false>, dim3(grid), dim3(kThreads), smem, stream, true, a, plan);
    return e == cudaSuccess ? QDG_OK : QDG_ECUDA;
}

}  // namespace

bool gemv_segn_supported(int64_t K, int64_t N) {
    if (N < 3 || N > 4 || K <= 0 || K % 256 != 0 || K > 16384) return false;
    return make_plan_n(K, static_cast<int>(N)).nslots >= 1;
}

int gemv_segn_launch(const void* W, const void* xq, float* y, int64_t ldy, int64_t O, int64_t K, int64_t N,
                     cudaStream_t stream, int32_t* dbg) {
    if (!W || !xq || (!y && !dbg) || O <= 0 || K <= 0 || (y && ldy < O)) return QDG_EINVAL;
    if (!gemv_segn_supported(K, N)) return QDG_ESHAPE;
    if (O >= (int64_t(1) << 31)) return QDG_ESHAPE;
    if (!aligned(W, 16) || !aligned(xq, 2) || !aligned(y, 4) || !aligned(dbg, 4)) return QDG_EALIGN;
    const DeviceInfo dev = device_info();
    if (dev.device < 0) return QDG_ECUDA;
    const int nv = static_cast<int>(N);
    const PlanN plan = make_plan_n(K, nv);
    if (plan.nslots < 1 || plan.rch < 1) return QDG_ESHAPE;
    ArgsN a{};
    a.W = static_cast<const uint8_t*>(W);
    a.xq = static_cast<const uint8_t*>(xq);
    a.xq_bulk = aligned(xq, 16) ? 1 : 0;
    a.y = y;
    a.ldy = y ? ldy : 0;
    a.dbg = dbg;
    a.O = O;
    const int grid = static_cast<int>(std::min<int64_t>(dev.sms, O));
    // nv vectors of up to 512 blocks: up to 4 x 512 x 34 bytes, past the default 48 KB
    const size_t smem = a.xq_bulk ? static_cast<size_t>(nv) * plan.nb * 34 : 0;
    const int rc = nv == 3 ? launch_nv<3>(a, plan, grid, smem, stream, dbg != nullptr)
                           : launch_nv<4>(a, plan, grid, smem, stream, dbg != nullptr);
    if (rc != QDG_OK) return rc;
    count_launch(13);
    return QDG_OK;
}

unsigned flags_read_clear_gemv_segn(cudaStream_t stream) {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_flags_gemv_segn, sizeof(v), 0, cudaMemcpyDeviceToHost, stream) !=
        cudaSuccess)
        return ~0u;
    if (cudaMemcpyToSymbolAsync(g_flags_gemv_segn, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream) !=
        cudaSuccess)
        return ~0u;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return ~0u;
    return v;
}

}  // namespace qdg
