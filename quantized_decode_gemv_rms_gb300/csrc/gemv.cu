// gemv.cu -- batch-1 Q4_0 x Q8_0 matrix-vector product (the "mmvq" route of
// batch-1 decode [GGML: Backend abstraction and hardware acceleration,
// section "CUDA: mmvq, mmq, cublas -- three matrix paths"]).
//
// The product is bound by the weight stream: 4.5 bits per weight, read once
// from HBM, against a few integer operations per weight.  Design (chosen by
// measurement on GB300: plain 16-byte loads with enough bytes in flight
// stream HBM faster than the bulk-copy engine fed through a barrier ring):
//   * A row of K weights is split into segments of 32 block pairs (2048
//     weights, 1152 bytes).  Lane l of a warp owns pair l of its segment and
//     keeps the matching 64 Q8_0 activations in registers for the whole
//     kernel.
//   * Each CTA owns a contiguous range of rows; warp w works on segment
//     w % nseg of rows slot, slot + nslots, ... (slot = w / nseg).  For every
//     row-segment the warp reads its 1152 bytes with coalesced 16-byte loads
//     (L1 bypassed), issued kDepth row-segments ahead of use, so each SM keeps
//     tens of kilobytes in flight.
//   * The 18-byte blocks are only 2-byte aligned, so the warp passes the
//     segment through a private shared-memory buffer: coalesced 16-byte
//     stores, then each lane reads its 36-byte pair as nine conflict-free
//     32-bit loads, unpacks the nibbles, forms the exact block sums with dp4a
//     (minus 8 * sum(q_x)), scales by d_w * d_x (exact in fp32), and the warp
//     reduces with shuffles.
//   * Segment partials are combined per row in a fixed order, so results are
//     deterministic.
//   * Programmatic dependent launch (optional): the first row-segments of W
//     are requested before the kernel waits for the preceding grid;
//     activations are read and y is written only after the wait.
#include "common.cuh"

#include <algorithm>

namespace qdg {

static __device__ unsigned g_flags_gemv;

namespace {

constexpr int kWarps = 16;
constexpr int kThreads = 32 * kWarps;
constexpr int kDepth = 3;                   // row-segments in flight per warp (the consume loop is unrolled by 3)
constexpr int kSegBytes = 1152;             // 32 pairs x 36 bytes
constexpr int kPartFloats = 4096;           // per-chunk partial sums (rows x segments)
constexpr uint32_t kNibbles = 0x0F0F0F0Fu;

struct Plan {
    int rowbytes;   // K/32 * 18
    int nb;         // K/32
    int P;          // block pairs per row (K/64)
    int nseg;       // segments per row, ceil(P / 32)
    int nslots;     // rows in flight per CTA = kWarps / nseg
    int rch;        // rows per chunk (partial-sum buffer capacity), multiple of nslots
};

Plan make_plan(int64_t K) {
    Plan p{};
    p.nb = static_cast<int>(K / 32);
    p.rowbytes = p.nb * 18;
    p.P = static_cast<int>(K / 64);
    p.nseg = (p.P + 31) / 32;
    p.nslots = kWarps / p.nseg;
    p.rch = (kPartFloats / p.nseg) / p.nslots * p.nslots;
    return p;
}

__device__ __forceinline__ uint4 ldg_stream(const uint8_t* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
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

// The 16-byte chunks of one row-segment held by a lane: indices lane, lane+32, lane+64.
struct SegRegs {
    uint4 v[3];
};

struct Args {
    const uint8_t* W;
    const uint8_t* xq;      // Q8_0 activations (unfused form)
    const float* x;         // fp32 activations (fused form)
    const float* gamma;     // fused form: NULL = plain quantization
    uint8_t* xq_out;        // fused form: optional copy of the Q8_0 activations (written by CTA 0)
    float* y;
    int32_t* dbg;
    int64_t O;
    int K;
    float eps;
};

// Fused form: RMS_NORM * gamma -> Q8_0 of the two blocks of pair p, computed by
// the lane that owns the pair, with exactly the arithmetic of the standalone
// quantize kernel (same s, same products, same IEEE divisions and rounding).
__device__ __forceinline__ void quantize_pair(const float* __restrict__ x, const float* __restrict__ gamma, float s,
                                              int p, uint32_t (&xa)[8], uint32_t (&xb)[8], float& dxa, float& dxb,
                                              int& sa, int& sb, uint32_t (&blk)[17]) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const float4* xv = reinterpret_cast<const float4*>(x + p * 64 + half * 32);
        const float4* gv = reinterpret_cast<const float4*>(gamma + p * 64 + half * 32);
        float v[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 a = __ldg(xv + i);
            v[4 * i] = a.x;
            v[4 * i + 1] = a.y;
            v[4 * i + 2] = a.z;
            v[4 * i + 3] = a.w;
        }
        if (gamma != nullptr) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 g = __ldg(gv + i);
                v[4 * i] = __fmul_rn(__fmul_rn(v[4 * i], s), g.x);
                v[4 * i + 1] = __fmul_rn(__fmul_rn(v[4 * i + 1], s), g.y);
                v[4 * i + 2] = __fmul_rn(__fmul_rn(v[4 * i + 2], s), g.z);
                v[4 * i + 3] = __fmul_rn(__fmul_rn(v[4 * i + 3], s), g.w);
            }
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
        const float d = __fdiv_rn(amax, 127.0f);
        const __half dh = __float2half_rn(d);
        if (__hisinf(dh)) atomicOr(&g_flags_gemv, FLAG_OVERFLOW);
        uint32_t w[8];
        int qs = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t word = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                int q = 0;
                if (d != 0.0f) {
                    float r = roundf(__fdiv_rn(v[4 * i + j], d));
                    r = fminf(fmaxf(r, -127.0f), 127.0f);
                    q = static_cast<int>(r);
                }
                qs += q;
                word |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * j);
            }
            w[i] = word;
        }
        const uint32_t dbits = __half_as_ushort(dh);
        if (half == 0) {
#pragma unroll
            for (int i = 0; i < 8; ++i) xa[i] = w[i];
            dxa = __half2float(dh);
            sa = qs;
            // Q8_0 block bytes: d (2 bytes) then 32 q, packed into the 68-byte pair
            blk[0] = dbits | (w[0] << 16);
#pragma unroll
            for (int i = 1; i < 8; ++i) blk[i] = (w[i - 1] >> 16) | (w[i] << 16);
            blk[8] = w[7] >> 16;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) xb[i] = w[i];
            dxb = __half2float(dh);
            sb = qs;
            blk[8] |= dbits << 16;
#pragma unroll
            for (int i = 0; i < 8; ++i) blk[9 + i] = w[i];
        }
    }
}

template <bool kFused, bool kDebug>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const Args a, Plan plan) {
    __shared__ __align__(16) uint8_t seg_buf[kWarps][kSegBytes];
    __shared__ float part[kPartFloats];
    __shared__ float norm_part[8];
    const uint8_t* __restrict__ W = a.W;
    float* __restrict__ y = a.y;
    int32_t* __restrict__ dbg = a.dbg;
    const int64_t O = a.O;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nseg = plan.nseg;
    const int seg = warp % nseg;
    const int slot = warp / nseg;
    const bool worker = slot < plan.nslots;   // warps beyond nslots * nseg stay idle
    const int p = seg * 32 + lane;            // block pair owned by this lane
    const bool active = worker && p < plan.P;
    // this warp's segment within a row: byte offset and number of 16-byte chunks
    const int seg_off = seg * kSegBytes;
    const int seg_vec = worker ? (min(plan.P, seg * 32 + 32) - seg * 32) * 36 / 16 : 0;

    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * O / gridDim.x;
    const int64_t r1 = static_cast<int64_t>(blockIdx.x + 1) * O / gridDim.x;
    const int nrows = static_cast<int>(r1 - r0);

    pdl_trigger();

    SegRegs pipe[kDepth];
    auto load_seg = [&](int64_t row, SegRegs& s) {
        const uint8_t* base = W + row * plan.rowbytes + seg_off;
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            const int idx = lane + 32 * k;
            if (idx < seg_vec) s.v[k] = ldg_stream(base + idx * 16);
        }
    };
    auto fill = [&](int64_t c0, int crows) {
#pragma unroll
        for (int d = 0; d < kDepth; ++d) {
            const int ri = slot + d * plan.nslots;
            if (ri < crows) load_seg(c0 + ri, pipe[d]);
        }
    };

    // ---- the first chunk's leading row-segments (W only) before the wait
    if (worker) fill(r0, min(nrows, plan.rch));

    pdl_wait();

    // ---- activations of this lane's pair, kept in registers
    uint32_t xa[8], xb[8];
    float dxa = 0.0f, dxb = 0.0f;
    int sa = 0, sb = 0;
    if (kFused) {
        // RMS statistic in the library's fixed order: chain j (threads 0..255)
        // sums x_i^2 over i = j (mod 256) ascending with fma; warp butterflies;
        // ((w0+w1)+(w2+w3))+((w4+w5)+(w6+w7)).
        float s = 1.0f;
        if (a.gamma != nullptr) {
            if (threadIdx.x < 256) {
                float acc = 0.0f;
                for (int i0 = threadIdx.x; i0 < a.K; i0 += 256 * 8) {
                    float v[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int i = i0 + u * 256;
                        v[u] = i < a.K ? __ldg(a.x + i) : 0.0f;
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (i0 + u * 256 < a.K) acc = __fmaf_rn(v[u], v[u], acc);
                }
                acc = warp_sum(acc);
                if (lane == 0) norm_part[warp] = acc;
            }
            __syncthreads();
            const float ss = __fadd_rn(__fadd_rn(__fadd_rn(norm_part[0], norm_part[1]), __fadd_rn(norm_part[2], norm_part[3])),
                                       __fadd_rn(__fadd_rn(norm_part[4], norm_part[5]), __fadd_rn(norm_part[6], norm_part[7])));
            const float mean = __fdiv_rn(ss, static_cast<float>(a.K));
            s = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, a.eps)));
        }
        if (active) {
            uint32_t blk[17];
            quantize_pair(a.x, a.gamma, s, p, xa, xb, dxa, dxb, sa, sb, blk);
            if (a.xq_out != nullptr && blockIdx.x == 0 && slot == 0) {
                uint32_t* dst = reinterpret_cast<uint32_t*>(a.xq_out + static_cast<size_t>(p) * 68);
#pragma unroll
                for (int i = 0; i < 17; ++i) dst[i] = blk[i];
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) xa[i] = xb[i] = 0u;
        }
    } else if (active) {
        const uint32_t* xp = reinterpret_cast<const uint32_t*>(a.xq + static_cast<size_t>(p) * 68);
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

    uint8_t* buf = seg_buf[warp];
    // One row-segment: stage it through shared memory, refill its ring entry
    // with the segment kDepth ahead, dot it, reduce it.
    auto consume = [&](int64_t c0, int crows, int ri, SegRegs& entry) {
        // Store first (this waits for the entry's loads, issued kDepth steps
        // ago), then reuse the same registers for the segment kDepth ahead.
#pragma unroll
        for (int q = 0; q < 3; ++q) {
            const int idx = lane + 32 * q;
            if (idx < seg_vec) *reinterpret_cast<uint4*>(buf + idx * 16) = entry.v[q];
        }
        const int ahead = ri + kDepth * plan.nslots;
        if (ahead < crows) load_seg(c0 + ahead, entry);
        __syncwarp();
        float acc = 0.0f;
        if (active) {
            const uint32_t* wp = reinterpret_cast<const uint32_t*>(buf + lane * 36);
            uint32_t w[9];
#pragma unroll
            for (int i = 0; i < 9; ++i) w[i] = wp[i];
            const int ia = block_dot(bytes_2_to_5(w[0], w[1]), bytes_2_to_5(w[1], w[2]), bytes_2_to_5(w[2], w[3]),
                                     bytes_2_to_5(w[3], w[4]), xa) -
                           8 * sa;
            const int ib = block_dot(w[5], w[6], w[7], w[8], xb) - 8 * sb;
            const float dwa = half_bits_to_float(w[0]);
            const float dwb = half_bits_to_float(w[4] >> 16);
            acc = __fmul_rn(__fmul_rn(dwa, dxa), static_cast<float>(ia));
            acc = __fmaf_rn(__fmul_rn(dwb, dxb), static_cast<float>(ib), acc);
            if (kDebug) {
                int32_t* d = dbg + (c0 + ri) * plan.nb + 2 * p;
                d[0] = ia;
                d[1] = ib;
            }
        }
        __syncwarp();
        acc = warp_sum(acc);
        if (lane == 0) part[ri * nseg + seg] = acc;
    };

    for (int64_t c0 = r0; c0 < r1; c0 += plan.rch) {
        const int crows = static_cast<int>((r1 - c0) < plan.rch ? (r1 - c0) : plan.rch);
        if (worker) {
            if (c0 != r0) fill(c0, crows);
            // The ring is consumed in a loop unrolled by its depth so every
            // access to it uses a compile-time index: each step then waits only
            // for its own loads, issued kDepth steps earlier.
            const int step = plan.nslots;
            for (int ri = slot; ri < crows; ri += kDepth * step) {
                consume(c0, crows, ri, pipe[0]);
                if (ri + step < crows) consume(c0, crows, ri + step, pipe[1]);
                if (ri + 2 * step < crows) consume(c0, crows, ri + 2 * step, pipe[2]);
            }
        }
        __syncthreads();
        if (!kDebug) {
            for (int t = threadIdx.x; t < crows; t += kThreads) {
                float v = part[t * nseg];
                for (int g = 1; g < nseg; ++g) v = __fadd_rn(v, part[t * nseg + g]);
                y[c0 + t] = v;
            }
        }
        __syncthreads();
    }
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
    const int grid = static_cast<int>(std::min<int64_t>(dev.sms, O));
    Args a{};
    a.W = static_cast<const uint8_t*>(W);
    a.xq = static_cast<const uint8_t*>(xq);
    a.y = y;
    a.dbg = dbg;
    a.O = O;
    a.K = static_cast<int>(K);
    cudaError_t e;
    if (dbg)
        e = launch(gemv_kernel<false, true>, dim3(grid), dim3(kThreads), 0, stream, false, a, plan);
    else
        e = launch(gemv_kernel<false, false>, dim3(grid), dim3(kThreads), 0, stream, true, a, plan);
    if (e != cudaSuccess) return QDG_ECUDA;
    count_launch(1);
    return QDG_OK;
}

int gemv_rmsnorm_launch(const void* W, const float* x, const float* gamma, float eps, float* y, int64_t O, int64_t K,
                        void* xq_out, cudaStream_t stream) {
    if (!W || !x || !y) return QDG_EINVAL;
    if (O <= 0 || K <= 0) return QDG_EINVAL;
    if (!(eps >= 0.0f) || std::isinf(eps)) return QDG_EINVAL;
    if (K % 256 != 0 || K > 32768 || O >= (int64_t(1) << 31)) return QDG_ESHAPE;
    if (!aligned(W, 16) || !aligned(x, 16) || (gamma && !aligned(gamma, 16)) || !aligned(y, 4) ||
        !aligned(xq_out, 4))
        return QDG_EALIGN;
    const DeviceInfo dev = device_info();
    if (dev.device < 0) return QDG_ECUDA;
    const Plan plan = make_plan(K);
    const int grid = static_cast<int>(std::min<int64_t>(dev.sms, O));
    Args a{};
    a.W = static_cast<const uint8_t*>(W);
    a.x = x;
    a.gamma = gamma;
    a.eps = eps;
    a.xq_out = static_cast<uint8_t*>(xq_out);
    a.y = y;
    a.O = O;
    a.K = static_cast<int>(K);
    const cudaError_t e = launch(gemv_kernel<true, false>, dim3(grid), dim3(kThreads), 0, stream, true, a, plan);
    if (e != cudaSuccess) return QDG_ECUDA;
    count_launch(5);
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

extern "C" int q4_0_gemv_rmsnorm(const void* W, const float* x, const float* gamma, float eps, float* y, int64_t O,
                                 int64_t K, void* xq_out, qdg_stream_t stream) {
    return qdg::gemv_rmsnorm_launch(W, x, gamma, eps, y, O, K, xq_out, reinterpret_cast<cudaStream_t>(stream));
}
