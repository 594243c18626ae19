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
constexpr int kL2Prefetch = 96 * 1024;      // bytes of W prefetched into L2 per CTA at start
constexpr int kFusedMaxK = 16384;           // fused form stages x and gamma in shared memory
constexpr uint32_t kNibbles = 0x0F0F0F0Fu;

// Weight types.  A lane owns one pair of consecutive blocks per segment of
// 32 pairs.  Q4_0: 18-byte blocks, 36-byte pairs, 1152-byte segments read as
// three 16-byte loads per lane, three segments in flight per warp.  Q8_0:
// 34-byte blocks, 68-byte pairs, 2176-byte segments read as five loads per
// lane, two segments in flight (about the same registers, more bytes).
enum { kQ4 = 0, kQ8 = 1 };
template <int kW>
struct WT {
    static constexpr int kBlockBytes = kW == kQ4 ? 18 : 34;
    static constexpr int kPairBytes = 2 * kBlockBytes;
    static constexpr int kSegBytes = 32 * kPairBytes;
    static constexpr int kLoads = (kSegBytes / 16 + 31) / 32;
    static constexpr int kDepth = kW == kQ4 ? 3 : 2;
    static constexpr int kPartFloats = kW == kQ4 ? 4096 : 2048;   // per-chunk partial sums (rows x segments)
};

struct Plan {
    int rowbytes;   // K/32 * block bytes
    int nb;         // K/32
    int P;          // block pairs per row (K/64)
    int nseg;       // segments per row, ceil(P / 32)
    int nslots;     // rows in flight per CTA = kWarps / nseg
    int rch;        // rows per chunk (partial-sum buffer capacity), multiple of nslots
};

template <int kW>
Plan make_plan(int64_t K) {
    Plan p{};
    p.nb = static_cast<int>(K / 32);
    p.rowbytes = p.nb * WT<kW>::kBlockBytes;
    p.P = static_cast<int>(K / 64);
    p.nseg = (p.P + 31) / 32;
    p.nslots = kWarps / p.nseg;
    p.rch = (WT<kW>::kPartFloats / p.nseg) / p.nslots * p.nslots;
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

// The 16-byte chunks of one row-segment held by a lane: indices lane, lane+32, ...
template <int kW>
struct SegRegs {
    uint4 v[WT<kW>::kLoads];
};

constexpr int kMaxGroup = 4;   // matrices sharing one input in a grouped launch

struct Args {
    // Grouped launch: matrices g = 0..ng-1 (same K, same input) are stacked;
    // global row r belongs to the last g with start[g] <= r.
    const uint8_t* Wg[kMaxGroup];
    float* yg[kMaxGroup];
    int64_t start[kMaxGroup];
    int ng;
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

// 96 registers a thread (no spills): one CTA of 512 threads then leaves room
// on its SM for a CTA of the quantize kernel, so the next vector's quantize
// can be resident, and start, while this product is still streaming.
template <int kW, bool kFused, bool kDebug>
__global__ void __maxnreg__(96) gemv_kernel(const Args a, Plan plan) {
    using T = WT<kW>;
    constexpr int kDepth = T::kDepth;
    constexpr int kSegBytes = T::kSegBytes;
    __shared__ __align__(16) uint8_t seg_buf[kWarps][kSegBytes];
    __shared__ float part[T::kPartFloats];
    __shared__ float norm_part[8];
    // fused form only: x [K] fp32, gamma [K] fp32, Q8_0 activations [K/32 x 34 B]
    extern __shared__ __align__(16) uint8_t fused_smem[];
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
    const int seg_vec = worker ? (min(plan.P, seg * 32 + 32) - seg * 32) * T::kPairBytes / 16 : 0;

    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * O / gridDim.x;
    const int64_t r1 = static_cast<int64_t>(blockIdx.x + 1) * O / gridDim.x;
    const int nrows = static_cast<int>(r1 - r0);

    pdl_trigger();

    SegRegs<kW> pipe[kDepth];
    auto load_seg = [&](int64_t row, SegRegs<kW>& s) {
        int g = 0;
#pragma unroll
        for (int i = 1; i < kMaxGroup; ++i)
            if (i < a.ng && row >= a.start[i]) g = i;
        const uint8_t* base = a.Wg[g] + (row - a.start[g]) * plan.rowbytes + seg_off;
#pragma unroll
        for (int k = 0; k < T::kLoads; ++k) {
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

    // ---- the first chunk's leading row-segments (W only) before the wait,
    // plus an L2 prefetch of the rows after them (up to kL2Prefetch bytes per
    // CTA) so the weight stream keeps flowing while the prologue runs.
    if (worker) fill(r0, min(nrows, plan.rch));
    if (threadIdx.x == 0) {
        // rows [r0 + ahead, r0 + ahead + n) may span matrices of the group
        int64_t row = r0 + static_cast<int64_t>(kDepth) * plan.nslots;
        int64_t budget = kL2Prefetch / plan.rowbytes;
        for (int g = 0; g < a.ng && budget > 0; ++g) {
            const int64_t gend = (g + 1 < a.ng) ? a.start[g + 1] : O;
            if (row >= gend || row >= r1) continue;
            const int64_t n = min(min(gend, r1) - row, budget);
            if (n > 0) {
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a.Wg[g] + (row - a.start[g]) *
                                                                                           plan.rowbytes),
                             "r"(static_cast<uint32_t>(n * plan.rowbytes))
                             : "memory");
                row += n;
                budget -= n;
            }
        }
    }

    pdl_wait();

    // ---- activations of this lane's pair, kept in registers
    uint32_t xa[8], xb[8];
    float dxa = 0.0f, dxb = 0.0f;
    int sa = 0, sb = 0;
    if (kFused) {
        const int K = a.K;
        const int nb = K >> 5;
        float* xs = reinterpret_cast<float*>(fused_smem);
        float* gs = xs + K;
        uint8_t* xqs = reinterpret_cast<uint8_t*>(gs + K);
        // (1) stage x and gamma with one wave of 16-byte loads
        {
            const float4* x4 = reinterpret_cast<const float4*>(a.x);
            const float4* g4 = reinterpret_cast<const float4*>(a.gamma);
            for (int i = threadIdx.x; i < K / 4; i += kThreads) {
                reinterpret_cast<float4*>(xs)[i] = __ldg(x4 + i);
                if (a.gamma != nullptr) reinterpret_cast<float4*>(gs)[i] = __ldg(g4 + i);
            }
        }
        __syncthreads();
        // (2) RMS statistic in the library's fixed order: chain j (threads
        // 0..255) sums x_i^2 over i = j (mod 256) ascending with fma; warp
        // butterflies; ((w0+w1)+(w2+w3))+((w4+w5)+(w6+w7)).
        float s = 1.0f;
        if (a.gamma != nullptr) {
            if (threadIdx.x < 256) {
                float acc = 0.0f;
                for (int i = threadIdx.x; i < K; i += 256) acc = __fmaf_rn(xs[i], xs[i], acc);
                acc = warp_sum(acc);
                if (lane == 0) norm_part[warp] = acc;
            }
            __syncthreads();
            const float ss = __fadd_rn(__fadd_rn(__fadd_rn(norm_part[0], norm_part[1]), __fadd_rn(norm_part[2], norm_part[3])),
                                       __fadd_rn(__fadd_rn(norm_part[4], norm_part[5]), __fadd_rn(norm_part[6], norm_part[7])));
            const float mean = __fdiv_rn(ss, static_cast<float>(K));
            s = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, a.eps)));
        }
        // (3) Q8_0 blocks, one per warp at a time (lane = element), four
        // independent blocks interleaved; the arithmetic of the standalone
        // quantize kernel: v = (x*s)*gamma, d = max|v|/127, q = round(v/d).
        for (int b0 = warp; b0 < nb; b0 += 4 * kWarps) {
            float v[4], d[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int b = b0 + u * kWarps;
                v[u] = 0.0f;
                if (b < nb) {
                    v[u] = xs[(b << 5) + lane];
                    if (a.gamma != nullptr) v[u] = __fmul_rn(__fmul_rn(v[u], s), gs[(b << 5) + lane]);
                }
                d[u] = fabsf(v[u]);
            }
#pragma unroll
            for (int h = 16; h >= 1; h >>= 1)
#pragma unroll
                for (int u = 0; u < 4; ++u) d[u] = fmaxf(d[u], __shfl_xor_sync(0xffffffffu, d[u], h));
            // the four blocks' divisions and roundings are independent: all
            // first (a block past nb has v = 0 and gives q = 0), then the
            // stores, so that the four dependent chains overlap
            float dd[4];
            int q[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                dd[u] = __fdiv_rn(d[u], 127.0f);
                q[u] = 0;
                if (dd[u] != 0.0f) {
                    float r = roundf(__fdiv_rn(v[u], dd[u]));
                    r = fminf(fmaxf(r, -127.0f), 127.0f);
                    q[u] = static_cast<int>(r);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int b = b0 + u * kWarps;
                if (b < nb) {
                    uint8_t* blk = xqs + b * 34;
                    if (lane == 0) {
                        const __half dh = __float2half_rn(dd[u]);
                        *reinterpret_cast<unsigned short*>(blk) = __half_as_ushort(dh);
                        if (__hisinf(dh)) atomicOr(&g_flags_gemv, FLAG_OVERFLOW);
                    }
                    blk[2 + lane] = static_cast<uint8_t>(static_cast<int8_t>(q[u]));
                }
            }
        }
        __syncthreads();
        if (a.xq_out != nullptr && blockIdx.x == 0) {
            const uint32_t* src = reinterpret_cast<const uint32_t*>(xqs);
            uint32_t* dst = reinterpret_cast<uint32_t*>(a.xq_out);
            for (int i = threadIdx.x; i < nb * 34 / 4; i += kThreads) dst[i] = src[i];
        }
        // (4) this lane's pair, from shared memory
        if (active) {
            const uint32_t* xp = reinterpret_cast<const uint32_t*>(xqs + static_cast<size_t>(p) * 68);
            uint32_t w[17];
#pragma unroll
            for (int i = 0; i < 17; ++i) w[i] = xp[i];
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
    auto consume = [&](int64_t c0, int crows, int ri, SegRegs<kW>& entry) -> float {
        // Store first (this waits for the entry's loads, issued kDepth steps
        // ago), then reuse the same registers for the segment kDepth ahead.
#pragma unroll
        for (int q = 0; q < T::kLoads; ++q) {
            const int idx = lane + 32 * q;
            if (idx < seg_vec) *reinterpret_cast<uint4*>(buf + idx * 16) = entry.v[q];
        }
        const int ahead = ri + kDepth * plan.nslots;
        if (ahead < crows) load_seg(c0 + ahead, entry);
        __syncwarp();
        float acc = 0.0f;
        if (active) {
            int ia, ib;
            float dwa, dwb;
            if (kW == kQ4) {
                const uint32_t* wp = reinterpret_cast<const uint32_t*>(buf + lane * 36);
                uint32_t w[9];
#pragma unroll
                for (int i = 0; i < 9; ++i) w[i] = wp[i];
                ia = block_dot(bytes_2_to_5(w[0], w[1]), bytes_2_to_5(w[1], w[2]), bytes_2_to_5(w[2], w[3]),
                               bytes_2_to_5(w[3], w[4]), xa) -
                     8 * sa;
                ib = block_dot(w[5], w[6], w[7], w[8], xb) - 8 * sb;
                dwa = half_bits_to_float(w[0]);
                dwb = half_bits_to_float(w[4] >> 16);
            } else {
                // Q8_0 pair: scale a, 32 codes of a (bytes 2..33), scale b, 32 codes of b (word aligned)
                const uint32_t* wp = reinterpret_cast<const uint32_t*>(buf + lane * 68);
                uint32_t w[17];
#pragma unroll
                for (int i = 0; i < 17; ++i) w[i] = wp[i];
                ia = 0;
                ib = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    ia = __dp4a(static_cast<int>(bytes_2_to_5(w[i], w[i + 1])), static_cast<int>(xa[i]), ia);
                    ib = __dp4a(static_cast<int>(w[9 + i]), static_cast<int>(xb[i]), ib);
                }
                dwa = half_bits_to_float(w[0]);
                dwb = half_bits_to_float(w[8] >> 16);
            }
            acc = __fmul_rn(__fmul_rn(dwa, dxa), static_cast<float>(ia));
            acc = __fmaf_rn(__fmul_rn(dwb, dxb), static_cast<float>(ib), acc);
            if (kDebug) {
                int32_t* d = dbg + (c0 + ri) * plan.nb + 2 * p;
                d[0] = ia;
                d[1] = ib;
            }
        }
        __syncwarp();
        if (kW == kQ4) {
            acc = warp_sum(acc);
            if (lane == 0) part[ri * nseg + seg] = acc;
        }
        return acc;
    };
    // Q8_0 weights: two row-segments (rows ri and ri2) reduced in one
    // butterfly; after the first exchange lanes 0..15 carry row ri and lanes
    // 16..31 row ri2, each summed in the order of a plain warp reduction.
    auto reduce2 = [&](int ri, int ri2, bool two, float acc0, float acc1) {
        const bool upper = (lane & 16) != 0;
        float v = upper ? acc1 : acc0;
        v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, upper ? acc0 : acc1, 16));
#pragma unroll
        for (int h = 8; h >= 1; h >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, h));
        if (lane == 0) part[ri * nseg + seg] = v;
        if (lane == 16 && two) part[ri2 * nseg + seg] = v;
    };

    for (int64_t c0 = r0; c0 < r1; c0 += plan.rch) {
        const int crows = static_cast<int>((r1 - c0) < plan.rch ? (r1 - c0) : plan.rch);
        if (worker) {
            if (c0 != r0) fill(c0, crows);
            // The ring is consumed in a loop unrolled by its depth so every
            // access to it uses a compile-time index: each step then waits only
            // for its own loads, issued kDepth steps earlier.
            const int step = plan.nslots;
            if (kW == kQ8) {
                for (int ri = slot; ri < crows; ri += 2 * step) {
                    const float p0 = consume(c0, crows, ri, pipe[0]);
                    const bool two = ri + step < crows;
                    const float p1 = two ? consume(c0, crows, ri + step, pipe[1]) : 0.0f;
                    reduce2(ri, ri + step, two, p0, p1);
                }
            } else {
                for (int ri = slot; ri < crows; ri += kDepth * step) {
                    consume(c0, crows, ri, pipe[0]);
                    if (ri + step < crows) consume(c0, crows, ri + step, pipe[1]);
                    if (kDepth > 2 && ri + 2 * step < crows)
                        consume(c0, crows, ri + 2 * step, pipe[kDepth > 2 ? 2 : 0]);
                }
            }
        }
        __syncthreads();
        if (!kDebug) {
            for (int t = threadIdx.x; t < crows; t += kThreads) {
                float v = part[t * nseg];
                for (int g = 1; g < nseg; ++g) v = __fadd_rn(v, part[t * nseg + g]);
                const int64_t row = c0 + t;
                int g = 0;
#pragma unroll
                for (int i = 1; i < kMaxGroup; ++i)
                    if (i < a.ng && row >= a.start[i]) g = i;
                a.yg[g][row - a.start[g]] = v;
            }
        }
        __syncthreads();
    }
}

template <int kW>
int gemv_launch_typed(const void* const* W, float* const* y, const int64_t* O, int count, const void* xq, int64_t K,
                      cudaStream_t stream, int32_t* dbg) {
    if (!W || !O || !xq || (!y && !dbg)) return QDG_EINVAL;
    if (count < 1 || count > kMaxGroup || K <= 0) return QDG_EINVAL;
    if (dbg && count != 1) return QDG_EINVAL;
    if (K % 256 != 0 || K > 32768) return QDG_ESHAPE;
    if (!aligned(xq, 4) || !aligned(dbg, 4)) return QDG_EALIGN;
    Args a{};
    int64_t total = 0;
    for (int g = 0; g < count; ++g) {
        if (!W[g] || (!dbg && !y[g]) || O[g] <= 0) return QDG_EINVAL;
        if (!aligned(W[g], 16) || (y && !aligned(y[g], 4))) return QDG_EALIGN;
        a.Wg[g] = static_cast<const uint8_t*>(W[g]);
        a.yg[g] = y ? y[g] : nullptr;
        a.start[g] = total;
        total += O[g];
    }
    if (total >= (int64_t(1) << 31)) return QDG_ESHAPE;
    const DeviceInfo dev = device_info();
    if (dev.device < 0) return QDG_ECUDA;
    const Plan plan = make_plan<kW>(K);
    const int grid = static_cast<int>(std::min<int64_t>(dev.sms, total));
    a.ng = count;
    a.W = a.Wg[0];
    a.xq = static_cast<const uint8_t*>(xq);
    a.y = a.yg[0];
    a.dbg = dbg;
    a.O = total;
    a.K = static_cast<int>(K);
    cudaError_t e;
    if (dbg)
        e = launch(gemv_kernel<kW, false, true>, dim3(grid), dim3(kThreads), 0, stream, false, a, plan);
    else
        e = launch(gemv_kernel<kW, false, false>, dim3(grid), dim3(kThreads), 0, stream, true, a, plan);
    if (e != cudaSuccess) return QDG_ECUDA;
    count_launch(kW == kQ4 ? 1 : 8);
    return QDG_OK;
}

}  // namespace

int gemv_launch_group(const void* const* W, float* const* y, const int64_t* O, int count, const void* xq, int64_t K,
                      cudaStream_t stream, int32_t* dbg) {
    return gemv_launch_typed<kQ4>(W, y, O, count, xq, K, stream, dbg);
}

int gemv_q8w_launch_group(const void* const* W, float* const* y, const int64_t* O, int count, const void* xq,
                          int64_t K, cudaStream_t stream, int32_t* dbg) {
    return gemv_launch_typed<kQ8>(W, y, O, count, xq, K, stream, dbg);
}

int gemv_q8w_launch(const void* W, const void* xq, float* y, int64_t O, int64_t K, cudaStream_t stream,
                    int32_t* dbg) {
    float* ys[1] = {y};
    return gemv_q8w_launch_group(&W, y ? ys : nullptr, &O, 1, xq, K, stream, dbg);
}

int gemv_launch(const void* W, const void* xq, float* y, int64_t O, int64_t K, cudaStream_t stream, int32_t* dbg) {
    float* ys[1] = {y};
    return gemv_launch_group(&W, y ? ys : nullptr, &O, 1, xq, K, stream, dbg);
}

int gemv_rmsnorm_launch(const void* const* W, float* const* y, const int64_t* O, int count, const float* x,
                        const float* gamma, float eps, int64_t K, void* xq_out, cudaStream_t stream) {
    if (!W || !y || !O || !x) return QDG_EINVAL;
    if (count < 1 || count > kMaxGroup || K <= 0) return QDG_EINVAL;
    if (!(eps >= 0.0f) || std::isinf(eps)) return QDG_EINVAL;
    if (K % 256 != 0 || K > kFusedMaxK) return QDG_ESHAPE;
    if (!aligned(x, 16) || (gamma && !aligned(gamma, 16)) || !aligned(xq_out, 4)) return QDG_EALIGN;
    Args a{};
    int64_t total = 0;
    for (int g = 0; g < count; ++g) {
        if (!W[g] || !y[g] || O[g] <= 0) return QDG_EINVAL;
        if (!aligned(W[g], 16) || !aligned(y[g], 4)) return QDG_EALIGN;
        a.Wg[g] = static_cast<const uint8_t*>(W[g]);
        a.yg[g] = y[g];
        a.start[g] = total;
        total += O[g];
    }
    if (total >= (int64_t(1) << 31)) return QDG_ESHAPE;
    const DeviceInfo dev = device_info();
    if (dev.device < 0) return QDG_ECUDA;
    const Plan plan = make_plan<kQ4>(K);
    const int grid = static_cast<int>(std::min<int64_t>(dev.sms, total));
    a.ng = count;
    a.W = a.Wg[0];
    a.x = x;
    a.gamma = gamma;
    a.eps = eps;
    a.xq_out = static_cast<uint8_t*>(xq_out);
    a.y = a.yg[0];
    a.O = total;
    a.K = static_cast<int>(K);
    const size_t smem = static_cast<size_t>(8) * K + static_cast<size_t>(K / 32) * 34;
    if (ensure_smem_limit(reinterpret_cast<const void*>(gemv_kernel<kQ4, true, false>), smem) != cudaSuccess)
        return QDG_ECUDA;
    const cudaError_t e = launch(gemv_kernel<kQ4, true, false>, dim3(grid), dim3(kThreads), smem, stream, true, a, plan);
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

extern "C" int q4_0_q8_0_gemv_group(const void* const* W, float* const* y, const int64_t* O, int count,
                                    const void* xq, int64_t K, qdg_stream_t stream) {
    if (!y) return QDG_EINVAL;
    return qdg::gemv_launch_group(W, y, O, count, xq, K, reinterpret_cast<cudaStream_t>(stream), nullptr);
}

extern "C" int q4_0_gemv_rmsnorm(const void* W, const float* x, const float* gamma, float eps, float* y, int64_t O,
                                 int64_t K, void* xq_out, qdg_stream_t stream) {
    return qdg::gemv_rmsnorm_launch(&W, &y, &O, 1, x, gamma, eps, K, xq_out, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int q4_0_gemv_rmsnorm_group(const void* const* W, float* const* y, const int64_t* O, int count,
                                       const float* x, const float* gamma, float eps, int64_t K, void* xq_out,
                                       qdg_stream_t stream) {
    return qdg::gemv_rmsnorm_launch(W, y, O, count, x, gamma, eps, K, xq_out, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int q8_0_q8_0_gemv(const void* W, const void* xq, float* y, int64_t O, int64_t K, qdg_stream_t stream) {
    if (!y) return QDG_EINVAL;
    return qdg::gemv_q8w_launch(W, xq, y, O, K, reinterpret_cast<cudaStream_t>(stream), nullptr);
}

extern "C" int q8_0_q8_0_gemv_group(const void* const* W, float* const* y, const int64_t* O, int count,
                                    const void* xq, int64_t K, qdg_stream_t stream) {
    if (!y) return QDG_EINVAL;
    return qdg::gemv_q8w_launch_group(W, y, O, count, xq, K, reinterpret_cast<cudaStream_t>(stream), nullptr);
}
