// gemv_q4k.cu -- batch-1 product with Q4_K weights: y = W * x, W in 256-weight
// k-quant super-blocks, x in Q8_0 blocks.  The conversion step picks Q4_K or
// Q8_0 for weights and every back end's kernels must know each type [GGML:
// Backend abstraction and hardware acceleration, sections "How one production
// call lands on the hardware" and "Metal and Vulkan"]; the block format is
// the library's reading of GGML's super-block (144 bytes: fp16 d, fp16 dmin,
// twelve bytes of 6-bit sub-block scales and mins, 128 code bytes).
//
// A 144-byte super-block is nine 16-byte words, so unlike the 18-byte Q4_0
// block it can be read straight into registers with aligned 16-byte loads:
// no repack and no shared-memory staging.  The row/segment split is the one
// of the segment-layout Q4_0 kernel (gemv_seg.cu):
//   * a segment is 8 super-blocks (2048 weights, 1152 bytes); lane l of the
//     warp on segment s owns sub-blocks 2(l%4), 2(l%4)+1 of super-block
//     8s + l/4, i.e. weights 64(32s + l) .. +63, and so Q8_0 blocks
//     2(32s + l) and 2(32s + l) + 1 of the activations, kept in registers;
//   * per row-segment the lane loads the super-block header (the four lanes
//     of a super-block read the same 16 bytes) and its 32 code bytes (two
//     16-byte loads; a warp reads 1152 contiguous bytes), four row-segments
//     ahead of use;
//   * exact sub-block sums by dp4a (low nibbles against the first block,
//     high nibbles against the second), the 6-bit scale and min decoded
//     from the header, d_x (d sc isum - dmin m xsum) in fp32; the ring's
//     four rows share one transposed warp butterfly; segment partials are
//     combined per row in a fixed order (deterministic).
//
// Q5_K weights (the 5-bit k-quant beside Q4_K [llama.cpp b10981: OpenVINO
// backend optimises stateful decode and GPU MoE inference, section "GPU MoE,
// env vars"]; the library reads it as GGML's 176-byte super-block: the Q4_K
// header, 32 bytes qh with bit j of qh[i] the top bit (16) of element i of
// sub-block j, then the low four bits placed as the Q4_K codes) take the
// same kernel with kQ5: a segment is 8 super-blocks of 176 bytes, a lane
// also loads the 32 qh bytes (shared with the three other lanes of its
// super-block) and merges bits 2g and 2g+1 of each byte into its codes
// before the dp4a, so that q runs over 0..31.
#include "common.cuh"

#include <algorithm>

namespace qdg {

static __device__ unsigned g_flags_gemv_q4k;

namespace {

constexpr int kWarps = 16;
constexpr int kThreads = 32 * kWarps;
constexpr int kDepth = 4;                   // row-segments in flight per warp
constexpr int kPartFloats = 3072;
constexpr int kMaxGroup = 4;
constexpr uint32_t kNibbles = 0x0F0F0F0Fu;

struct Plan {
    int rowbytes;   // K/256 * 144
    int nb;         // K/32
    int nseg;       // ceil(K/2048)
    int slast;      // super-blocks in the last segment (1..8)
    int nslots;     // rows in flight per CTA = kWarps / nseg
    int rch;        // rows per chunk of partial sums, a multiple of nslots
};

// bytes of one super-block: Q4_K 144, Q5_K 176
template <bool kQ5>
constexpr int kSuper = kQ5 ? 176 : 144;

Plan make_plan(int64_t K, int sb_bytes) {
    Plan p{};
    const int nsb = static_cast<int>(K / 256);
    p.nb = static_cast<int>(K / 32);
    p.rowbytes = nsb * sb_bytes;
    p.nseg = (nsb + 7) / 8;
    p.slast = nsb - 8 * (p.nseg - 1);
    p.nslots = kWarps / p.nseg;
    p.rch = p.nslots > 0 ? (kPartFloats / p.nseg) / p.nslots * p.nslots : 0;
    return p;
}

__device__ __forceinline__ uint4 ldg_stream16(const uint8_t* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

struct Entry {
    uint4 h;        // d | dmin << 16, then the twelve scale bytes
    uint4 c0, c1;   // the pair's 32 code bytes (Q5_K: their low four bits)
    uint4 q0, q1;   // Q5_K: the super-block's 32 qh bytes (unused for Q4_K)
};

struct Args {
    const uint8_t* Wg[kMaxGroup];
    float* yg[kMaxGroup];
    int64_t start[kMaxGroup];
    int ng;
    const uint8_t* xq;
    int xq_bulk;
    int32_t* dbg;   // [O][K/32] exact sub-block sums instead of y
    int64_t O;
};

// Q8_0 block b of the activations from shared memory (2-byte loads: a
// 34-byte block is only 2-byte aligned): scale, 8 code words, code sum.
__device__ __forceinline__ void load_act(const uint8_t* xq, int b, uint32_t* x, float& d, int& sum) {
    const unsigned short* h = reinterpret_cast<const unsigned short*>(xq + static_cast<size_t>(b) * 34);
    d = half_bits_to_float(h[0]);
    sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        x[i] = static_cast<uint32_t>(h[1 + 2 * i]) | (static_cast<uint32_t>(h[2 + 2 * i]) << 16);
        sum = __dp4a(static_cast<int>(x[i]), 0x01010101, sum);
    }
}

// Q4_K: 96 registers a thread (a quantize CTA fits beside it on the decode
// step); Q5_K: 128, for its 80-byte ring entries.
template <bool kQ5, bool kDebug>
__global__ void __maxnreg__(kQ5 ? 128 : 96) gemv_q4k_kernel(const __grid_constant__ Args a,
                                                            const __grid_constant__ Plan plan) {
    __shared__ float part[kPartFloats];
    __shared__ uint64_t xbar;
    extern __shared__ __align__(16) uint8_t xs[];   // the Q8_0 vector when a.xq_bulk
    const int64_t O = a.O;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nseg = plan.nseg;
    const int seg = warp % nseg;
    const int slot = warp / nseg;
    const bool worker = slot < plan.nslots;
    const int nsb_here = (seg == nseg - 1) ? plan.slast : 8;
    const bool has = worker && (lane >> 2) < nsb_here;
    const int g = lane & 3;                                  // sub-blocks 2g, 2g+1 of the super-block
    const int hdr_off = (seg * 8 + (lane >> 2)) * kSuper<kQ5>;
    const int p = seg * 32 + lane;                           // Q8_0 blocks 2p, 2p+1

    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * O / gridDim.x;
    const int64_t r1 = static_cast<int64_t>(blockIdx.x + 1) * O / gridDim.x;
    const int nrows = static_cast<int>(r1 - r0);

    if (threadIdx.x == 0) {
        mbar_init(&xbar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    pdl_trigger();

    Entry pipe[kDepth] = {};
    auto load_at = [&](const uint8_t* sb, Entry& e) {
        if (has) {
            e.h = ldg_stream16(sb);
            if (kQ5) {
                e.q0 = ldg_stream16(sb + 16);
                e.q1 = ldg_stream16(sb + 32);
            }
            constexpr int kCodes = kQ5 ? 48 : 16;
            e.c0 = ldg_stream16(sb + kCodes + 32 * g);
            e.c1 = ldg_stream16(sb + kCodes + 16 + 32 * g);
        }
    };
    // the super-block of this lane in row `row` (of whichever grouped matrix
    // holds it)
    auto row_ptr = [&](int64_t row) {
        int m = 0;
#pragma unroll
        for (int i = 1; i < kMaxGroup; ++i)
            if (i < a.ng && row >= a.start[i]) m = i;
        return a.Wg[m] + (row - a.start[m]) * plan.rowbytes + hdr_off;
    };
    auto load_seg = [&](int64_t row, Entry& e) { load_at(row_ptr(row), e); };
    auto fill = [&](int64_t c0, int crows) {
#pragma unroll
        for (int d = 0; d < kDepth; ++d) {
            const int ri = slot + d * plan.nslots;
            if (ri < crows) load_seg(c0 + ri, pipe[d]);
        }
    };
    if (worker) fill(r0, min(nrows, plan.rch));

    pdl_wait();

    uint32_t xa[8], xb[8];
    float dxa = 0.0f, dxb = 0.0f;
    int sa = 0, sb = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) xa[i] = xb[i] = 0u;
    const uint8_t* xsrc = a.xq;
    if (a.xq_bulk) {
        if (threadIdx.x == 0) {
            const uint32_t bytes = static_cast<uint32_t>(plan.nb * 34);
            mbar_arrive_expect_tx(&xbar, bytes);
            bulk_g2s_plain(xs, a.xq, bytes, &xbar);
        }
        if (!mbar_wait(&xbar, 0)) atomicOr(&g_flags_gemv_q4k, FLAG_TIMEOUT);
        xsrc = xs;
    }
    if (has) {
        load_act(xsrc, 2 * p, xa, dxa, sa);
        load_act(xsrc, 2 * p + 1, xb, dxb, sb);
    }

    // the 6-bit scale and min of sub-blocks 2g and 2g+1 (t = 2(g mod 2) and
    // t + 1 within the scale words): sub-blocks 0..3 take the low six bits of
    // scale bytes t and 4+t; 4..7 the nibbles of byte 8+t topped by the high
    // two bits of bytes t and 4+t.  Both sub-blocks at once on byte pairs:
    // P1 = bytes (t, t+1) of word 1 (scale bytes 0..3), P2 of word 2, P3 of
    // word 3, each in the low 16 bits by one byte permute.
    const uint8_t* wnext = nullptr;
    const int64_t wstride = static_cast<int64_t>(plan.nslots) * plan.rowbytes;
    const uint32_t sel = (g & 1) ? 0x3232u : 0x1010u;       // bytes (2, 3) or (0, 1), twice
    const bool high = g >= 2;
    auto consume = [&](int64_t c0, int crows, int ri, Entry& entry) -> float {
        const Entry& e = entry;
        const uint32_t cw[8] = {e.c0.x, e.c0.y, e.c0.z, e.c0.w, e.c1.x, e.c1.y, e.c1.z, e.c1.w};
        const uint32_t qh[8] = {e.q0.x, e.q0.y, e.q0.z, e.q0.w, e.q1.x, e.q1.y, e.q1.z, e.q1.w};
        int ia = 0, ib = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t ca = cw[i] & kNibbles, cb = (cw[i] >> 4) & kNibbles;
            if (kQ5) {
                // top bits of sub-blocks 2g (bit 2g of each qh byte) and 2g+1
                const uint32_t t = qh[i] >> (2 * g);
                ca |= (t & 0x01010101u) << 4;
                cb |= (t & 0x02020202u) << 3;
            }
            ia = __dp4a(static_cast<int>(ca), static_cast<int>(xa[i]), ia);
            ib = __dp4a(static_cast<int>(cb), static_cast<int>(xb[i]), ib);
        }
        const uint32_t P1 = __byte_perm(e.h.y, 0, sel) & 0xFFFFu;
        const uint32_t P2 = __byte_perm(e.h.z, 0, sel) & 0xFFFFu;
        const uint32_t P3 = __byte_perm(e.h.w, 0, sel) & 0xFFFFu;
        const uint32_t SC = high ? ((P3 & 0x0F0Fu) | ((P1 >> 2) & 0x3030u)) : (P1 & 0x3F3Fu);
        const uint32_t MN = high ? (((P3 >> 4) & 0x0F0Fu) | ((P2 >> 2) & 0x3030u)) : (P2 & 0x3F3Fu);
        // integer products first (sc isum < 2^23, m xsum < 2^18: exact), then
        // one rounding each against the fp16 d and dmin
        const float d = half_bits_to_float(e.h.x), dmin = half_bits_to_float(e.h.x >> 16);
        const float ta = __fmaf_rn(d, static_cast<float>(static_cast<int>(SC & 0xFFu) * ia),
                                   -__fmul_rn(dmin, static_cast<float>(static_cast<int>(MN & 0xFFu) * sa)));
        const float tb = __fmaf_rn(d, static_cast<float>(static_cast<int>(SC >> 8) * ib),
                                   -__fmul_rn(dmin, static_cast<float>(static_cast<int>(MN >> 8) * sb)));
        float acc = __fmul_rn(dxa, ta);
        acc = __fmaf_rn(dxb, tb, acc);   // lanes without a super-block hold zero activations and codes
        if (kDebug && has) {
            int32_t* dst = a.dbg + (c0 + ri) * plan.nb + 2 * p;
            dst[0] = ia;
            dst[1] = ib;
        }
        const int ahead = ri + kDepth * plan.nslots;
        if (ahead < crows) {
            // one matrix: the refills of a slot are consecutive rows of it, a
            // running pointer; grouped matrices: look the row up
            if (a.ng == 1) {
                load_at(wnext, entry);
                wnext += wstride;
            } else {
                load_seg(c0 + ahead, entry);
            }
        }
        return acc;
    };
    // four row-segments (rows ri + k step) in one butterfly: after the xor-16
    // and xor-8 exchanges each group of eight lanes carries one row, summed in
    // the order of a plain warp reduction; row k ends in lane 8k
    auto reduce4 = [&](int ri, int step, int crows, float v0, float v1, float v2, float v3) {
        const bool up16 = (lane & 16) != 0, up8 = (lane & 8) != 0;
        float k0 = up16 ? v2 : v0, k1 = up16 ? v3 : v1;
        k0 = __fadd_rn(k0, __shfl_xor_sync(0xffffffffu, up16 ? v0 : v2, 16));
        k1 = __fadd_rn(k1, __shfl_xor_sync(0xffffffffu, up16 ? v1 : v3, 16));
        float m = up8 ? k1 : k0;
        m = __fadd_rn(m, __shfl_xor_sync(0xffffffffu, up8 ? k0 : k1, 8));
#pragma unroll
        for (int h = 4; h >= 1; h >>= 1) m = __fadd_rn(m, __shfl_xor_sync(0xffffffffu, m, h));
        const int k = lane >> 3;
        if ((lane & 7) == 0 && ri + k * step < crows) part[(ri + k * step) * nseg + seg] = m;
    };

    for (int64_t c0 = r0; c0 < r1; c0 += plan.rch) {
        const int crows = static_cast<int>((r1 - c0) < plan.rch ? (r1 - c0) : plan.rch);
        if (worker) {
            if (c0 != r0) fill(c0, crows);
            if (a.ng == 1) wnext = row_ptr(c0 + slot + static_cast<int64_t>(kDepth) * plan.nslots);
            const int step = plan.nslots;
            for (int ri = slot; ri < crows; ri += kDepth * step) {
                const float q0 = consume(c0, crows, ri, pipe[0]);
                const float q1 = ri + step < crows ? consume(c0, crows, ri + step, pipe[1]) : 0.0f;
                const float q2 = ri + 2 * step < crows ? consume(c0, crows, ri + 2 * step, pipe[2]) : 0.0f;
                const float q3 = ri + 3 * step < crows ? consume(c0, crows, ri + 3 * step, pipe[3]) : 0.0f;
                reduce4(ri, step, crows, q0, q1, q2, q3);
            }
        }
        __syncthreads();
        if (!kDebug) {
            for (int t = threadIdx.x; t < crows; t += kThreads) {
                float v = part[t * nseg];
                for (int s = 1; s < nseg; ++s) v = __fadd_rn(v, part[t * nseg + s]);
                const int64_t row = c0 + t;
                int m = 0;
#pragma unroll
                for (int i = 1; i < kMaxGroup; ++i)
                    if (i < a.ng && row >= a.start[i]) m = i;
                a.yg[m][row - a.start[m]] = v;
            }
        }
        __syncthreads();
    }
}

template <bool kQ5>
int kquant_launch_group(const void* const* W, float* const* y, const int64_t* O, int count, const void* xq,
                        int64_t K, cudaStream_t stream, int32_t* dbg) {
    if (!W || !O || !xq || (!y && !dbg)) return QDG_EINVAL;
    if (count < 1 || count > kMaxGroup || K <= 0) return QDG_EINVAL;
    if (dbg && count != 1) return QDG_EINVAL;
    if (K % 256 != 0 || K > 32768) return QDG_ESHAPE;
    if (!aligned(xq, 2) || !aligned(dbg, 4)) return QDG_EALIGN;
    Args a{};
    int64_t total = 0;
    for (int m = 0; m < count; ++m) {
        if (!W[m] || (!dbg && !y[m]) || O[m] <= 0) return QDG_EINVAL;
        if (!aligned(W[m], 16) || (y && !aligned(y[m], 4))) return QDG_EALIGN;
        a.Wg[m] = static_cast<const uint8_t*>(W[m]);
        a.yg[m] = y ? y[m] : nullptr;
        a.start[m] = total;
        total += O[m];
    }
    if (total >= (int64_t(1) << 31)) return QDG_ESHAPE;
    const DeviceInfo dev = device_info();
    if (dev.device < 0) return QDG_ECUDA;
    const Plan plan = make_plan(K, kSuper<kQ5>);
    if (plan.nslots < 1 || plan.rch < 1) return QDG_ESHAPE;   // cannot happen for K <= 32768: 16 segments at most
    const int grid = static_cast<int>(std::min<int64_t>(dev.sms, total));
    a.ng = count;
    a.xq = static_cast<const uint8_t*>(xq);
    a.xq_bulk = aligned(xq, 16) ? 1 : 0;
    const size_t smem = a.xq_bulk ? static_cast<size_t>(plan.nb) * 34 : 0;   // a multiple of 16 (K % 256 == 0)
    a.dbg = dbg;
    a.O = total;
    cudaError_t e;
    if (dbg)
        e = launch(gemv_q4k_kernel<kQ5, true>, dim3(grid), dim3(kThreads), smem, stream, false, a, plan);
    else
        e = launch(gemv_q4k_kernel<kQ5, false>, dim3(grid), dim3(kThreads), smem, stream, true, a, plan);
    if (e != cudaSuccess) return QDG_ECUDA;
    count_launch(kQ5 ? 14 : 12);
    return QDG_OK;
}

}  // namespace

int gemv_q4k_launch(const void* W, const void* xq, float* y, int64_t O, int64_t K, cudaStream_t stream,
                    int32_t* dbg) {
    float* ys[1] = {y};
    return kquant_launch_group<false>(&W, y ? ys : nullptr, &O, 1, xq, K, stream, dbg);
}

int gemv_q5k_launch(const void* W, const void* xq, float* y, int64_t O, int64_t K, cudaStream_t stream,
                    int32_t* dbg) {
    float* ys[1] = {y};
    return kquant_launch_group<true>(&W, y ? ys : nullptr, &O, 1, xq, K, stream, dbg);
}

unsigned flags_read_clear_gemv_q4k(cudaStream_t stream) {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_flags_gemv_q4k, sizeof(v), 0, cudaMemcpyDeviceToHost, stream) !=
        cudaSuccess)
        return ~0u;
    if (cudaMemcpyToSymbolAsync(g_flags_gemv_q4k, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream) !=
        cudaSuccess)
        return ~0u;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return ~0u;
    return v;
}

}  // namespace qdg

using namespace qdg;

extern "C" int q4_k_q8_0_gemv(const void* W, const void* xq, float* y, int64_t O, int64_t K, qdg_stream_t stream) {
    if (!y) return QDG_EINVAL;
    return gemv_q4k_launch(W, xq, y, O, K, reinterpret_cast<cudaStream_t>(stream), nullptr);
}

extern "C" int q4_k_q8_0_gemv_group(const void* const* W, float* const* y, const int64_t* O, int count,
                                    const void* xq, int64_t K, qdg_stream_t stream) {
    if (!y) return QDG_EINVAL;
    return kquant_launch_group<false>(W, y, O, count, xq, K, reinterpret_cast<cudaStream_t>(stream), nullptr);
}

extern "C" int q5_k_q8_0_gemv(const void* W, const void* xq, float* y, int64_t O, int64_t K, qdg_stream_t stream) {
    if (!y) return QDG_EINVAL;
    return gemv_q5k_launch(W, xq, y, O, K, reinterpret_cast<cudaStream_t>(stream), nullptr);
}

extern "C" int q5_k_q8_0_gemv_group(const void* const* W, float* const* y, const int64_t* O, int count,
                                    const void* xq, int64_t K, qdg_stream_t stream) {
    if (!y) return QDG_EINVAL;
    return kquant_launch_group<true>(W, y, O, count, xq, K, reinterpret_cast<cudaStream_t>(stream), nullptr);
}
