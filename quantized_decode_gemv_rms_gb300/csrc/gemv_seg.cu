// gemv_seg.cu -- batch-1 Q4_0 x Q8_0 matrix-vector product on weights held in
// the segment layout, and the load-time repack that produces that layout.
//
// The CPU back end of GGML rearranges Q4 weights once, when they are loaded,
// into a layout its dot-product kernels read faster [GGML: Backend
// abstraction and hardware acceleration, section "How build switches become
// runtime capabilities", build-option table, GGML_CPU_REPACK].  This file is
// the GPU counterpart.  The plain Q4_0 block is 18 bytes, so its nibbles are
// only 2-byte aligned and a coalesced reader has to pass them through shared
// memory; the segment layout separates nibbles from scales so that every
// lane reads its own blocks straight into registers:
//   a row of nb = K/32 blocks is cut into segments of 64 blocks; segment s
//   starts at byte 1152*s and holds the 16 nibble bytes of each of its r
//   blocks (block 64s+i at 16*i, bytes as in the Q4_0 block), then 32 words,
//   word l = fp16 scale of block 64s+l (low half) and of block 64s+32+l (high
//   half), 0 where that block does not exist.  Row bytes = 1152*(nseg-1) +
//   16*r_last + 128, equal to 18*nb when 64 divides nb.
//
// GEMV design (same row/segment work split as the plain-layout kernel):
//   * Each CTA (16 warps, one per SM) owns a contiguous range of rows; warp w
//     works on segment w % nseg of rows slot, slot + nslots, ...
//   * Lane l of a warp owns blocks 64s+l and 64s+32+l of its segment: two
//     coalesced 16-byte nibble loads (512 contiguous bytes per warp each) and
//     one 4-byte scale-word load per row-segment, issued four row-segments
//     ahead of use (74 KB in flight per SM, 96 registers, so that a CTA of
//     the quantize kernel fits beside it); launches with at least 384 rows
//     per CTA (a vocabulary head) go eight row-segments ahead at 128
//     registers; the matching Q8_0 activations stay in registers.
//   * Exact block sums with dp4a (minus 8 * sum(q_x)), scaled by d_w * d_x;
//     each four rows of the ring share one warp butterfly; segment partials
//     combined per row in a fixed order (deterministic, and the same bits for
//     either ring depth).
//   * Programmatic dependent launch: the first row-segments of W are
//     requested before the kernel waits for the preceding grid.
#include "common.cuh"

#include <algorithm>

namespace qdg {

static __device__ unsigned g_flags_gemv_seg;

namespace {

constexpr int kWarps = 16;
constexpr int kThreads = 32 * kWarps;
constexpr int kDepth1 = 4;                  // row-segments in flight per warp, reduced together in one butterfly
constexpr int kDepthDeep = 8;               // the same for long launches (128 registers: no quantize CTA fits beside)
constexpr int kDeepRows = 384;              // rows per CTA from which a launch takes the deep ring
constexpr int kSegStride = 1152;            // bytes from one segment to the next: 64 x 16 nibble bytes + 128
constexpr int kPartFloats = 3072;           // per-chunk partial sums (rows x segments)
constexpr int kL2Prefetch = 96 * 1024;      // bytes of W prefetched into L2 per CTA at start
constexpr int kMaxGroup = 4;
constexpr int kFusedMaxK = 16384;           // fused form: x and gamma staged whole in shared memory (128 KB)
constexpr uint32_t kNibbles = 0x0F0F0F0Fu;

struct Plan {
    int rowbytes;   // bytes of one row in the segment layout
    int nb;         // K/32
    int nseg;       // segments per row, ceil(nb / 64)
    int rlast;      // blocks in the last segment (8..64)
    int nslots;     // rows in flight per CTA = kWarps / nseg
    int rch;        // rows per chunk (partial-sum buffer capacity), multiple of nslots
};

int64_t seg_row_bytes(int64_t K) {
    const int64_t nb = K / 32;
    const int64_t nseg = (nb + 63) / 64;
    return kSegStride * (nseg - 1) + 16 * (nb - 64 * (nseg - 1)) + 128;
}

Plan make_plan(int64_t K) {
    Plan p{};
    p.nb = static_cast<int>(K / 32);
    p.nseg = (p.nb + 63) / 64;
    p.rlast = p.nb - 64 * (p.nseg - 1);
    p.rowbytes = static_cast<int>(seg_row_bytes(K));
    p.nslots = kWarps / p.nseg;
    p.rch = p.nslots > 0 ? (kPartFloats / p.nseg) / p.nslots * p.nslots : 0;
    return p;
}

// Every segment of a row needs a warp: K <= 32768 gives at most kWarps
// segments, so a plan always has a row slot and a positive chunk.
static_assert(kWarps * 64 * 32 >= 32768, "one warp per segment at the largest K");
bool plan_ok(const Plan& p) { return p.nslots >= 1 && p.rch >= 1; }

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

// Sum over one block of (code) * q_x, codes unsigned 0..15: low nibbles of
// word i are elements 4i..4i+3, high nibbles elements 16+4i..16+4i+3.
__device__ __forceinline__ int block_dot(const uint4& q, const uint32_t* x) {
    int acc = 0;
    acc = __dp4a(static_cast<int>(q.x & kNibbles), static_cast<int>(x[0]), acc);
    acc = __dp4a(static_cast<int>((q.x >> 4) & kNibbles), static_cast<int>(x[4]), acc);
    acc = __dp4a(static_cast<int>(q.y & kNibbles), static_cast<int>(x[1]), acc);
    acc = __dp4a(static_cast<int>((q.y >> 4) & kNibbles), static_cast<int>(x[5]), acc);
    acc = __dp4a(static_cast<int>(q.z & kNibbles), static_cast<int>(x[2]), acc);
    acc = __dp4a(static_cast<int>((q.z >> 4) & kNibbles), static_cast<int>(x[6]), acc);
    acc = __dp4a(static_cast<int>(q.w & kNibbles), static_cast<int>(x[3]), acc);
    acc = __dp4a(static_cast<int>((q.w >> 4) & kNibbles), static_cast<int>(x[7]), acc);
    return acc;
}

// One lane's share of one row-segment.
struct Entry {
    uint4 a, b;     // nibbles of blocks 64s+l and 64s+32+l
    uint32_t sc;    // their scales (low, high half)
};

struct Args {
    const uint8_t* Wg[kMaxGroup];   // stacked matrices sharing one input
    float* yg[kMaxGroup];
    int64_t start[kMaxGroup];
    int ng;
    const uint8_t* xq;
    int xq_bulk;            // xq is 16-byte aligned: one bulk copy brings it into shared memory
    int32_t* dbg;
    int64_t O;
    // fused form: fp32 activations, gamma (NULL = no norm), epsilon, optional
    // copy of the Q8_0 vector (written by CTA 0)
    const float* x;
    const float* gamma;
    float eps;
    uint8_t* xq_out;
};

// Q8_0 block b of the activations: scale and the 32 codes as 8 words, from
// 2-byte loads (a 34-byte block is only 2-byte aligned), out of shared memory
// (kShared) or global memory.
template <bool kShared>
__device__ __forceinline__ void load_act(const uint8_t* xq, int b, uint32_t* x, float& d, int& sum) {
    const unsigned short* h = reinterpret_cast<const unsigned short*>(xq + static_cast<size_t>(b) * 34);
    auto ld = [&](int i) -> uint32_t { return kShared ? h[i] : __ldg(h + i); };
    d = half_bits_to_float(ld(0));
    sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        x[i] = ld(1 + 2 * i) | (ld(2 + 2 * i) << 16);
        sum = __dp4a(static_cast<int>(x[i]), 0x01010101, sum);
    }
}

// 96 registers a thread: one CTA of 512 threads leaves room on its SM for a
// CTA of the quantize kernel that prepares the next input.
//
// Fused form (kFused): the RMS_NORM, the MUL by gamma and the Q8_0
// quantization of the input run in every CTA before its product, with the
// arithmetic and the summation order of the standalone quantize kernel, so
// that the Q8_0 vector is the same bit for bit:
//   x and gamma arrive in shared memory by two bulk copies (one round trip);
//   chain j (threads 0..255) sums x_i^2 over i = j (mod 256) ascending with
//   fma; xor butterflies (16, 8, 4, 2, 1) in each warp; warp totals
//   ((w0+w1)+(w2+w3))+((w4+w5)+(w6+w7)); s = 1/sqrt(sum/K + eps);
//   block b (warp b mod 16, lane = element): v = (x*s)*gamma, d = max|v|/127,
//   q = round(v/d) (halves away from zero), clamped to +-127.
template <bool kFused, bool kDebug, bool kDeep = false>
__global__ void __maxnreg__(kDeep ? 128 : 96) gemv_seg_kernel(const __grid_constant__ Args a,
                                                              const __grid_constant__ Plan plan) {
    constexpr int kDepth = kDeep ? kDepthDeep : kDepth1;
    __shared__ float part[kPartFloats];
    __shared__ float norm_part[8];
    __shared__ uint64_t xbar;                       // the bulk copies of xq (or of x and gamma)
    // xq (K/32 x 34 bytes) when a.xq_bulk or kFused; fused form: then x, gamma (K fp32 each)
    extern __shared__ __align__(16) uint8_t xs[];
    const int64_t O = a.O;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nseg = plan.nseg;
    const int seg = warp % nseg;
    const int slot = warp / nseg;
    const bool worker = slot < plan.nslots;
    const int r = (seg == nseg - 1) ? plan.rlast : 64;     // blocks in this warp's segment
    const bool has_a = worker && lane < r;
    const bool has_b = worker && lane + 32 < r;
    const int nib_off = seg * kSegStride + 16 * lane;      // block 64s+l; block 64s+32+l is 512 bytes on
    const int sc_off = seg * kSegStride + 16 * r + 4 * lane;

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
    auto load_seg = [&](int64_t row, Entry& e) {
        int g = 0;
#pragma unroll
        for (int i = 1; i < kMaxGroup; ++i)
            if (i < a.ng && row >= a.start[i]) g = i;
        const uint8_t* base = a.Wg[g] + (row - a.start[g]) * plan.rowbytes;
        if (has_a) e.a = ldg_stream16(base + nib_off);
        if (has_b) e.b = ldg_stream16(base + nib_off + 512);
        e.sc = ldg_stream4(base + sc_off);
    };
    auto fill = [&](int64_t c0, int crows) {
#pragma unroll
        for (int d = 0; d < kDepth; ++d) {
            const int ri = slot + d * plan.nslots;
            if (ri < crows) load_seg(c0 + ri, pipe[d]);
        }
    };

    if (worker) fill(r0, min(nrows, plan.rch));
    if (threadIdx.x == 0) {
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

    uint32_t xa[8], xb[8];
    float dxa = 0.0f, dxb = 0.0f;
    int sa = 0, sb = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) xa[i] = xb[i] = 0u;
    if (kFused) {
        const int nb = plan.nb;
        const int K = nb * 32;
        float* xf = reinterpret_cast<float*>(xs + nb * 34);   // nb * 34 is a multiple of 16
        float* gf = xf + K;
        if (threadIdx.x == 0) {
            const uint32_t bytes = static_cast<uint32_t>(K) * 4;
            mbar_arrive_expect_tx(&xbar, a.gamma != nullptr ? 2 * bytes : bytes);
            bulk_g2s_plain(xf, a.x, bytes, &xbar);
            if (a.gamma != nullptr) bulk_g2s_plain(gf, a.gamma, bytes, &xbar);
        }
        if (!mbar_wait(&xbar, 0)) atomicOr(&g_flags_gemv_seg, FLAG_TIMEOUT);
        float s = 1.0f;
        if (a.gamma != nullptr) {
            if (threadIdx.x < 256) {
                float acc = 0.0f;
                for (int i = threadIdx.x; i < K; i += 256) acc = __fmaf_rn(xf[i], xf[i], acc);
                acc = warp_sum(acc);
                if (lane == 0) norm_part[warp] = acc;
            }
            __syncthreads();
            const float ss = __fadd_rn(__fadd_rn(__fadd_rn(norm_part[0], norm_part[1]), __fadd_rn(norm_part[2], norm_part[3])),
                                       __fadd_rn(__fadd_rn(norm_part[4], norm_part[5]), __fadd_rn(norm_part[6], norm_part[7])));
            const float mean = __fdiv_rn(ss, static_cast<float>(K));
            s = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, a.eps)));
        }
        for (int b0 = warp; b0 < nb; b0 += 4 * kWarps) {
            float v[4], d[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int b = b0 + u * kWarps;
                v[u] = 0.0f;
                if (b < nb) {
                    v[u] = xf[(b << 5) + lane];
                    if (a.gamma != nullptr) v[u] = __fmul_rn(__fmul_rn(v[u], s), gf[(b << 5) + lane]);
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
                    float rr = roundf(__fdiv_rn(v[u], dd[u]));
                    rr = fminf(fmaxf(rr, -127.0f), 127.0f);
                    q[u] = static_cast<int>(rr);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int b = b0 + u * kWarps;
                if (b < nb) {
                    uint8_t* blk = xs + b * 34;
                    if (lane == 0) {
                        const __half dh = __float2half_rn(dd[u]);
                        *reinterpret_cast<unsigned short*>(blk) = __half_as_ushort(dh);
                        if (__hisinf(dh)) atomicOr(&g_flags_gemv_seg, FLAG_OVERFLOW);
                    }
                    blk[2 + lane] = static_cast<uint8_t>(static_cast<int8_t>(q[u]));
                }
            }
        }
        __syncthreads();
        if (a.xq_out != nullptr && blockIdx.x == 0) {
            const uint32_t* src = reinterpret_cast<const uint32_t*>(xs);
            uint32_t* dst = reinterpret_cast<uint32_t*>(a.xq_out);
            for (int i = threadIdx.x; i < nb * 34 / 4; i += kThreads) dst[i] = src[i];
        }
        if (has_a) load_act<true>(xs, seg * 64 + lane, xa, dxa, sa);
        if (has_b) load_act<true>(xs, seg * 64 + 32 + lane, xb, dxb, sb);
    } else if (a.xq_bulk) {
        // one bulk copy of the whole vector (one round trip), then the
        // lanes' blocks out of shared memory (measured on GB300: 16-byte
        // cp.async copies from every thread queue behind the weight loads
        // already in flight and arrived 0.5-1 us later)
        if (threadIdx.x == 0) {
            const uint32_t bytes = static_cast<uint32_t>(plan.nb * 34);
            mbar_arrive_expect_tx(&xbar, bytes);
            bulk_g2s_plain(xs, a.xq, bytes, &xbar);
        }
        if (!mbar_wait(&xbar, 0)) atomicOr(&g_flags_gemv_seg, FLAG_TIMEOUT);
        if (has_a) load_act<true>(xs, seg * 64 + lane, xa, dxa, sa);
        if (has_b) load_act<true>(xs, seg * 64 + 32 + lane, xb, dxb, sb);
    } else {
        if (has_a) load_act<false>(a.xq, seg * 64 + lane, xa, dxa, sa);
        if (has_b) load_act<false>(a.xq, seg * 64 + 32 + lane, xb, dxb, sb);
    }

    // One row-segment: dot the entry, then refill it with the segment kDepth
    // ahead (the refill goes into the registers just read, so no copy of the
    // entry is kept alive across the loads); returns the lane's partial.
    // Measured on GB300 this order streams about 20% faster than refilling
    // before the dot; sharing one butterfly between the ring's rows (reduce4)
    // took the 8B decode step from 88.3 to 84.6 us.
    auto consume = [&](int64_t c0, int crows, int ri, Entry& entry) -> float {
        const Entry& cur = entry;
        // lanes without a block hold zero activations and zero scales
        const int ia = block_dot(cur.a, xa) - 8 * sa;
        const int ib = block_dot(cur.b, xb) - 8 * sb;
        const float dwa = half_bits_to_float(cur.sc);
        const float dwb = half_bits_to_float(cur.sc >> 16);
        float acc = __fmul_rn(__fmul_rn(dwa, dxa), static_cast<float>(ia));
        acc = __fmaf_rn(__fmul_rn(dwb, dxb), static_cast<float>(ib), acc);
        if (kDebug) {
            int32_t* d = a.dbg + (c0 + ri) * plan.nb + seg * 64 + lane;
            if (has_a) d[0] = ia;
            if (has_b) d[32] = ib;
        }
        const int ahead = ri + kDepth * plan.nslots;
        if (ahead < crows) load_seg(c0 + ahead, entry);
        return acc;
    };
    // four row-segments (rows ri + k * step) reduced in one butterfly: the
    // xor-16 exchange leaves rows 0, 1 in lanes 0..15 and rows 2, 3 in lanes
    // 16..31, the xor-8 exchange one row per eight lanes; every row is summed
    // in the order of a plain warp reduction and ends in lane 8 * k
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
            const int step = plan.nslots;
            for (int ri = slot; ri < crows; ri += kDepth * step) {
                // four ring entries (rows ri + k step) per butterfly; the deep
                // ring turns through two such groups
#pragma unroll
                for (int h = 0; h < kDepth / 4; ++h) {
                    const int rj = ri + 4 * h * step;
                    if (h > 0 && rj >= crows) break;
                    const float p0 = consume(c0, crows, rj, pipe[4 * h]);
                    const float p1 = rj + step < crows ? consume(c0, crows, rj + step, pipe[4 * h + 1]) : 0.0f;
                    const float p2 = rj + 2 * step < crows ? consume(c0, crows, rj + 2 * step, pipe[4 * h + 2]) : 0.0f;
                    const float p3 = rj + 3 * step < crows ? consume(c0, crows, rj + 3 * step, pipe[4 * h + 3]) : 0.0f;
                    reduce4(rj, step, crows, p0, p1, p2, p3);
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

// Repack: one warp per (row, segment).  Lane l moves the nibbles of blocks
// 64s+l and 64s+32+l (eight 2-byte loads each, one 16-byte store) and writes
// scale word l.
__global__ void __launch_bounds__(256) repack_seg_kernel(const uint8_t* __restrict__ W, uint8_t* __restrict__ out,
                                                         int64_t O, int nb, int nseg, int64_t rowbytes) {
    const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (gw >= O * nseg) return;
    const int64_t o = gw / nseg;
    const int s = static_cast<int>(gw - o * nseg);
    const int first = 64 * s;
    const int r = min(64, nb - first);
    const uint8_t* row = W + o * static_cast<int64_t>(nb) * 18;
    uint8_t* seg = out + o * rowbytes + static_cast<int64_t>(kSegStride) * s;
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h;
        if (i >= r) continue;
        const unsigned short* blk = reinterpret_cast<const unsigned short*>(row + static_cast<int64_t>(first + i) * 18);
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = static_cast<uint32_t>(blk[1 + 2 * k]) | (static_cast<uint32_t>(blk[2 + 2 * k]) << 16);
        *reinterpret_cast<uint4*>(seg + 16 * i) = make_uint4(w[0], w[1], w[2], w[3]);
        if (h == 0)
            lo = blk[0];
        else
            hi = blk[0];
    }
    *reinterpret_cast<uint32_t*>(seg + 16 * r + 4 * lane) = lo | (hi << 16);
}

// Two activation vectors that share one pass over the weights (the smallest
// case of the small-N product): the same row/segment split and register ring
// as the one-vector kernel, the nibbles of each block unpacked once and dotted
// with both vectors by dp4a.  y[n][row] at y + n * ldy.  One matrix per
// launch.  A separate kernel, so that the one-vector kernel's code is not
// touched by the second vector's registers.
struct Args2 {
    const uint8_t* W;
    const uint8_t* xq;      // two Q8_0 vectors, K/32 blocks each, back to back
    int xq_bulk;
    float* y;
    int64_t ldy;
    int32_t* dbg;           // [2][O][K/32] exact block sums instead of y
    int64_t O;
};

__device__ __forceinline__ int nib_dot(const uint32_t* lo, const uint32_t* hi, const uint32_t* x) {
    int acc = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc = __dp4a(static_cast<int>(lo[i]), static_cast<int>(x[i]), acc);
        acc = __dp4a(static_cast<int>(hi[i]), static_cast<int>(x[4 + i]), acc);
    }
    return acc;
}

template <bool kDebug>
__global__ void __maxnreg__(128) gemv_seg2_kernel(const __grid_constant__ Args2 a, const __grid_constant__ Plan plan) {
    __shared__ float part[kPartFloats];
    __shared__ uint64_t xbar;
    extern __shared__ __align__(16) uint8_t xs[];   // both Q8_0 vectors when a.xq_bulk
    const int64_t O = a.O;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nseg = plan.nseg;
    const int seg = warp % nseg;
    const int slot = warp / nseg;
    const bool worker = slot < plan.nslots;
    const int r = (seg == nseg - 1) ? plan.rlast : 64;
    const bool has_a = worker && lane < r;
    const bool has_b = worker && lane + 32 < r;
    const int nib_off = seg * kSegStride + 16 * lane;
    const int sc_off = seg * kSegStride + 16 * r + 4 * lane;

    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * O / gridDim.x;
    const int64_t r1 = static_cast<int64_t>(blockIdx.x + 1) * O / gridDim.x;
    const int nrows = static_cast<int>(r1 - r0);

    if (threadIdx.x == 0) {
        mbar_init(&xbar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    pdl_trigger();

    Entry pipe[kDepth1] = {};
    auto load_seg = [&](int64_t row, Entry& e) {
        const uint8_t* base = a.W + row * plan.rowbytes;
        if (has_a) e.a = ldg_stream16(base + nib_off);
        if (has_b) e.b = ldg_stream16(base + nib_off + 512);
        e.sc = ldg_stream4(base + sc_off);
    };
    auto fill = [&](int64_t c0, int crows) {
#pragma unroll
        for (int d = 0; d < kDepth1; ++d) {
            const int ri = slot + d * plan.nslots;
            if (ri < crows) load_seg(c0 + ri, pipe[d]);
        }
    };
    if (worker) fill(r0, min(nrows, plan.rch));

    pdl_wait();

    uint32_t xa[2][8], xb[2][8];
    float dxa[2] = {0.0f, 0.0f}, dxb[2] = {0.0f, 0.0f};
    int sa[2] = {0, 0}, sb[2] = {0, 0};
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int i = 0; i < 8; ++i) xa[n][i] = xb[n][i] = 0u;
    const int vec = plan.nb * 34;   // bytes of one Q8_0 vector
    if (a.xq_bulk) {
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(&xbar, static_cast<uint32_t>(2 * vec));
            bulk_g2s_plain(xs, a.xq, static_cast<uint32_t>(2 * vec), &xbar);
        }
        if (!mbar_wait(&xbar, 0)) atomicOr(&g_flags_gemv_seg, FLAG_TIMEOUT);
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            if (has_a) load_act<true>(xs + n * vec, seg * 64 + lane, xa[n], dxa[n], sa[n]);
            if (has_b) load_act<true>(xs + n * vec, seg * 64 + 32 + lane, xb[n], dxb[n], sb[n]);
        }
    } else {
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            if (has_a) load_act<false>(a.xq + n * vec, seg * 64 + lane, xa[n], dxa[n], sa[n]);
            if (has_b) load_act<false>(a.xq + n * vec, seg * 64 + 32 + lane, xb[n], dxb[n], sb[n]);
        }
    }

    // dot the entry with both vectors, refill it; returns the lane's two partials
    auto consume = [&](int64_t c0, int crows, int ri, Entry& entry, float& r0v, float& r1v) {
        const Entry& cur = entry;
        const uint32_t la[4] = {cur.a.x & kNibbles, cur.a.y & kNibbles, cur.a.z & kNibbles, cur.a.w & kNibbles};
        const uint32_t ha[4] = {(cur.a.x >> 4) & kNibbles, (cur.a.y >> 4) & kNibbles, (cur.a.z >> 4) & kNibbles,
                                (cur.a.w >> 4) & kNibbles};
        const uint32_t lb[4] = {cur.b.x & kNibbles, cur.b.y & kNibbles, cur.b.z & kNibbles, cur.b.w & kNibbles};
        const uint32_t hb[4] = {(cur.b.x >> 4) & kNibbles, (cur.b.y >> 4) & kNibbles, (cur.b.z >> 4) & kNibbles,
                                (cur.b.w >> 4) & kNibbles};
        const float dwa = half_bits_to_float(cur.sc);
        const float dwb = half_bits_to_float(cur.sc >> 16);
        float acc[2];
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            const int ia = nib_dot(la, ha, xa[n]) - 8 * sa[n];
            const int ib = nib_dot(lb, hb, xb[n]) - 8 * sb[n];
            acc[n] = __fmul_rn(__fmul_rn(dwa, dxa[n]), static_cast<float>(ia));
            acc[n] = __fmaf_rn(__fmul_rn(dwb, dxb[n]), static_cast<float>(ib), acc[n]);
            if (kDebug) {
                int32_t* d = a.dbg + (n * O + c0 + ri) * plan.nb + seg * 64 + lane;
                if (has_a) d[0] = ia;
                if (has_b) d[32] = ib;
            }
        }
        const int ahead = ri + kDepth1 * plan.nslots;
        if (ahead < crows) load_seg(c0 + ahead, entry);
        r0v = acc[0];
        r1v = acc[1];
    };

    // eight partials (four rows x two vectors, v[2 r + n]) in one butterfly:
    // the xor-16, xor-8 and xor-4 exchanges leave value 4 b16 + 2 b8 + b4 in
    // the lanes whose bits 4, 3, 2 are b16, b8, b4, each summed in the order of
    // a plain warp reduction; the totals end in lanes 4 g
    auto reduce8 = [&](int ri, int step, int crows, const float (&v)[8]) {
        const bool u16 = (lane & 16) != 0, u8 = (lane & 8) != 0, u4 = (lane & 4) != 0;
        float w4[4], w2[2];
#pragma unroll
        for (int q = 0; q < 4; ++q)
            w4[q] = __fadd_rn(u16 ? v[4 + q] : v[q], __shfl_xor_sync(0xffffffffu, u16 ? v[q] : v[4 + q], 16));
#pragma unroll
        for (int q = 0; q < 2; ++q)
            w2[q] = __fadd_rn(u8 ? w4[2 + q] : w4[q], __shfl_xor_sync(0xffffffffu, u8 ? w4[q] : w4[2 + q], 8));
        float c = __fadd_rn(u4 ? w2[1] : w2[0], __shfl_xor_sync(0xffffffffu, u4 ? w2[0] : w2[1], 4));
        c = __fadd_rn(c, __shfl_xor_sync(0xffffffffu, c, 2));
        c = __fadd_rn(c, __shfl_xor_sync(0xffffffffu, c, 1));
        const int g = lane >> 2;
        const int row = ri + (g >> 1) * step;
        if ((lane & 3) == 0 && row < crows) part[(row * nseg + seg) * 2 + (g & 1)] = c;
    };

    for (int64_t c0 = r0; c0 < r1; c0 += plan.rch) {
        const int crows = static_cast<int>((r1 - c0) < plan.rch ? (r1 - c0) : plan.rch);
        if (worker) {
            if (c0 != r0) fill(c0, crows);
            const int step = plan.nslots;
            for (int ri = slot; ri < crows; ri += kDepth1 * step) {
                float v[8] = {};
                consume(c0, crows, ri, pipe[0], v[0], v[1]);
                if (ri + step < crows) consume(c0, crows, ri + step, pipe[1], v[2], v[3]);
                if (ri + 2 * step < crows) consume(c0, crows, ri + 2 * step, pipe[2], v[4], v[5]);
                if (ri + 3 * step < crows) consume(c0, crows, ri + 3 * step, pipe[3], v[6], v[7]);
                reduce8(ri, step, crows, v);
            }
        }
        __syncthreads();
        if (!kDebug) {
            for (int t = threadIdx.x; t < 2 * crows; t += kThreads) {
                const int row = t >> 1, n = t & 1;
                float v = part[row * nseg * 2 + n];
                for (int g = 1; g < nseg; ++g) v = __fadd_rn(v, part[(row * nseg + g) * 2 + n]);
                a.y[n * a.ldy + c0 + row] = v;
            }
        }
        __syncthreads();
    }
}

}  // namespace

int gemv_seg_launch_group(const void* const* W, float* const* y, const int64_t* O, int count, const void* xq,
                          int64_t K, cudaStream_t stream, int32_t* dbg) {
    if (!W || !O || !xq || (!y && !dbg)) return QDG_EINVAL;
    if (count < 1 || count > kMaxGroup || K <= 0) return QDG_EINVAL;
    if (dbg && count != 1) return QDG_EINVAL;
    if (K % 256 != 0 || K > 32768) return QDG_ESHAPE;
    if (!aligned(xq, 2) || !aligned(dbg, 4)) return QDG_EALIGN;
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
    const Plan plan = make_plan(K);
    if (!plan_ok(plan)) return QDG_ESHAPE;
    const int grid = static_cast<int>(std::min<int64_t>(dev.sms, total));
    a.ng = count;
    a.xq = static_cast<const uint8_t*>(xq);
    a.xq_bulk = aligned(xq, 16) ? 1 : 0;
    const size_t smem = a.xq_bulk ? static_cast<size_t>(plan.nb) * 34 : 0;   // a multiple of 16 (K % 256 == 0)
    a.dbg = dbg;
    a.O = total;
    cudaError_t e;
    // a long launch (the vocabulary head) takes the eight-deep ring: twice the
    // bytes in flight per warp; the following quantize kernel then waits for
    // SMs to free up, which the CTAs' spread of finishing times provides
    const bool deep = (total + grid - 1) / grid >= kDeepRows;
    if (dbg)
        e = deep ? launch(gemv_seg_kernel<false, true, true>, dim3(grid), dim3(kThreads), smem, stream, false, a, plan)
                 : launch(gemv_seg_kernel<false, true>, dim3(grid), dim3(kThreads), smem, stream, false, a, plan);
    else
        e = deep ? launch(gemv_seg_kernel<false, false, true>, dim3(grid), dim3(kThreads), smem, stream, true, a, plan)
                 : launch(gemv_seg_kernel<false, false>, dim3(grid), dim3(kThreads), smem, stream, true, a, plan);
    if (e != cudaSuccess) return QDG_ECUDA;
    count_launch(6);
    return QDG_OK;
}

int gemv_seg_rmsnorm_launch(const void* const* W, float* const* y, const int64_t* O, int count, const float* x,
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
    const Plan plan = make_plan(K);
    if (!plan_ok(plan)) return QDG_ESHAPE;
    const int grid = static_cast<int>(std::min<int64_t>(dev.sms, total));
    a.ng = count;
    a.x = x;
    a.gamma = gamma;
    a.eps = eps;
    a.xq_out = static_cast<uint8_t*>(xq_out);
    a.O = total;
    const size_t smem = static_cast<size_t>(plan.nb) * 34 + static_cast<size_t>(8) * K;
    if (ensure_smem_limit(reinterpret_cast<const void*>(gemv_seg_kernel<true, false>), smem) != cudaSuccess)
        return QDG_ECUDA;
    const cudaError_t e = launch(gemv_seg_kernel<true, false>, dim3(grid), dim3(kThreads), smem, stream, true, a, plan);
    if (e != cudaSuccess) return QDG_ECUDA;
    count_launch(9);
    return QDG_OK;
}

int gemv_seg2_launch(const void* W, const void* xq, float* y, int64_t ldy, int64_t O, int64_t K,
                     cudaStream_t stream, int32_t* dbg) {
    if (!W || !xq || (!y && !dbg) || O <= 0 || K <= 0 || (y && ldy < O)) return QDG_EINVAL;
    if (K % 256 != 0 || K > 32768) return QDG_ESHAPE;
    if (O >= (int64_t(1) << 31)) return QDG_ESHAPE;
    if (!aligned(W, 16) || !aligned(xq, 2) || !aligned(y, 4) || !aligned(dbg, 4)) return QDG_EALIGN;
    const DeviceInfo dev = device_info();
    if (dev.device < 0) return QDG_ECUDA;
    Plan plan = make_plan(K);
    if (!plan_ok(plan)) return QDG_ESHAPE;
    plan.rch = (kPartFloats / (plan.nseg * 2)) / plan.nslots * plan.nslots;
    Args2 a{};
    a.W = static_cast<const uint8_t*>(W);
    a.xq = static_cast<const uint8_t*>(xq);
    a.xq_bulk = aligned(xq, 16) ? 1 : 0;
    a.y = y;
    a.ldy = ldy;
    a.dbg = dbg;
    a.O = O;
    const int grid = static_cast<int>(std::min<int64_t>(dev.sms, O));
    const size_t smem = a.xq_bulk ? static_cast<size_t>(2) * plan.nb * 34 : 0;
    // both vectors of a large K (up to 2 x 1024 x 34 bytes) exceed the default 48 KB
    if (ensure_smem_limit(reinterpret_cast<const void*>(gemv_seg2_kernel<false>), smem) != cudaSuccess ||
        ensure_smem_limit(reinterpret_cast<const void*>(gemv_seg2_kernel<true>), smem) != cudaSuccess)
        return QDG_ECUDA;
    cudaError_t e;
    if (dbg)
        e = launch(gemv_seg2_kernel<true>, dim3(grid), dim3(kThreads), smem, stream, false, a, plan);
    else
        e = launch(gemv_seg2_kernel<false>, dim3(grid), dim3(kThreads), smem, stream, true, a, plan);
    if (e != cudaSuccess) return QDG_ECUDA;
    count_launch(6);
    return QDG_OK;
}

int gemv_seg_launch(const void* W, const void* xq, float* y, int64_t O, int64_t K, cudaStream_t stream,
                    int32_t* dbg) {
    float* ys[1] = {y};
    return gemv_seg_launch_group(&W, y ? ys : nullptr, &O, 1, xq, K, stream, dbg);
}

unsigned flags_read_clear_gemv_seg(cudaStream_t stream) {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_flags_gemv_seg, sizeof(v), 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return ~0u;
    if (cudaMemcpyToSymbolAsync(g_flags_gemv_seg, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream) !=
        cudaSuccess)
        return ~0u;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return ~0u;
    return v;
}

}  // namespace qdg

using namespace qdg;

extern "C" int64_t q4_0_seg_row_bytes(int64_t K) {
    if (K <= 0) return QDG_EINVAL;
    if (K % 256 != 0 || K > 32768) return QDG_ESHAPE;
    return seg_row_bytes(K);
}

extern "C" int q4_0_repack_seg(const void* W, void* Wr, int64_t O, int64_t K, qdg_stream_t stream) {
    if (!W || !Wr || O <= 0 || K <= 0) return QDG_EINVAL;
    if (K % 256 != 0 || K > 32768) return QDG_ESHAPE;
    if (!aligned(W, 2) || !aligned(Wr, 16)) return QDG_EALIGN;
    const int nb = static_cast<int>(K / 32);
    const int nseg = (nb + 63) / 64;
    const int64_t warps = O * nseg;
    const int64_t blocks = (warps + 7) / 8;
    if (blocks > 0x7fffffff) return QDG_ESHAPE;
    repack_seg_kernel<<<static_cast<unsigned>(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t*>(W), static_cast<uint8_t*>(Wr), O, nb, nseg, seg_row_bytes(K));
    if (cudaGetLastError() != cudaSuccess) return QDG_ECUDA;
    count_launch(7);
    return QDG_OK;
}

extern "C" int q4_0s_q8_0_gemv(const void* Wr, const void* xq, float* y, int64_t O, int64_t K,
                               qdg_stream_t stream) {
    if (!y) return QDG_EINVAL;
    return gemv_seg_launch(Wr, xq, y, O, K, reinterpret_cast<cudaStream_t>(stream), nullptr);
}

extern "C" int q4_0s_q8_0_gemv_group(const void* const* Wr, float* const* y, const int64_t* O, int count,
                                     const void* xq, int64_t K, qdg_stream_t stream) {
    if (!y) return QDG_EINVAL;
    return gemv_seg_launch_group(Wr, y, O, count, xq, K, reinterpret_cast<cudaStream_t>(stream), nullptr);
}

extern "C" int q4_0s_gemv_rmsnorm_group(const void* const* Wr, float* const* y, const int64_t* O, int count,
                                        const float* x, const float* gamma, float eps, int64_t K, void* xq_out,
                                        qdg_stream_t stream) {
    return gemv_seg_rmsnorm_launch(Wr, y, O, count, x, gamma, eps, K, xq_out, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int q4_0s_q8_0_gemm_small_n(const void* Wr, const void* xq, float* y, int64_t ldy, int64_t O, int64_t K,
                                       int64_t N, qdg_stream_t stream) {
    if (!y) return QDG_EINVAL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (N == 1) {
        if (ldy < O) return QDG_EINVAL;
        return gemv_seg_launch(Wr, xq, y, O, K, s, nullptr);
    }
    if (N == 2) return gemv_seg2_launch(Wr, xq, y, ldy, O, K, s, nullptr);
    if (gemv_segn_supported(K, N)) return gemv_segn_launch(Wr, xq, y, ldy, O, K, N, s, nullptr);
    return small_n_seg_launch(Wr, xq, y, ldy, O, K, N, s, nullptr);
}
