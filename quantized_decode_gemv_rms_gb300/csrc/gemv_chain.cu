// gemv_chain.cu -- the stages of a decode step (RMS_NORM * gamma -> Q8_0 of
// a stage's input, then the Q4_0 x Q8_0 products that read it) run by one
// persistent launch, each stage after every output of the stage before it.
//
// Why one launch.  A stage boundary on the chain of separate launches
// (quantize kernel, then GEMV) costs two grid completions, a launch and a
// round trip for the Q8_0 vector that queues behind the GEMV's own weight
// loads: measured per-CTA timelines of the 8B-shaped step on GB300 showed
// 4.5-5.5 us from the end of one GEMV to the first block dot of the next,
// with HBM mostly idle, at each of five boundaries.  The pages tie a lost
// RMS_NORM+MUL fusion to a ~5% token-generation loss [llama.cpp b10909:
// Metal backend fusion-table refactor, introduction]; the fusion here goes
// one step further and takes the launch boundary out as well.
//
// Design (one CTA of 16 warps per SM, cooperative launch: every CTA is
// resident, so CTAs may wait on one another):
//   * Stage input.  After the stage barrier every CTA copies x (and gamma)
//     into shared memory with 16-byte cp.async copies cached in L2 only,
//     forms sum(x^2) in the library's fixed order and quantizes every block
//     with the arithmetic of the standalone quantize kernel, so its Q8_0
//     vector is the same bit for bit (CTA 0 also writes it out when asked).
//     The codes go to two shared planes (bytes 0-15 and 16-31 of each block)
//     so that lanes reading consecutive blocks hit distinct banks; the fp32
//     scale and the code sum of each block sit beside them.
//   * Products.  The stage's matrices are stacked row by row.  Work comes in
//     units of U consecutive rows (U = 4, 2 or 1 by the segment count, so a
//     unit has at least four row-segments), dealt to the warps of the grid
//     in turn.  A warp runs
//     a unit's row-segments segment by segment through an eight-deep
//     register ring (two 16-byte nibble loads and one scale word per lane,
//     the segment layout of gemv_seg.cu), reloads its activation blocks from
//     shared memory once per segment, accumulates each row in a lane
//     register, and reduces the unit's rows in one transposed butterfly.
//     The order of every row's sum is fixed, whichever warp takes the unit.
//   * Stage boundary.  While a stage streams, its successor's input vectors
//     are prefetched into L2 (marked to stay), so that reading them after the
//     barrier does not queue behind weight traffic in HBM.  A warp that runs
//     out of units asks L2 to prefetch its first three units of the next
//     stage, so HBM keeps streaming while the CTAs meet at the barrier
//     (release/acquire through an arrival counter) and requantize the input.
//   * The sync words (arrival counters) start at zero; the last CTA to
//     finish returns them to zero for the next launch.
// Every wait is bounded; a timeout sets the device flag (QDG_ETIMEOUT).
#include "common.cuh"

#include <algorithm>

namespace qdg {

static __device__ unsigned g_flags_chain;

namespace {

constexpr int kWarps = 16;
constexpr int kThreads = 32 * kWarps;
constexpr int kMaxStages = 8;
constexpr int kMaxMats = 4;
constexpr int kMaxK = 16384;
constexpr int kMaxBlocks = kMaxK / 32;
constexpr int kDepth = 8;                   // row-segments in flight per warp
constexpr int kSegStride = 1152;            // segment layout: 64 x 16 nibble bytes + 128 bytes of scale words
constexpr int kPrefetchCap = 9216;          // bytes of its first unit a warp prefetches into L2 at a stage change
constexpr uint32_t kNibbles = 0x0F0F0F0Fu;
constexpr size_t kImageBytes = static_cast<size_t>(kMaxBlocks) * (16 + 16 + 8);   // a stage input's block image
constexpr size_t kSmemBytes = static_cast<size_t>(kMaxK) * 4 + kImageBytes;
constexpr int kCounters = 16;   // [0, 8): stage-done barriers, [8, 16): input-ready barriers

struct Stage {
    const float* x;
    const float* gamma;          // nullptr: plain quantization
    uint8_t* xq_out;             // nullptr: the Q8_0 vector is not written out
    const uint8_t* W[kMaxMats];  // segment layout
    float* y[kMaxMats];
    int64_t start[kMaxMats];     // first stacked row of matrix i
    int64_t rows;                // stacked rows
    int units;                   // ceil(rows / U)
    int count;
    int K, nb, nseg, rlast, rowbytes;
    int U;                       // rows per unit: 4, 2 or 1
};

struct ChainArgs {
    Stage st[kMaxStages];
    int nstages;
    float eps;
    unsigned* sync;              // kCounters arrival counters, then the block image (kImageBytes)
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

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void l2_prefetch(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// The same, marked to stay in L2 ahead of the streamed weights.
__device__ __forceinline__ void l2_prefetch_keep(const void* p, uint32_t bytes) {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(p), "r"(bytes), "l"(pol)
                 : "memory");
}

// A stage's input vectors into L2 (one thread).  Reading them later after
// the stage barrier still sees every write before it: L2 is the point of
// coherence, so the prefetch only moves the copy closer.
__device__ __forceinline__ void prefetch_input(const Stage& S) {
    l2_prefetch_keep(S.x, static_cast<uint32_t>(S.K) * 4);
    if (S.gamma != nullptr) l2_prefetch_keep(S.gamma, static_cast<uint32_t>(S.K) * 4);
}

// Sum over one block of code * q_x, codes unsigned 0..15: low nibbles of
// word i are elements 4i..4i+3, high nibbles elements 16+4i..16+4i+3.
__device__ __forceinline__ int block_dot(const uint4& q, const uint4& x0, const uint4& x1) {
    int acc = 0;
    acc = __dp4a(static_cast<int>(q.x & kNibbles), static_cast<int>(x0.x), acc);
    acc = __dp4a(static_cast<int>((q.x >> 4) & kNibbles), static_cast<int>(x1.x), acc);
    acc = __dp4a(static_cast<int>(q.y & kNibbles), static_cast<int>(x0.y), acc);
    acc = __dp4a(static_cast<int>((q.y >> 4) & kNibbles), static_cast<int>(x1.y), acc);
    acc = __dp4a(static_cast<int>(q.z & kNibbles), static_cast<int>(x0.z), acc);
    acc = __dp4a(static_cast<int>((q.z >> 4) & kNibbles), static_cast<int>(x1.z), acc);
    acc = __dp4a(static_cast<int>(q.w & kNibbles), static_cast<int>(x0.w), acc);
    acc = __dp4a(static_cast<int>((q.w >> 4) & kNibbles), static_cast<int>(x1.w), acc);
    return acc;
}

struct Entry {
    uint4 a, b;     // nibbles of blocks 64s+l and 64s+32+l
    uint32_t sc;    // their scales (low, high half)
};

// Shared-memory image of a stage's quantized input.
struct ActSmem {
    uint4* p0;      // [nb] codes 0..15 of each block
    uint4* p1;      // [nb] codes 16..31
    int2* ds;       // [nb] (fp32 bits of the fp16 scale, sum of the codes)
};

// A warp's units of a stage: c + G (w + 16 k), k = 0, 1, ... for warp w of
// CTA c (G CTAs), so that consecutive units go to consecutive CTAs and even
// a stage of fewer units than warps keeps every SM streaming.  (Measured on
// GB300 against warps taking units one by one from a global counter: 112
// against 130 us for the 8B-shaped step; the counter's atomics serialise.)
struct UnitSource {
    int next;
    __device__ __forceinline__ void reset() {
        next = static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) * (threadIdx.x >> 5);
    }
    __device__ __forceinline__ int take() {
        const int u = next;
        next += static_cast<int>(gridDim.x) * kWarps;
        return u;
    }
};

__device__ __forceinline__ int matrix_of(const Stage& S, int64_t row) {
    int g = 0;
#pragma unroll
    for (int i = 1; i < kMaxMats; ++i)
        if (i < S.count && row >= S.start[i]) g = i;
    return g;
}

__device__ __forceinline__ void prefetch_unit(const Stage& S, int unit, int lane) {
    if (lane != 0 || unit >= S.units) return;
    const int64_t row = static_cast<int64_t>(unit) * S.U;
    const int g = matrix_of(S, row);
    const int64_t mend = (g + 1 < S.count) ? S.start[g + 1] : S.rows;
    const int64_t n = min(static_cast<int64_t>(S.U), mend - row);
    const int64_t bytes = min(n * S.rowbytes, static_cast<int64_t>(kPrefetchCap));
    l2_prefetch(S.W[g] + (row - S.start[g]) * S.rowbytes, static_cast<uint32_t>(bytes));
}

// Bounded wait of thread 0 until `count` CTAs have arrived.
__device__ __forceinline__ void wait_arrivals(const unsigned* arrive, unsigned count) {
    if (ld_acquire(arrive) >= count) return;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0; i < kSpinLimit; ++i) {
        __nanosleep(20);
        if (ld_acquire(arrive) >= count) return;
        if (global_ns() - t0 > kWaitNs) break;
    }
    atomicOr(&g_flags_chain, FLAG_TIMEOUT);
}

// Bounded grid-wide barrier on an arrival counter: the CTA's writes are
// released by its arrival (after the CTA barrier, so every thread's), and
// the acquiring load of the full count orders the reads that follow (the
// CTA barrier after it passes the order on to every thread).
__device__ __forceinline__ void grid_barrier(unsigned* ctr) {
    __syncthreads();
    if (threadIdx.x == 0) {
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ctr) : "memory");
        wait_arrivals(ctr, gridDim.x);
    }
    __syncthreads();
}

// Stage input: the statistic, this CTA's share of the Q8_0 blocks, a grid
// barrier, then every block's image in shared memory.  Same arithmetic and
// order as qnorm_q8_kernel: chains j = i mod 256 summed with fma in
// ascending i, xor butterflies (16, 8, 4, 2, 1),
// ((w0+w1)+(w2+w3))+((w4+w5)+(w6+w7)), s = 1/sqrt(sum/K + eps);
// v = (x*s)*gamma; d = max|v|/127; q = round(v/d) (halves away from zero),
// clamped to +-127; stored scale fp16(d).
//   Every CTA forms the statistic (it needs all of x, 16 KB at K = 4096);
//   block b is quantized by warp b / G of CTA b mod G (G CTAs) and written
//   to the workspace image (and to xq_out when asked); after the barrier
//   each CTA copies the whole image into shared memory.  (Quantizing every
//   block in every CTA measured 2.5 us per 4096 elements on GB300: about
//   40 cycles a block on the SM, times K/32 blocks.)
__device__ void stage_input(const Stage& S, float eps, float* xs, const ActSmem& act, float* wsum, uint8_t* image,
                            unsigned* ready) {
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int K = S.K, nb = S.nb;
    const float* x = S.x;
    const float* gamma = S.gamma;
    uint8_t* xq_out = S.xq_out;
    float s = 1.0f;
    if (gamma != nullptr) {
        for (int i = tid * 4; i < K; i += kThreads * 4) cp_async16(xs + i, x + i);
        cp_async_wait_all();
        __syncthreads();
        if (tid < 256) {
            float acc = 0.0f;
            for (int i = tid; i < K; i += 256) acc = __fmaf_rn(xs[i], xs[i], acc);
            acc = warp_sum(acc);
            if (lane == 0) wsum[warp] = acc;
        }
        __syncthreads();
        const float ss = __fadd_rn(__fadd_rn(__fadd_rn(wsum[0], wsum[1]), __fadd_rn(wsum[2], wsum[3])),
                                   __fadd_rn(__fadd_rn(wsum[4], wsum[5]), __fadd_rn(wsum[6], wsum[7])));
        const float mean = __fdiv_rn(ss, static_cast<float>(K));
        s = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
    }
    const int b = static_cast<int>(blockIdx.x) + warp * static_cast<int>(gridDim.x);
    if (b < nb) {
        float v;
        if (gamma != nullptr)
            v = __fmul_rn(__fmul_rn(xs[(b << 5) + lane], s), __ldg(gamma + (b << 5) + lane));
        else
            v = __ldcg(x + (b << 5) + lane);   // x may be an earlier stage's output: read it at L2
        float m = fabsf(v);
#pragma unroll
        for (int h = 16; h >= 1; h >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, h));
        const float d = __fdiv_rn(m, 127.0f);
        int q = 0;
        if (d != 0.0f) {
            float r = roundf(__fdiv_rn(v, d));
            r = fminf(fmaxf(r, -127.0f), 127.0f);
            q = static_cast<int>(r);
        }
        const int qsum = __reduce_add_sync(0xffffffffu, q);
        const __half dh = __float2half_rn(d);
        const uint8_t code = static_cast<uint8_t>(static_cast<int8_t>(q));
        image[(lane < 16 ? 0 : 16 * kMaxBlocks - 16) + 16 * b + lane] = code;
        if (lane == 0) {
            reinterpret_cast<int2*>(image + 32 * kMaxBlocks)[b] = make_int2(__float_as_int(__half2float(dh)), qsum);
            if (__hisinf(dh)) atomicOr(&g_flags_chain, FLAG_OVERFLOW);
        }
        if (xq_out != nullptr) {
            uint8_t* blk = xq_out + static_cast<int64_t>(b) * 34;
            if (lane == 0) *reinterpret_cast<unsigned short*>(blk) = __half_as_ushort(dh);
            blk[2 + lane] = code;
        }
    }
    grid_barrier(ready);
    // the image: planes of nb x 16 bytes at 0 and 16 kMaxBlocks, (scale, sum) pairs at 32 kMaxBlocks
    uint8_t* dst = reinterpret_cast<uint8_t*>(act.p0);
    for (int i = tid * 16; i < 16 * nb; i += kThreads * 16) {
        cp_async16(dst + i, image + i);
        cp_async16(dst + 16 * kMaxBlocks + i, image + 16 * kMaxBlocks + i);
    }
    for (int i = tid * 16; i < 8 * nb; i += kThreads * 16) cp_async16(dst + 32 * kMaxBlocks + i, image + 32 * kMaxBlocks + i);
    cp_async_wait_all();
    __syncthreads();
}

// A warp's place in a stage's items.  Items are a unit's row-segments in the
// order (segment s, row r), r fastest; U * nseg >= 4 items a unit, so the
// loader, kDepth items ahead of the consumer, is at most two units ahead.
struct WarpState {
    int cu, n1, n2;     // the unit being consumed and the next two
    int lk, ls, lr;     // loader: unit slot (0: cu, 1: n1, 2: n2), segment, row
};

// Load the loader's item into e and advance the loader.
template <int U>
__device__ __forceinline__ void load_item(const Stage& S, WarpState& w, Entry& e, int lane) {
    const int unit = w.lk == 0 ? w.cu : (w.lk == 1 ? w.n1 : w.n2);
    const int64_t row = static_cast<int64_t>(unit) * U + w.lr;
    e.a = make_uint4(0, 0, 0, 0);
    e.b = e.a;
    e.sc = 0;
    if (unit < S.units && row < S.rows) {
        const int g = matrix_of(S, row);
        const int r = (w.ls == S.nseg - 1) ? S.rlast : 64;
        const uint8_t* base = S.W[g] + (row - S.start[g]) * S.rowbytes + w.ls * kSegStride;
        if (lane < r) e.a = ldg_stream16(base + 16 * lane);
        if (lane + 32 < r) e.b = ldg_stream16(base + 16 * lane + 512);
        e.sc = ldg_stream4(base + 16 * r + 4 * lane);
    }
    if (++w.lr == U) {
        w.lr = 0;
        if (++w.ls == S.nseg) {
            w.ls = 0;
            ++w.lk;
        }
    }
}

// Take the warp's first three units of a stage and fill the ring with its
// first kDepth items (weights only: this may run before the stage's input
// is ready); the rows of the later units head for L2.
template <int U>
__device__ __forceinline__ void fill_ring(const Stage& S, WarpState& w, Entry (&ring)[kDepth], UnitSource& src,
                                          int lane) {
    w.cu = src.take();
    w.n1 = src.take();
    w.n2 = src.take();
    w.lk = w.ls = w.lr = 0;
#pragma unroll
    for (int k = 0; k < kDepth; ++k) load_item<U>(S, w, ring[k], lane);
    prefetch_unit(S, w.n1, lane);
    prefetch_unit(S, w.n2, lane);
}

__device__ __forceinline__ void fill_ring_any(const Stage& S, WarpState& w, Entry (&ring)[kDepth], UnitSource& src,
                                              int lane) {
    if (S.U == 4)
        fill_ring<4>(S, w, ring, src, lane);
    else if (S.U == 2)
        fill_ring<2>(S, w, ring, src, lane);
    else
        fill_ring<1>(S, w, ring, src, lane);
}

// One stage's products, one warp, from a filled ring: consume every unit the
// warp takes; each item is dotted and its ring entry refilled with the item
// kDepth ahead.
template <int U>
__device__ __forceinline__ void stage_products(const Stage& S, const ActSmem& act, UnitSource& src, WarpState& w,
                                               Entry (&ring)[kDepth]) {
    static_assert(kDepth % U == 0 && U <= 4, "unit rows divide the ring");
    const int lane = threadIdx.x & 31;
    const int nseg = S.nseg;
    // consumer: segment of the current item; activations of that segment
    int cs = 0;
    uint4 xa0, xa1, xb0, xb1;
    float dxa = 0.0f, dxb = 0.0f;
    int sa = 0, sb = 0;
    float acc[U];
#pragma unroll
    for (int r = 0; r < U; ++r) acc[r] = 0.0f;

    while (w.cu < S.units) {
#pragma unroll
        for (int k = 0; k < kDepth; ++k) {
            const int r = k % U;
            if (r == 0) {
                // a new segment: this lane's two activation blocks
                const int ba = 64 * cs + lane, bb = ba + 32;
                const int rseg = (cs == nseg - 1) ? S.rlast : 64;
                xa0 = xa1 = xb0 = xb1 = make_uint4(0, 0, 0, 0);
                dxa = dxb = 0.0f;
                sa = sb = 0;
                if (lane < rseg) {
                    xa0 = act.p0[ba];
                    xa1 = act.p1[ba];
                    const int2 t = act.ds[ba];
                    dxa = __int_as_float(t.x);
                    sa = t.y;
                }
                if (lane + 32 < rseg) {
                    xb0 = act.p0[bb];
                    xb1 = act.p1[bb];
                    const int2 t = act.ds[bb];
                    dxb = __int_as_float(t.x);
                    sb = t.y;
                }
            }
            Entry& e = ring[k];
            const int ia = block_dot(e.a, xa0, xa1) - 8 * sa;
            const int ib = block_dot(e.b, xb0, xb1) - 8 * sb;
            const float dwa = half_bits_to_float(e.sc);
            const float dwb = half_bits_to_float(e.sc >> 16);
            float p = __fmul_rn(__fmul_rn(dwa, dxa), static_cast<float>(ia));
            p = __fmaf_rn(__fmul_rn(dwb, dxb), static_cast<float>(ib), p);
            acc[r] = __fadd_rn(acc[r], p);
            load_item<U>(S, w, e, lane);   // refill with the item kDepth ahead
            if (r == U - 1) {
                if (++cs == nseg) {
                    // the unit is complete: its U rows in one transposed butterfly
                    const bool up16 = (lane & 16) != 0, up8 = (lane & 8) != 0;
                    const float v0 = acc[0], v1 = U > 1 ? acc[1] : 0.0f;
                    const float v2 = U > 2 ? acc[2] : 0.0f, v3 = U > 3 ? acc[3] : 0.0f;
                    float k0 = up16 ? v2 : v0, k1 = up16 ? v3 : v1;
                    k0 = __fadd_rn(k0, __shfl_xor_sync(0xffffffffu, up16 ? v0 : v2, 16));
                    k1 = __fadd_rn(k1, __shfl_xor_sync(0xffffffffu, up16 ? v1 : v3, 16));
                    float mm = up8 ? k1 : k0;
                    mm = __fadd_rn(mm, __shfl_xor_sync(0xffffffffu, up8 ? k0 : k1, 8));
#pragma unroll
                    for (int h = 4; h >= 1; h >>= 1) mm = __fadd_rn(mm, __shfl_xor_sync(0xffffffffu, mm, h));
                    const int q = lane >> 3;
                    const int64_t row = static_cast<int64_t>(w.cu) * U + q;
                    if ((lane & 7) == 0 && q < U && row < S.rows) {
                        const int g = matrix_of(S, row);
                        S.y[g][row - S.start[g]] = mm;
                    }
#pragma unroll
                    for (int rr = 0; rr < U; ++rr) acc[rr] = 0.0f;
                    cs = 0;
                    w.cu = w.n1;
                    w.n1 = w.n2;
                    w.n2 = src.take();
                    --w.lk;
                    if (w.cu >= S.units) break;
                }
            }
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1) gemv_chain_kernel(const __grid_constant__ ChainArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ float wsum[8];
    // The current stage's description, copied out of the parameter block:
    // the loops read its fields at shared-memory latency (read through the
    // parameter block's generic address, each field cost a cached global
    // load on the dependent path; measured: 2.8 us of every 4096-element
    // stage input went to the quantize loop's field reads).
    __shared__ __align__(16) Stage cur;
    static_assert(sizeof(Stage) % 4 == 0 && sizeof(Stage) / 4 <= kThreads, "stage copy by one word a thread");
    float* xs = reinterpret_cast<float*>(smem);
    ActSmem act;
    act.p0 = reinterpret_cast<uint4*>(xs + kMaxK);
    act.p1 = act.p0 + kMaxBlocks;
    act.ds = reinterpret_cast<int2*>(act.p1 + kMaxBlocks);
    const int lane = threadIdx.x & 31;
    unsigned* arrive = a.sync;
    uint8_t* image = reinterpret_cast<uint8_t*>(a.sync + kCounters);

    // Stage 0's first items are loaded (and its next units prefetched into
    // L2) before the wait for the preceding grid: weights never depend on it.
    if (threadIdx.x < sizeof(Stage) / 4)
        reinterpret_cast<uint32_t*>(&cur)[threadIdx.x] = reinterpret_cast<const uint32_t*>(&a.st[0])[threadIdx.x];
    __syncthreads();
    UnitSource src;
    src.reset();
    WarpState w;
    Entry ring[kDepth];
    fill_ring_any(cur, w, ring, src, lane);
    if (blockIdx.x == 0 && threadIdx.x == 0) prefetch_input(cur);
    pdl_wait();

    for (int g = 0; g < a.nstages; ++g) {
        const Stage& S = cur;
        stage_input(S, a.eps, xs, act, wsum, image, &arrive[kMaxStages + g]);
        // the next stage's input heads for L2 while this stage streams
        if (g + 1 < a.nstages && blockIdx.x == 0 && threadIdx.x == 0) prefetch_input(a.st[g + 1]);
        if (S.U == 4)
            stage_products<4>(S, act, src, w, ring);
        else if (S.U == 2)
            stage_products<2>(S, act, src, w, ring);
        else
            stage_products<1>(S, act, src, w, ring);
        if (g + 1 < a.nstages) {
            // the next stage's first items are in flight while the CTAs meet
            // at the barrier and quantize its input
            __syncthreads();
            if (threadIdx.x < sizeof(Stage) / 4)
                reinterpret_cast<uint32_t*>(&cur)[threadIdx.x] =
                    reinterpret_cast<const uint32_t*>(&a.st[g + 1])[threadIdx.x];
            __syncthreads();
            src.reset();
            fill_ring_any(cur, w, ring, src, lane);
            grid_barrier(&arrive[g]);   // every output of stage g is written
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(&arrive[a.nstages - 1], 1u);
        if (prev == gridDim.x - 1) {
            // every CTA is past every use of the counters: back to zero
            for (int c = 0; c < kCounters; ++c) atomicExch(&arrive[c], 0u);
            __threadfence();
        }
    }
}

}  // namespace

unsigned flags_read_clear_chain(cudaStream_t stream) {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_flags_chain, sizeof(v), 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return ~0u;
    if (cudaMemcpyToSymbolAsync(g_flags_chain, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream) !=
        cudaSuccess)
        return ~0u;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return ~0u;
    return v;
}

int chain_launch(const qdg_chain_stage* stages, int nstages, float eps, void* sync, cudaStream_t stream) {
    if (!stages || !sync) return QDG_EINVAL;
    if (nstages < 1 || nstages > kMaxStages) return QDG_EINVAL;
    if (!(eps >= 0.0f) || std::isinf(eps)) return QDG_EINVAL;
    if (!aligned(sync, 16)) return QDG_EALIGN;
    ChainArgs a{};
    a.nstages = nstages;
    a.eps = eps;
    a.sync = static_cast<unsigned*>(sync);
    for (int g = 0; g < nstages; ++g) {
        const qdg_chain_stage& in = stages[g];
        Stage& S = a.st[g];
        if (!in.x || in.count < 1 || in.count > kMaxMats || in.K <= 0) return QDG_EINVAL;
        if (in.K % 256 != 0 || in.K > kMaxK) return QDG_ESHAPE;
        if (!aligned(in.x, 16) || (in.gamma && !aligned(in.gamma, 16)) || !aligned(in.xq_out, 2)) return QDG_EALIGN;
        S.x = in.x;
        S.gamma = in.gamma;
        S.xq_out = static_cast<uint8_t*>(in.xq_out);
        int64_t total = 0;
        for (int i = 0; i < in.count; ++i) {
            if (!in.W[i] || !in.y[i] || in.O[i] <= 0) return QDG_EINVAL;
            if (!aligned(in.W[i], 16) || !aligned(in.y[i], 4)) return QDG_EALIGN;
            S.W[i] = static_cast<const uint8_t*>(in.W[i]);
            S.y[i] = in.y[i];
            S.start[i] = total;
            total += in.O[i];
        }
        if (total >= (int64_t(1) << 30)) return QDG_ESHAPE;   // unit indices stay far from the int range
        S.count = in.count;
        S.rows = total;
        S.K = static_cast<int>(in.K);
        S.nb = S.K / 32;
        S.nseg = (S.nb + 63) / 64;
        S.rlast = S.nb - 64 * (S.nseg - 1);
        S.rowbytes = static_cast<int>(q4_0_seg_row_bytes(in.K));
        S.U = S.nseg <= 2 ? 4 : (S.nseg <= 4 ? 2 : 1);
        S.units = static_cast<int>((total + S.U - 1) / S.U);
    }
    const DeviceInfo dev = device_info();
    if (dev.device < 0) return QDG_ECUDA;
    if (kSmemBytes > dev.smem_optin) return QDG_ECUDA;
    if (ensure_smem_limit(reinterpret_cast<const void*>(gemv_chain_kernel), kSmemBytes) != cudaSuccess)
        return QDG_ECUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(dev.sms));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;   // every CTA resident: they wait on one another
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (pdl_enabled()) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 2;
    }
    cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_chain_kernel, a);
    if (e != cudaSuccess && cfg.numAttrs == 2) {
        // a cooperative launch that may not also be a programmatic dependent:
        // launch it stream-ordered instead
        cudaGetLastError();
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, gemv_chain_kernel, a);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return QDG_ECUDA;
    }
    count_launch(11);
    return QDG_OK;
}

}  // namespace qdg

using namespace qdg;

extern "C" int64_t q4_0s_gemv_chain_workspace_bytes(void) {
    return static_cast<int64_t>(kCounters * sizeof(unsigned) + kImageBytes);
}

extern "C" int q4_0s_gemv_chain(const qdg_chain_stage* stages, int nstages, float eps, void* workspace,
                                qdg_stream_t stream) {
    return chain_launch(stages, nstages, eps, workspace, reinterpret_cast<cudaStream_t>(stream));
}
