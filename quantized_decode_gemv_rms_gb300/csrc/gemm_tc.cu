// gemm_tc.cu -- prefill Q4_0 x Q8_0 product on the fifth-generation tensor
// cores (the "mmq" route for long batches [GGML: Backend abstraction and
// hardware acceleration, section "CUDA: mmvq, mmq, cublas -- three matrix
// paths": other quantized matrices go to mmq; prefill keeps it busier]).
//
// Y[t][o] = sum_b d_w(o,b) d_x(t,b) isum(t,o,b).  The integer block sums are
// formed by tcgen05.mma kind::f16 on operands holding the integer codes
// exactly in fp16 (q_w - 8 in -8..7, q_x in -127..127): every product and
// every partial sum of a 32-element block is an integer below 2^15, so the
// fp32 accumulation in tensor memory is exact.  (The integer MMA kind is not
// available for sm_103a; the exact fp16 route gives the same sums.)  Scales
// differ per block, so each block's 128x128 sum tile is drained from tensor
// memory and scaled into fp32 registers on the CUDA cores while the tensor
// core works on the next block (two accumulator buffers).
//
// Warp roles in one persistent CTA per SM (tile 128 weight rows x 128 tokens):
//   warp 0      producer: 1-D bulk copies (TMA engine) of raw Q4_0 / Q8_0
//               bytes, 8 blocks per stage, into a ring of shared memory
//   warp 1      tensor-memory allocator and MMA issuer (one thread)
//   warps 2-5   converters: raw blocks -> fp16 operand tiles in the
//               canonical no-swizzle K-major layout (8x16-byte core
//               matrices), plus per-block fp32 scales
//   warps 6-21  drain: tcgen05.ld of the block sums, y += d_w d_x isum
// Every wait is bounded; a timeout sets a flag, the CTA stops working,
// waits for its copies and MMAs in flight, frees tensor memory and exits.
#include "common.cuh"

#include <algorithm>
#include <mutex>

namespace qdg {

static __device__ unsigned g_flags_gemm;

namespace {

constexpr int BM = 128;                  // weight rows per tile (MMA M)
constexpr int BN = 128;                  // tokens per tile (MMA N)
constexpr int CHUNK = 8;                 // blocks per raw stage (144 / 272 bytes per row: 16-byte multiples)
constexpr int RAW_W = BM * CHUNK * 18;   // 18432
constexpr int RAW_X = BN * CHUNK * 34;   // 34816
constexpr int RAW_BYTES = RAW_W + RAW_X; // 53248
constexpr int RS = 2;                    // raw stages
constexpr int OPA = BM * 32 * 2;         // fp16 A tile of one block
constexpr int OPB = BN * 32 * 2;         // fp16 B tile of one block
constexpr int OP_BYTES = OPA + OPB + (BM + BN) * 4;
constexpr int OS = 4;                    // operand slots
constexpr int TMEM_COLS = 2 * BN;        // two accumulator buffers
constexpr int kConvWarps = 4;
constexpr int kDrainWarps = 16;                         // 4 lane quarters x 4 column groups of 32
constexpr int kWarps = 2 + kConvWarps + kDrainWarps;
constexpr int kThreads = 32 * kWarps;
constexpr int OFF_OPS = RS * RAW_BYTES;                  // 106496 (1024-aligned)
constexpr int OFF_BAR = OFF_OPS + OS * OP_BYTES;         // 176128
constexpr int NBARS = 2 * RS + 2 * OS + 4;
constexpr size_t kSmem = OFF_BAR + NBARS * 8 + 16;

static_assert(OFF_OPS % 1024 == 0 && OP_BYTES % 1024 == 0, "operand alignment");

// Instruction descriptor, kind::f16: D fp32, A/B fp16, both K-major, N>>3, M>>4.
constexpr uint32_t kIdesc = (1u << 4) | (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(BM >> 4) << 24);

// Shared-memory matrix descriptor, no swizzle, K-major: core matrices of
// 8 rows x 16 bytes; LBO = distance between K-adjacent core matrices (128 B),
// SBO = distance between row-adjacent 8-row groups (512 B).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
    const uint64_t lbo = 128, sbo = 512;
    return (static_cast<uint64_t>((addr >> 4) & 0x3FFFu)) | (((lbo >> 4) & 0x3FFFull) << 16) |
           (((sbo >> 4) & 0x3FFFull) << 32) | (1ull << 46);
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Four bytes (0..255 each) -> two fp16x2 words holding 1024 + byte.
__device__ __forceinline__ void bytes_to_f16x2(uint32_t w, uint32_t& h01, uint32_t& h23) {
    h01 = __byte_perm(w, 0x64646464u, 0x4140);
    h23 = __byte_perm(w, 0x64646464u, 0x4342);
}

// Wait that also gives up as soon as another warp raised the abort flag.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1; i < kSpinLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 15u) == 0) {
            if (*abort_flag) return false;
            if (global_ns() - t0 > kWaitNs) break;
        }
        if (i >= 32) __nanosleep(64);
    }
    *abort_flag = 1;
    atomicOr(&g_flags_gemm, FLAG_TIMEOUT);
    return false;
}

struct Args {
    const uint8_t* W;
    const uint8_t* xq;
    float* y;
    int32_t* dbg;
    int64_t ldy;
    int O;
    int T;
    int nb;          // K/32
    int rowbytes;    // nb * 18
    int xrow;        // nb * 34
    int mtiles;
    int ntiles;
};

template <bool kDebug>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(Args a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* raw_full = bars;
    uint64_t* raw_empty = raw_full + RS;
    uint64_t* op_full = raw_empty + RS;
    uint64_t* op_empty = op_full + OS;
    uint64_t* tm_full = op_empty + OS;
    uint64_t* tm_empty = tm_full + 2;
    uint32_t* taddr_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(taddr_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int total_tiles = a.mtiles * a.ntiles;
    const int nchunks = a.nb / CHUNK;

    if (threadIdx.x == 0) {
        for (int i = 0; i < RS; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], kConvWarps);
        }
        for (int i = 0; i < OS; ++i) {
            mbar_init(&op_full[i], kConvWarps);
            mbar_init(&op_empty[i], kDrainWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tm_full[i], 1);
            mbar_init(&tm_empty[i], kDrainWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(taddr_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *taddr_slot;
    pdl_trigger();
    pdl_wait();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        const uint64_t policy = l2_policy_evict_first();
        int c = 0;
        for (int tile = blockIdx.x; tile < total_tiles && !*abort_flag; tile += gridDim.x) {
            const int m0 = (tile / a.ntiles) * BM;
            const int n0 = (tile % a.ntiles) * BN;
            const int vrows = min(BM, a.O - m0);
            const int vtoks = min(BN, a.T - n0);
            for (int ch = 0; ch < nchunks; ++ch, ++c) {
                const int s = c % RS;
                if (c >= RS && !__all_sync(0xffffffffu, wait_or_abort(&raw_empty[s], ((c / RS) - 1) & 1, abort_flag)))
                    break;
                uint8_t* st = smem + s * RAW_BYTES;
                if (lane == 0) mbar_arrive_expect_tx(&raw_full[s], vrows * (CHUNK * 18) + vtoks * (CHUNK * 34));
                __syncwarp();
                for (int i = lane; i < vrows; i += 32)
                    bulk_g2s(st + i * (CHUNK * 18),
                             a.W + static_cast<int64_t>(m0 + i) * a.rowbytes + static_cast<int64_t>(ch) * CHUNK * 18,
                             CHUNK * 18, &raw_full[s], policy);
                for (int i = lane; i < vtoks; i += 32)
                    bulk_g2s(st + RAW_W + i * (CHUNK * 34),
                             a.xq + static_cast<int64_t>(n0 + i) * a.xrow + static_cast<int64_t>(ch) * CHUNK * 34,
                             CHUNK * 34, &raw_full[s], policy);
                __syncwarp();
            }
        }
        // Copies still in flight must land before the CTA may exit.
        if (lane == 0)
            for (int k = (c - RS > 0 ? c - RS : 0); k < c; ++k) mbar_wait(&raw_full[k % RS], (k / RS) & 1);
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        int g = 0;
        const uint32_t ops = smem_u32(smem + OFF_OPS);
        for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
            for (int b = 0; b < a.nb; ++b, ++g) {
                const int o = g % OS;
                const int buf = g & 1;
                bool ok = true;
                if (lane == 0) {
                    ok = !*abort_flag && wait_or_abort(&op_full[o], (g / OS) & 1, abort_flag);
                    if (ok && g >= 2) ok = wait_or_abort(&tm_empty[buf], ((g / 2) - 1) & 1, abort_flag);
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t abase = ops + o * OP_BYTES;
                    const uint32_t bbase = abase + OPA;
                    const uint32_t d = tmem + static_cast<uint32_t>(buf * BN);
                    mma_f16(d, smem_desc(abase), smem_desc(bbase), 0u);
                    mma_f16(d, smem_desc(abase + 256), smem_desc(bbase + 256), 1u);
                    mma_commit(&tm_full[buf]);
                }
                __syncwarp();
            }
            if (*abort_flag) break;
        }
        // MMAs in flight must finish before tensor memory is freed.
        if (lane == 0 && g > 0) mbar_wait(&tm_full[(g - 1) & 1], ((g - 1) / 2) & 1);
        __syncwarp();
    } else if (warp < 2 + kConvWarps) {
        // ------------------------------------------------------------ converters
        const int t = threadIdx.x - 64;   // 0..127: weight row t and token t of the tile
        int g = 0;
        for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
            const int m0 = (tile / a.ntiles) * BM;
            const int n0 = (tile % a.ntiles) * BN;
            const bool vrow = m0 + t < a.O;
            const bool vtok = n0 + t < a.T;
            bool ok = true;
            for (int b = 0; b < a.nb; ++b, ++g) {
                const int c = g / CHUNK;
                const int s = c % RS;
                const int bl = g % CHUNK;
                const int o = g % OS;
                if (bl == 0) ok = __all_sync(0xffffffffu, wait_or_abort(&raw_full[s], (c / RS) & 1, abort_flag));
                if (ok && g >= OS)
                    ok = __all_sync(0xffffffffu, wait_or_abort(&op_empty[o], ((g / OS) - 1) & 1, abort_flag));
                if (!ok) break;
                const uint8_t* st = smem + s * RAW_BYTES;
                uint8_t* op = smem + OFF_OPS + o * OP_BYTES;
                float* dws = reinterpret_cast<float*>(op + OPA + OPB);
                float* dxs = dws + BM;
                // ---- A: weight row t, block bl -> 32 fp16 (q - 8)
                uint4 av[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                               make_uint4(0, 0, 0, 0)};
                float dw = 0.0f;
                if (vrow) {
                    const uint8_t* p = st + t * (CHUNK * 18) + bl * 18;
                    uint32_t q[4];
                    uint32_t dbits;
                    if ((bl & 1) == 0) {
                        const uint32_t* pw = reinterpret_cast<const uint32_t*>(p);
                        uint32_t w[5];
#pragma unroll
                        for (int i = 0; i < 5; ++i) w[i] = pw[i];
                        dbits = w[0];
#pragma unroll
                        for (int i = 0; i < 4; ++i) q[i] = bytes_2_to_5(w[i], w[i + 1]);
                    } else {
                        dbits = *reinterpret_cast<const uint32_t*>(p - 2) >> 16;
                        const uint32_t* pw = reinterpret_cast<const uint32_t*>(p + 2);
#pragma unroll
                        for (int i = 0; i < 4; ++i) q[i] = pw[i];
                    }
                    dw = half_bits_to_float(dbits);
                    const uint32_t k1032 = 0x64086408u;
                    uint32_t h[16];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint32_t a01, a23, b01, b23;
                        bytes_to_f16x2(q[i] & 0x0F0F0F0Fu, a01, a23);
                        bytes_to_f16x2((q[i] >> 4) & 0x0F0F0F0Fu, b01, b23);
                        h[2 * i] = hsub2(a01, k1032);          // elements 4i, 4i+1
                        h[2 * i + 1] = hsub2(a23, k1032);      // 4i+2, 4i+3
                        h[8 + 2 * i] = hsub2(b01, k1032);      // 16+4i, 16+4i+1
                        h[8 + 2 * i + 1] = hsub2(b23, k1032);
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) av[j] = make_uint4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    *reinterpret_cast<uint4*>(op + ((t >> 3) * 4 + j) * 128 + (t & 7) * 16) = av[j];
                dws[t] = dw;
                // ---- B: token t, block bl -> 32 fp16 q
                uint4 bv[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                               make_uint4(0, 0, 0, 0)};
                float dx = 0.0f;
                if (vtok) {
                    const uint8_t* p = st + RAW_W + t * (CHUNK * 34) + bl * 34;
                    uint32_t q[8];
                    uint32_t dbits;
                    if ((bl & 1) == 0) {
                        const uint32_t* pw = reinterpret_cast<const uint32_t*>(p);
                        uint32_t w[9];
#pragma unroll
                        for (int i = 0; i < 9; ++i) w[i] = pw[i];
                        dbits = w[0];
#pragma unroll
                        for (int i = 0; i < 8; ++i) q[i] = bytes_2_to_5(w[i], w[i + 1]);
                    } else {
                        dbits = *reinterpret_cast<const uint32_t*>(p - 2) >> 16;
                        const uint32_t* pw = reinterpret_cast<const uint32_t*>(p + 2);
#pragma unroll
                        for (int i = 0; i < 8; ++i) q[i] = pw[i];
                    }
                    dx = half_bits_to_float(dbits);
                    const uint32_t k1152 = 0x64806480u;
                    uint32_t h[16];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        uint32_t h01, h23;
                        bytes_to_f16x2(q[i] ^ 0x80808080u, h01, h23);
                        h[2 * i] = hsub2(h01, k1152);
                        h[2 * i + 1] = hsub2(h23, k1152);
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) bv[j] = make_uint4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    *reinterpret_cast<uint4*>(op + OPA + ((t >> 3) * 4 + j) * 128 + (t & 7) * 16) = bv[j];
                dxs[t] = dx;
                // generic-proxy writes -> visible to the tensor core (async proxy)
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&op_full[o]);
                    if (bl == CHUNK - 1) mbar_arrive(&raw_empty[s]);
                }
            }
            if (!ok) break;
        }
    } else {
        // ------------------------------------------------------------ drain
        const int dq = warp & 3;                    // tensor-memory lane quarter of this warp
        const int h = (warp - 2 - kConvWarps) >> 2; // column group 0..3 (32 tokens each)
        const int r = dq * 32 + lane;               // row within the tile
        float acc[32];
        int g = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
            const int m0 = (tile / a.ntiles) * BM;
            const int n0 = (tile % a.ntiles) * BN;
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[j] = 0.0f;
            for (int b = 0; b < a.nb; ++b, ++g) {
                const int buf = g & 1;
                const int o = g % OS;
                ok = __all_sync(0xffffffffu, wait_or_abort(&tm_full[buf], (g / 2) & 1, abort_flag));
                if (!ok) break;
                tc_fence_after();
                uint32_t v[32];
                tmem_ld32(tmem + (static_cast<uint32_t>(dq * 32) << 16) + static_cast<uint32_t>(buf * BN + 32 * h), v);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tm_empty[buf]);
                const uint8_t* op = smem + OFF_OPS + o * OP_BYTES;
                const float* dws = reinterpret_cast<const float*>(op + OPA + OPB);
                const float4* dx4 = reinterpret_cast<const float4*>(dws + BM + 32 * h);
                const float dw = dws[r];
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const float4 dx = dx4[j4];
                    acc[4 * j4 + 0] = __fmaf_rn(__fmul_rn(dw, dx.x), __uint_as_float(v[4 * j4 + 0]), acc[4 * j4 + 0]);
                    acc[4 * j4 + 1] = __fmaf_rn(__fmul_rn(dw, dx.y), __uint_as_float(v[4 * j4 + 1]), acc[4 * j4 + 1]);
                    acc[4 * j4 + 2] = __fmaf_rn(__fmul_rn(dw, dx.z), __uint_as_float(v[4 * j4 + 2]), acc[4 * j4 + 2]);
                    acc[4 * j4 + 3] = __fmaf_rn(__fmul_rn(dw, dx.w), __uint_as_float(v[4 * j4 + 3]), acc[4 * j4 + 3]);
                }
                if (kDebug) {
                    if (m0 + r < a.O) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const int tok = n0 + 32 * h + j;
                            if (tok < a.T)
                                a.dbg[(static_cast<int64_t>(tok) * a.O + m0 + r) * a.nb + b] =
                                    static_cast<int32_t>(__uint_as_float(v[j]));
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&op_empty[o]);
            }
            if (!ok) break;
            if (a.y != nullptr && m0 + r < a.O) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int tok = n0 + 32 * h + j;
                    if (tok < a.T) a.y[static_cast<int64_t>(tok) * a.ldy + m0 + r] = acc[j];
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
}

std::mutex g_attr_mutex;
bool g_attr_done[2] = {false, false};

template <bool kDebug>
cudaError_t ensure_smem() {
    std::lock_guard<std::mutex> lock(g_attr_mutex);
    if (g_attr_done[kDebug]) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<kDebug>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmem));
    if (e == cudaSuccess) g_attr_done[kDebug] = true;
    return e;
}

}  // namespace

int gemm_launch(const void* W, const void* xq, float* y, int64_t ldy, int64_t O, int64_t K, int64_t T,
                cudaStream_t stream, int32_t* dbg) {
    if (!W || !xq || (!y && !dbg)) return QDG_EINVAL;
    if (O <= 0 || K <= 0 || T <= 0) return QDG_EINVAL;
    if (y && ldy < O) return QDG_EINVAL;
    if (K % 256 != 0 || K > 65536 || O > (1 << 30) || T > (1 << 30)) return QDG_ESHAPE;
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
    a.O = static_cast<int>(O);
    a.T = static_cast<int>(T);
    a.nb = static_cast<int>(K / 32);
    a.rowbytes = a.nb * 18;
    a.xrow = a.nb * 34;
    a.mtiles = static_cast<int>((O + BM - 1) / BM);
    a.ntiles = static_cast<int>((T + BN - 1) / BN);
    const int64_t tiles = static_cast<int64_t>(a.mtiles) * a.ntiles;
    if (tiles > (1 << 30)) return QDG_ESHAPE;
    const int grid = static_cast<int>(std::min<int64_t>(dev.sms, tiles));
    cudaError_t e;
    if (dbg) {
        e = ensure_smem<true>();
        if (e == cudaSuccess) e = launch(gemm_tc_kernel<true>, dim3(grid), dim3(kThreads), kSmem, stream, false, a);
    } else {
        e = ensure_smem<false>();
        if (e == cudaSuccess) e = launch(gemm_tc_kernel<false>, dim3(grid), dim3(kThreads), kSmem, stream, true, a);
    }
    if (e != cudaSuccess) return QDG_ECUDA;
    count_launch(3);
    return QDG_OK;
}

unsigned flags_read_clear_gemm(cudaStream_t stream) {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_flags_gemm, sizeof(v), 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return ~0u;
    if (cudaMemcpyToSymbolAsync(g_flags_gemm, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream) !=
        cudaSuccess)
        return ~0u;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return ~0u;
    return v;
}

}  // namespace qdg

extern "C" int q4_0_q8_0_gemm(const void* W, const void* xq, float* y, int64_t ldy, int64_t O, int64_t K, int64_t T,
                              qdg_stream_t stream) {
    if (!y) return QDG_EINVAL;
    return qdg::gemm_launch(W, xq, y, ldy, O, K, T, reinterpret_cast<cudaStream_t>(stream), nullptr);
}
