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
// core works on the next blocks (four block-sum buffers).
//
// The activations are shared by every 128-row tile of W, so a small first
// kernel converts each Q8_0 block once into the tensor core's operand form
// (fp16 codes in the canonical no-swizzle K-major layout of 8x16-byte core
// matrices, plus the fp32 scale) in a caller-provided workspace; the main
// kernel loads one such 8704-byte record per block with a bulk copy.
//
// Warp roles in one persistent CTA per SM (tile 128 weight rows x 128 tokens):
//   warp 0      producer: a 2-D tensor copy of a 128-row box of raw Q4_0
//               bytes, 8 blocks wide, per raw stage, and the two bulk copies
//               of each block's activation record (fp16 tile into the operand
//               slot, scales into the scale ring), issued from eight lanes at
//               once for four blocks
//   warp 1      tensor-memory allocator and MMA issuer (one thread)
//   warps 2-9   weight converters (row quarter x block parity, two per SMSP):
//               raw blocks -> fp16 operand tiles in the canonical layout plus
//               per-block fp32 scales; raw rows are read as 16-byte vectors
//   warps 10-25 drain: tcgen05.ld of the block sums, y += d_w d_x isum with
//               packed fp32x2 arithmetic
// The converters are spread two per SMSP (measured: a drain warp sharing its
// SMSP with two busy roles fell blocks behind and paced the whole pipeline),
// and the producer and MMA issuer are separate warps (as lanes of one warp
// they serialised each other's waits).
// Every wait is bounded; a timeout sets a flag, the CTA stops working,
// waits for its copies and MMAs in flight, frees tensor memory and exits.
#include "common.cuh"
#include "tma.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

namespace qdg {

static __device__ unsigned g_flags_gemm;

namespace {

constexpr int BM = 128;                  // weight rows per tile (MMA M)
constexpr int BN = 128;                  // tokens per tile (MMA N)
constexpr int CHUNK = 8;                 // blocks per raw stage (144 bytes per row: a 16-byte multiple)
constexpr int RAW_W = BM * CHUNK * 18;   // 18432
constexpr int RS = 3;                    // raw weight stages
constexpr int OPA = BM * 32 * 2;         // fp16 A tile of one block
constexpr int OPB = BN * 32 * 2;         // fp16 B tile of one block
constexpr int XREC = OPB + BN * 4;       // activation record of the workspace: B tile + d_x (8704 bytes)
constexpr int OP_BYTES = OPA + OPB;      // operand slot: [A tile][B tile], released when its MMAs complete
constexpr int OS = 8;                    // operand slots
constexpr int SC_BYTES = (BN + BM) * 4;  // scale entry: [d_x of 128 tokens][d_w of 128 rows], released by the drain
constexpr int SR = 32;                   // scale entries
constexpr int kCopyGroup = 4;            // blocks whose records the producer issues together
constexpr int TB = 4;                    // block-sum buffers in tensor memory
constexpr int TMEM_COLS = TB * BN;       // all 512 columns
constexpr int kConvWarps = 8;                           // weight converters: 4 row quarters x 2 block parities
constexpr int kConvPerBlock = kConvWarps / 2;           // converter warps that write one block
constexpr int kDrainWarps = 16;                         // 4 lane quarters x 4 column groups of 32
constexpr int kWarps = 2 + kConvWarps + kDrainWarps;   // warp 0: producer, warp 1: MMA issuer
constexpr int kThreads = 32 * kWarps;
constexpr int OFF_OPS = RS * RAW_W;                      // 55296 (1024-aligned)
constexpr int OFF_SC = OFF_OPS + OS * OP_BYTES;          // 186368
constexpr int OFF_BAR = OFF_SC + SR * SC_BYTES;           // 194560
constexpr int NBARS = 2 * RS + 2 * OS + 2 * SR + 2 * TB;
constexpr size_t kSmem = OFF_BAR + NBARS * 8 + 16;

static_assert(OFF_OPS % 1024 == 0 && OP_BYTES % 1024 == 0 && RAW_W % 1024 == 0 && XREC % 16 == 0 &&
                  OFF_SC % 16 == 0,
              "operand and stage alignment");

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

// 16 columns of this warp's 32 lanes; completes only at the next tmem_wait.
__device__ __forceinline__ void tmem_ld16_issue(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// Wait for this thread's tensor-memory loads; the registers of a are tied to
// the wait so that no use of them is scheduled before it.
__device__ __forceinline__ void tmem_wait(uint32_t (&a)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]),
                   "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]),
                   "+r"(a[15])
                 :
                 : "memory");
}


__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}



// The 4-byte word starting at byte offset `off` (even, compile-time) of w[].
template <int off>
__device__ __forceinline__ uint32_t word_at(const uint32_t* w) {
    if constexpr ((off & 3) == 0)
        return w[off >> 2];
    else
        return bytes_2_to_5(w[off >> 2], w[(off >> 2) + 1]);
}

// Four bytes (0..255 each) -> two fp16x2 words holding 1024 + byte.
__device__ __forceinline__ void bytes_to_f16x2(uint32_t w, uint32_t& h01, uint32_t& h23) {
    h01 = __byte_perm(w, 0x64646464u, 0x4140);
    h23 = __byte_perm(w, 0x64646464u, 0x4342);
}

// Wait that also gives up as soon as another warp raised the abort flag.
// Each try suspends the thread in hardware until the phase completes (or up
// to kSuspendNs), so waiting warps take no issue slots from working ones.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1; i < kSpinLimit; ++i) {
        if (mbar_try_wait_suspend(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_ns() - t0 > kWaitNs) break;
    }
    *abort_flag = 1;
    atomicOr(&g_flags_gemm, FLAG_TIMEOUT);
    return false;
}

struct Args {
    CUtensorMap wmap;    // Q4_0 bytes: inner dim = row bytes (uint8), outer = O rows
    const uint8_t* W;
    const uint8_t* xrec; // activation records [ntiles][nb][XREC]
    float* y;
    int32_t* dbg;
    int64_t ldy;
    int O;
    int T;
    int nb;          // K/32
    int rowbytes;    // nb * 18
    int mtiles;
    int ntiles;
};

// Weight row t of the tile, block bl0 + kU of the raw chunk at `row` (the
// row's 144 bytes): fp16 codes q - 8 into the A tile at op (canonical layout:
// core matrix (t / 8) * 4 + j holds elements 8j..8j+7, one 16-byte row per
// weight row) and the fp32 scale into dws[t].  Raw rows are read as two
// 16-byte vectors (row stride 9 x 16 bytes: conflict-free).
template <int kU>
__device__ __forceinline__ void convert_block(const uint8_t* row, int bl0, int t, bool valid, uint8_t* op,
                                              float* dws) {
    const int bl = bl0 + kU;
    const int off = (bl * 18) & 15;
    const uint4* rv = reinterpret_cast<const uint4*>(row) + ((bl * 18) >> 4);
    const uint4 c0v = rv[0], c1v = rv[1];
    const uint32_t w[8] = {c0v.x, c0v.y, c0v.z, c0v.w, c1v.x, c1v.y, c1v.z, c1v.w};
    uint32_t q[4] = {0u, 0u, 0u, 0u};
    float dsc = 0.0f;
    if (valid) {
        const uint32_t dbits = (off & 3) == 0 ? w[off >> 2] : (w[off >> 2] >> 16);
        dsc = half_bits_to_float(dbits);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int bo = off + 2 + 4 * i;
            q[i] = (bo & 3) == 0 ? w[bo >> 2] : bytes_2_to_5(w[bo >> 2], w[(bo >> 2) + 1]);
        }
    }
    // core matrix j holds elements 8j..8j+7: low nibbles of words 2j, 2j+1
    // for j < 2, high nibbles of words 2(j-2), 2(j-2)+1 after
    const uint32_t k1032 = 0x64086408u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t wa = q[(2 * j) & 3], wb = q[(2 * j + 1) & 3];
        const uint32_t na = j < 2 ? (wa & 0x0F0F0F0Fu) : ((wa >> 4) & 0x0F0F0F0Fu);
        const uint32_t nb2 = j < 2 ? (wb & 0x0F0F0F0Fu) : ((wb >> 4) & 0x0F0F0F0Fu);
        uint32_t a01, a23, b01, b23;
        bytes_to_f16x2(na, a01, a23);
        bytes_to_f16x2(nb2, b01, b23);
        uint4 v = make_uint4(hsub2(a01, k1032), hsub2(a23, k1032), hsub2(b01, k1032), hsub2(b23, k1032));
        if (!valid) v = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(op + ((t >> 3) * 4 + j) * 128 + (t & 7) * 16) = v;
    }
    dws[t] = dsc;
}

template <bool kDebug>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ Args a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* raw_full = bars;
    uint64_t* raw_empty = raw_full + RS;
    uint64_t* op_full = raw_empty + RS;
    uint64_t* op_empty = op_full + OS;
    uint64_t* sc_full = op_empty + OS;
    uint64_t* sc_empty = sc_full + SR;
    uint64_t* tm_full = sc_empty + SR;
    uint64_t* tm_empty = tm_full + TB;
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
            mbar_init(&op_full[i], kConvPerBlock + 1);   // the converters and the B-tile copy
            mbar_init(&op_empty[i], 1);               // MMA completion
        }
        for (int i = 0; i < SR; ++i) {
            mbar_init(&sc_full[i], kConvPerBlock + 1);   // the converters (d_w) and the d_x copy
            mbar_init(&sc_empty[i], kDrainWarps);
        }
        for (int i = 0; i < TB; ++i) {
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

    if (warp < 2) {
        if (warp == 0) {
            // -------------------------------------------------------- producer (one warp)
            // One issuing thread manages about one bulk copy per 600 cycles
            // (measured), so the copies of a group of four blocks go out from
            // eight lanes at once: lanes 0-3 the fp16 tiles, lanes 4-7 the
            // scales; lane 0 also issues the raw weight stage.
            int c = 0;   // raw weight chunks issued
            int g = 0;   // blocks whose records were issued
            bool ok = true;
            for (int tile = blockIdx.x; tile < total_tiles && ok && !*abort_flag; tile += gridDim.x) {
                const int m0 = (tile / a.ntiles) * BM;
                const int nt = tile % a.ntiles;
                for (int b = 0; b < a.nb; b += kCopyGroup, g += kCopyGroup) {
                    if (b % CHUNK == 0) {
                        const int s = c % RS;
                        bool w = true;
                        if (lane == 0 && c >= RS) w = wait_or_abort(&raw_empty[s], ((c / RS) - 1) & 1, abort_flag);
                        ok = __shfl_sync(0xffffffffu, w, 0);
                        if (!ok) break;
                        if (lane == 0) {
                            // Rows past O are zero-filled by the copy and
                            // still count toward the transaction bytes.
                            mbar_arrive_expect_tx(&raw_full[s], RAW_W);
                            tma_load_2d(smem + s * RAW_W, &a.wmap, (b / CHUNK) * (CHUNK * 18), m0, &raw_full[s]);
                        }
                        ++c;
                    }
                    // Slots and scale entries free in order: waiting for the
                    // last of the group covers the group.
                    const int gl = g + kCopyGroup - 1;
                    bool w = true;
                    if (lane == 0) {
                        if (gl >= OS) w = wait_or_abort(&op_empty[gl % OS], ((gl / OS) - 1) & 1, abort_flag);
                        if (w && gl >= SR) w = wait_or_abort(&sc_empty[gl % SR], ((gl / SR) - 1) & 1, abort_flag);
                    }
                    ok = __shfl_sync(0xffffffffu, w, 0);
                    if (!ok) break;
                    if (lane < 2 * kCopyGroup) {
                        const int u = lane % kCopyGroup;
                        const int gu = g + u;
                        const uint8_t* rec = a.xrec + (static_cast<int64_t>(nt) * a.nb + b + u) * XREC;
                        if (lane < kCopyGroup) {
                            mbar_arrive_expect_tx(&op_full[gu % OS], OPB);
                            bulk_g2s_plain(smem + OFF_OPS + (gu % OS) * OP_BYTES + OPA, rec, OPB, &op_full[gu % OS]);
                        } else {
                            mbar_arrive_expect_tx(&sc_full[gu % SR], BN * 4);
                            bulk_g2s_plain(smem + OFF_SC + (gu % SR) * SC_BYTES, rec + OPB, BN * 4, &sc_full[gu % SR]);
                        }
                    }
                    __syncwarp();
                }
            }
            // Copies still in flight must land before the CTA may exit.
            if (lane == 0) {
                for (int k = (c - RS > 0 ? c - RS : 0); k < c; ++k) mbar_wait(&raw_full[k % RS], (k / RS) & 1);
                if (*abort_flag) {
                    for (int k = (g - OS > 0 ? g - OS : 0); k < g; ++k) mbar_wait(&op_full[k % OS], (k / OS) & 1);
                    for (int k = (g - SR > 0 ? g - SR : 0); k < g; ++k) mbar_wait(&sc_full[k % SR], (k / SR) & 1);
                }
            }
        } else if (warp == 1 && lane == 0) {
            // -------------------------------------------------------- MMA issuer (one thread)
            int g = 0;
            bool ok = true;
            const uint32_t ops = smem_u32(smem + OFF_OPS);
            for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
                for (int b = 0; b < a.nb; ++b, ++g) {
                    const int o = g % OS;
                    const int buf = g % TB;
                    ok = !*abort_flag && wait_or_abort(&op_full[o], (g / OS) & 1, abort_flag) &&
                         (g < TB || wait_or_abort(&tm_empty[buf], ((g / TB) - 1) & 1, abort_flag));
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t abase = ops + o * OP_BYTES;
                    const uint32_t bbase = abase + OPA;
                    const uint32_t d = tmem + static_cast<uint32_t>(buf * BN);
                    mma_f16(d, smem_desc(abase), smem_desc(bbase), 0u);
                    mma_f16(d, smem_desc(abase + 256), smem_desc(bbase + 256), 1u);
                    mma_commit(&tm_full[buf]);
                    mma_commit(&op_empty[o]);   // the operand slot is free once these MMAs complete
                }
            }
            // MMAs in flight must finish before tensor memory is freed.
            if (g > 0) {
                mbar_wait(&tm_full[(g - 1) % TB], ((g - 1) / TB) & 1);
                mbar_wait(&op_empty[(g - 1) % OS], ((g - 1) / OS) & 1);
            }
        }
        __syncwarp();
    } else if (warp < 2 + kConvWarps) {
        // ------------------------------------------------------------ converters
        // Warps 2..9: rows 32 (ci & 3) .. + 31 of the blocks of parity ci >> 2,
        // two warps per SMSP.  Two blocks per step:
        // independent conversions interleave, and the proxy fence and the
        // barrier traffic are paid once per pair.
        const int ci = warp - 2;
        const int t = (ci & 3) * 32 + lane;          // weight row within the tile
        const int par = ci >> 2;
        int g0 = 0;                                   // first block of the current chunk
        bool ok = true;
        for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
            const int m0 = (tile / a.ntiles) * BM;
            const bool valid = m0 + t < a.O;
            for (int ch = 0; ch < nchunks && ok; ++ch, g0 += CHUNK) {
                const int c = g0 / CHUNK;
                const int s = c % RS;
                ok = __all_sync(0xffffffffu, wait_or_abort(&raw_full[s], (c / RS) & 1, abort_flag));
                if (!ok) break;
                const uint8_t* st = smem + s * RAW_W + t * (CHUNK * 18);
#pragma unroll
                for (int bl = 0; bl < CHUNK; bl += 4) {
                    const int ga = g0 + bl + par, gb = ga + 2;
                    bool w_ok = true;
                    if (ga >= OS) w_ok = w_ok && wait_or_abort(&op_empty[ga % OS], ((ga / OS) - 1) & 1, abort_flag);
                    if (ga >= SR) w_ok = w_ok && wait_or_abort(&sc_empty[ga % SR], ((ga / SR) - 1) & 1, abort_flag);
                    if (gb >= OS) w_ok = w_ok && wait_or_abort(&op_empty[gb % OS], ((gb / OS) - 1) & 1, abort_flag);
                    if (gb >= SR) w_ok = w_ok && wait_or_abort(&sc_empty[gb % SR], ((gb / SR) - 1) & 1, abort_flag);
                    ok = __all_sync(0xffffffffu, w_ok);
                    if (!ok) break;
                    if (par == 0) {
                        convert_block<0>(st, bl, t, valid, smem + OFF_OPS + (ga % OS) * OP_BYTES,
                                         reinterpret_cast<float*>(smem + OFF_SC + (ga % SR) * SC_BYTES) + BN);
                        convert_block<2>(st, bl, t, valid, smem + OFF_OPS + (gb % OS) * OP_BYTES,
                                         reinterpret_cast<float*>(smem + OFF_SC + (gb % SR) * SC_BYTES) + BN);
                    } else {
                        convert_block<1>(st, bl, t, valid, smem + OFF_OPS + (ga % OS) * OP_BYTES,
                                         reinterpret_cast<float*>(smem + OFF_SC + (ga % SR) * SC_BYTES) + BN);
                        convert_block<3>(st, bl, t, valid, smem + OFF_OPS + (gb % OS) * OP_BYTES,
                                         reinterpret_cast<float*>(smem + OFF_SC + (gb % SR) * SC_BYTES) + BN);
                    }
                    // generic-proxy writes -> visible to the tensor core (async proxy)
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&op_full[ga % OS]);
                        mbar_arrive(&sc_full[ga % SR]);
                        mbar_arrive(&op_full[gb % OS]);
                        mbar_arrive(&sc_full[gb % SR]);
                        if (bl + 4 == CHUNK) mbar_arrive(&raw_empty[s]);
                    }
                }
            }
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
                const int buf = g % TB;
                const int e = g % SR;
                ok = __all_sync(0xffffffffu, wait_or_abort(&tm_full[buf], (g / TB) & 1, abort_flag) &&
                                                 wait_or_abort(&sc_full[e], (g / SR) & 1, abort_flag));
                if (!ok) break;
                tc_fence_after();
                const uint32_t taddr =
                    tmem + (static_cast<uint32_t>(dq * 32) << 16) + static_cast<uint32_t>(buf * BN + 32 * h);
                const float* sc = reinterpret_cast<const float*>(smem + OFF_SC + e * SC_BYTES);
                const float4* dx4 = reinterpret_cast<const float4*>(sc) + 8 * h;
                const float dw = sc[BN + r];
                // two halves of 16 columns keep the live registers down
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t v[16];
                    tmem_ld16_issue(taddr + 16 * half, v);
                    tmem_wait(v);
                    if (half == 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&tm_empty[buf]);
                    }
#pragma unroll
                    for (int j4 = 0; j4 < 4; ++j4) {
                        const float4 dx = dx4[4 * half + j4];
                        const int j = 16 * half + 4 * j4;
                        float s0, s1, s2, s3;
                        fmul2(s0, s1, dw, dw, dx.x, dx.y);   // per-element scale d_w * d_x
                        fmul2(s2, s3, dw, dw, dx.z, dx.w);
                        ffma2(acc[j], acc[j + 1], s0, s1, __uint_as_float(v[4 * j4]), __uint_as_float(v[4 * j4 + 1]));
                        ffma2(acc[j + 2], acc[j + 3], s2, s3, __uint_as_float(v[4 * j4 + 2]),
                              __uint_as_float(v[4 * j4 + 3]));
                    }
                    if (kDebug) {
                        if (m0 + r < a.O) {
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj) {
                                const int tok = n0 + 32 * h + 16 * half + jj;
                                if (tok < a.T)
                                    a.dbg[(static_cast<int64_t>(tok) * a.O + m0 + r) * a.nb + b] =
                                        static_cast<int32_t>(__uint_as_float(v[jj]));
                            }
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sc_empty[e]);
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

// Activation records: one CTA per (token tile, block), one thread per token.
// Record = fp16 codes of 128 tokens x 32 elements in the canonical K-major
// layout (core matrix (r / 8) * 4 + j holds elements 8j..8j+7 of tokens
// 8 (r / 8) .. + 7, one 16-byte row per token), then the 128 fp32 scales.
// Tokens past T get zero codes and zero scales.
__global__ void __launch_bounds__(BN) act_records_kernel(const uint8_t* __restrict__ xq, int T, int nb,
                                                         uint8_t* __restrict__ rec) {
    const int64_t id = blockIdx.x;             // record = token tile * nb + block
    const int nt = static_cast<int>(id / nb);
    const int b = static_cast<int>(id - static_cast<int64_t>(nt) * nb);
    const int r = threadIdx.x;
    const int t = nt * BN + r;
    uint8_t* out = rec + id * XREC;
    pdl_trigger();
    pdl_wait();
    uint4 v[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    float d = 0.0f;
    if (t < T) {
        const unsigned short* h =
            reinterpret_cast<const unsigned short*>(xq + static_cast<int64_t>(t) * nb * 34 + static_cast<int64_t>(b) * 34);
        d = half_bits_to_float(h[0]);
        const uint32_t k1152 = 0x64806480u;   // fp16 (1152, 1152): (x + 128) + 1024 - 1152 = x
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t hv[4];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int e = 8 * j + 4 * u;   // elements e..e+3
                const uint32_t q = static_cast<uint32_t>(h[1 + e / 2]) | (static_cast<uint32_t>(h[2 + e / 2]) << 16);
                uint32_t h01, h23;
                bytes_to_f16x2(q ^ 0x80808080u, h01, h23);
                hv[2 * u] = hsub2(h01, k1152);
                hv[2 * u + 1] = hsub2(h23, k1152);
            }
            v[j] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) *reinterpret_cast<uint4*>(out + ((r >> 3) * 4 + j) * 128 + (r & 7) * 16) = v[j];
    reinterpret_cast<float*>(out + OPB)[r] = d;
}

template <bool kDebug>
cudaError_t ensure_smem() {
    return ensure_smem_limit(reinterpret_cast<const void*>(gemm_tc_kernel<kDebug>), kSmem);
}

}  // namespace

int64_t gemm_workspace_bytes(int64_t K, int64_t T) {
    if (K <= 0 || T <= 0) return QDG_EINVAL;
    if (K % 256 != 0 || K > 65536 || T > (1 << 30)) return QDG_ESHAPE;
    return (T + BN - 1) / BN * (K / 32) * static_cast<int64_t>(XREC);
}

int gemm_launch(const void* W, const void* xq, float* y, int64_t ldy, int64_t O, int64_t K, int64_t T, void* ws,
                int64_t ws_bytes, cudaStream_t stream, int32_t* dbg) {
    if (!W || !xq || (!y && !dbg) || !ws) return QDG_EINVAL;
    if (O <= 0 || K <= 0 || T <= 0) return QDG_EINVAL;
    if (y && ldy < O) return QDG_EINVAL;
    if (K % 256 != 0 || K > 65536 || O > (1 << 30) || T > (1 << 30)) return QDG_ESHAPE;
    if (!aligned(W, 16) || !aligned(xq, 16) || (y && !aligned(y, 4)) || !aligned(ws, 16)) return QDG_EALIGN;
    if (ws_bytes < gemm_workspace_bytes(K, T)) return QDG_EINVAL;
    const DeviceInfo dev = device_info();
    if (dev.device < 0) return QDG_ECUDA;
    if (kSmem > dev.smem_optin) return QDG_ECUDA;
    Args a{};
    a.W = static_cast<const uint8_t*>(W);
    a.xrec = static_cast<const uint8_t*>(ws);
    a.y = y;
    a.dbg = dbg;
    a.ldy = ldy;
    a.O = static_cast<int>(O);
    a.T = static_cast<int>(T);
    a.nb = static_cast<int>(K / 32);
    a.rowbytes = a.nb * 18;
    a.mtiles = static_cast<int>((O + BM - 1) / BM);
    a.ntiles = static_cast<int>((T + BN - 1) / BN);
    if (!encode_rows(&a.wmap, W, a.rowbytes, O, CHUNK * 18, 128, false)) return QDG_ECUDA;
    const int64_t tiles = static_cast<int64_t>(a.mtiles) * a.ntiles;
    if (tiles > (1 << 30)) return QDG_ESHAPE;
    const int64_t records = static_cast<int64_t>(a.ntiles) * a.nb;
    if (records >= (int64_t(1) << 31)) return QDG_ESHAPE;
    const int grid = static_cast<int>(std::min<int64_t>(dev.sms, tiles));
    cudaError_t e = launch(act_records_kernel, dim3(static_cast<unsigned>(records)), dim3(BN), 0, stream, !dbg,
                           static_cast<const uint8_t*>(xq), a.T, a.nb, static_cast<uint8_t*>(ws));
    if (e != cudaSuccess) return QDG_ECUDA;
    count_launch(3);
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

extern "C" int64_t q4_0_q8_0_gemm_workspace_bytes(int64_t K, int64_t T) { return qdg::gemm_workspace_bytes(K, T); }

extern "C" int64_t q4_0_q8_0_gemm_workspace_size(int64_t O, int64_t K, int64_t T) {
    if (O < 1) return QDG_EINVAL;
    if (O > (1 << 30)) return QDG_ESHAPE;   // the product refuses such an O as well
    return qdg::gemm_workspace_bytes(K, T);
}

extern "C" int q4_0_q8_0_gemm(const void* W, const void* xq, float* y, int64_t ldy, int64_t O, int64_t K, int64_t T,
                              void* workspace, int64_t workspace_bytes, qdg_stream_t stream) {
    if (!y) return QDG_EINVAL;
    return qdg::gemm_launch(W, xq, y, ldy, O, K, T, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream),
                            nullptr);
}

// ---------------------------------------------------------------------------
// q4_0_q8_0_gemm_static: the same product for callers that cannot allocate
// device memory.  Its activation records live in a file-scope device array of
// kStaticWorkspaceBytes (16 MiB); larger problems are rejected with
// QDG_ESHAPE.  The array's device address is looked up once per device, on
// that device's first call (which should therefore come before any stream
// capture).  Nothing in the array needs to start at zero: every call writes
// all the records it reads before reading them.  All calls share the array,
// so calls that overlap on the GPU race.
namespace qdg {
namespace {

constexpr int64_t kStaticWorkspaceBytes = int64_t(16) << 20;
constexpr int kMaxDevices = 64;
static __device__ __align__(256) uint8_t g_static_ws[kStaticWorkspaceBytes];

std::mutex g_static_mutex;
void* g_static_ptr[kMaxDevices] = {};

// Device address of g_static_ws on the current device (set-up on first use).
void* static_workspace() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_static_mutex);
    if (g_static_ptr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_ws) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_static_ptr[dev] = ptr;
    }
    return g_static_ptr[dev];
}

}  // namespace
}  // namespace qdg

extern "C" int q4_0_q8_0_gemm_static(const void* W, const void* xq, float* y, int64_t ldy, int64_t O, int64_t K,
                                     int64_t T, qdg_stream_t stream) {
    if (!y) return QDG_EINVAL;
    const int64_t bytes = qdg::gemm_workspace_bytes(K, T);
    if (bytes < 0) return static_cast<int>(bytes);
    if (bytes > qdg::kStaticWorkspaceBytes) return QDG_ESHAPE;
    void* ws = qdg::static_workspace();
    if (ws == nullptr) return QDG_ECUDA;
    return qdg::gemm_launch(W, xq, y, ldy, O, K, T, ws, qdg::kStaticWorkspaceBytes,
                            reinterpret_cast<cudaStream_t>(stream), nullptr);
}
