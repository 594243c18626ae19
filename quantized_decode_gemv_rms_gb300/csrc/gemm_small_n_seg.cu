// gemm_small_n_seg.cu -- the small-N product (3..8 activation vectors sharing
// one pass over W) on weights in the segment layout, the GPU weight layout the
// library repacks Q4_0 rows into at load time [GGML: Backend abstraction and
// hardware acceleration, section "CUDA: mmvq, mmq, cublas -- three matrix
// paths": the vector case of the quantized matrix-vector route].
//
// Arithmetic and work split are those of the plain-layout kernel
// (gemm_small_n.cu), so the results are the same bit for bit: exact block
// sums from the fp16 warp MMA m16n8k16 on integer-valued operands, a warp per
// 8-block chunk of K with its activation fragments in registers, 16-row
// tiles, partial sums combined in a fixed order across the CTA's warps and,
// for K > 4096, across a thread-block cluster.  What differs is the weight
// path.  In the segment layout a chunk's bytes of one row are 128 contiguous
// nibble bytes and 32 contiguous scale bytes, so each warp stages only what
// it reads itself: per tile, five 16-byte asynchronous copies a lane (every
// warp instruction moving four whole 128-byte row pieces) into a private
// three-tile ring in shared memory, with no hand-off between warps.  The
// staged rows are 144 and 48 bytes apart, so the 8 rows a fragment load
// touches fall in 8 different bank groups; a lane's word t of block i
// (elements 4t..4t+3 and 16+4t..16+4t+3) is one aligned 32-bit load, and a
// block's fp16 scale one broadcast 32-bit load.
#include "common.cuh"
#include "small_n.cuh"
#include "tma.cuh"

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

namespace qdg {

static __device__ unsigned g_flags_small_n_seg;

namespace {

constexpr int kSegBytes = 1152;      // bytes from one 64-block segment of a row to the next

struct SArgs {
    const uint8_t* W;    // segment layout, O rows of rowbytes
    const uint8_t* xq;   // N Q8_0 vectors of nb blocks, back to back
    float* y;
    int32_t* dbg;
    int64_t ldy;
    int64_t O;
    int64_t rowbytes;
    int nb;          // K / 32
    int N;
    int chunks;      // K / 256
    int csize;       // CTAs per cluster
    int wmax;        // chunk warps per CTA
    int nslots;      // row slots (warps = wmax * nslots)
    int bt;          // row tiles per batch of partial sums (a multiple of nslots)
    int nseg;        // segments per row
    int rlast;       // blocks in the last segment
    int part_floats; // partial-sum area (also receives the activations)
};

// 16-byte asynchronous copy global -> shared (L2 only); src_bytes 0 writes
// zeros and reads nothing.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int kPending>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(kPending) : "memory");
}

// A warp's stage: its chunk's bytes of one 16-row tile, [16 rows][128 nibble
// bytes + 16 pad] then [16 rows][32 scale bytes + 16 pad].  The 144- and
// 48-byte row strides put the 8 rows a fragment load touches in 8 different
// bank groups.
constexpr int kNibStride = 144;
constexpr int kScStride = 48;
constexpr int kWarpStage = kTileRows * (kNibStride + kScStride);   // 3072 bytes
constexpr int kSegStages = 3;                                       // tiles of a warp in flight

// Block kJ of the chunk for rows g, g + 8 of a staged tile, columns 2t, 2t + 1:
// the exact block sums (d0..d3) and acc += d_w d_x isum, as in the
// plain-layout kernel.  hs: 0 or 16, the half of the scale words that holds
// this chunk's scales.
template <int kJ>
__device__ __forceinline__ void staged_block_step(const uint8_t* st, int g, int t, int hs, const XBlock& x,
                                                  const XTab* tab, float (&acc)[4], float (&isum)[4]) {
    const uint32_t w0 = *reinterpret_cast<const uint32_t*>(st + g * kNibStride + 16 * kJ + 4 * t);
    const uint32_t w1 = *reinterpret_cast<const uint32_t*>(st + (g + 8) * kNibStride + 16 * kJ + 4 * t);
    const uint8_t* sc = st + kTileRows * kNibStride;
    const uint32_t dw0 = *reinterpret_cast<const uint32_t*>(sc + g * kScStride + 4 * kJ) >> hs;
    const uint32_t dw1 = *reinterpret_cast<const uint32_t*>(sc + (g + 8) * kScStride + 4 * kJ) >> hs;
    const uint32_t v0 = w0 >> 8, v1 = w1 >> 8;
    const XTab e = tab[kJ * 4 + t];
    float d0, d1, d2, d3;
    hmma2(d0, d1, d2, d3, lo_pair(w0), lo_pair(w1), lo_pair(v0), lo_pair(v1), x.b[0], x.b[1], hi_pair(w0),
          hi_pair(w1), hi_pair(v0), hi_pair(v1), x.b[2], x.b[3]);
    fadd2(d0, d1, e.m0, e.m1);
    fadd2(d2, d3, e.m0, e.m1);
    const float dwa = half_bits_to_float(dw0), dwb = half_bits_to_float(dw1);
    float s0, s1, s2, s3;
    fmul2(s0, s1, dwa, dwa, e.dx0, e.dx1);
    fmul2(s2, s3, dwb, dwb, e.dx0, e.dx1);
    ffma2(acc[0], acc[1], s0, s1, d0, d1);
    ffma2(acc[2], acc[3], s2, s3, d2, d3);
    isum[0] = d0;
    isum[1] = d1;
    isum[2] = d2;
    isum[3] = d3;
}

// Shared memory: [head: activation barrier, abort flag][per-warp tables]
// [per-warp stage rings][partial sums, which first receive the
// activations][cluster partials].
constexpr int kSHeadBytes = 128;
constexpr int kSTabBytes = kMaxWarps * kChunkBlocks * 4 * 16;     // 8 KB
constexpr int kSRingBytes = kMaxWarps * kSegStages * kWarpStage;   // 144 KB
constexpr int kSegBatchTiles = 6;                                  // row tiles per slot and batch of partial sums

template <bool kDebug, bool kCluster>
__global__ void __launch_bounds__(kMaxWarps * 32, 1) small_n_seg_kernel(const __grid_constant__ SArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;
    const int t = lane & 3;
    const int wmax = a.wmax;
    const int nslots = a.nslots;
    const int bt = a.bt;
    uint64_t* xbar = reinterpret_cast<uint64_t*>(smem);
    volatile int* abort_sh = reinterpret_cast<volatile int*>(smem + 8);
    XTab* tab = reinterpret_cast<XTab*>(smem + kSHeadBytes) + warp * kChunkBlocks * 4;   // [8 blocks][4]
    uint8_t* wring = smem + kSHeadBytes + kSTabBytes + warp * kSegStages * kWarpStage;
    float* part = reinterpret_cast<float*>(smem + kSHeadBytes + kSTabBytes + kSRingBytes);   // [bt][wmax][128]
    float* loc = part + a.part_floats;                                                       // [2][bt * 128]

    const int csize = kCluster ? a.csize : 1;
    const int rank = kCluster ? static_cast<int>(cluster_rank()) : 0;
    const int ncl = static_cast<int>(gridDim.x) / csize;
    const int cid = static_cast<int>(blockIdx.x) / csize;
    const int64_t O = a.O;
    const int64_t tiles = (O + kTileRows - 1) / kTileRows;
    const int64_t tile0 = static_cast<int64_t>(cid) * tiles / ncl;
    const int ntiles = static_cast<int>(static_cast<int64_t>(cid + 1) * tiles / ncl - tile0);
    const int nbatch = (ntiles + bt - 1) / bt;

    // this CTA's chunks of K (as in the plain-layout kernel), this warp's
    // chunk and row slot, and where the chunk's bytes sit in a row
    const int ch0 = rank * a.chunks / csize;
    const int cq = (rank + 1) * a.chunks / csize - ch0;
    const int wl = warp % wmax;
    const int slot = warp / wmax;
    const bool worker = wl < cq;
    const int chunk = ch0 + wl;
    const int seg = chunk >> 3;                            // 8 chunks of 8 blocks per segment
    const int i0 = (chunk & 7) * kChunkBlocks;             // first block of the chunk within its segment
    const int rs = seg == a.nseg - 1 ? a.rlast : 64;       // blocks in that segment
    const int64_t nib_off = static_cast<int64_t>(seg) * kSegBytes + 16 * i0;
    const int64_t sc_off = static_cast<int64_t>(seg) * kSegBytes + 16 * rs + 4 * (i0 & 31);
    const int hs = i0 >= 32 ? 16 : 0;

    // The warp's own tiles are tau = slot, slot + nslots, ...; the k-th of
    // them goes to stage k % kSegStages of the warp's ring.  One call: the
    // chunk's 128 nibble bytes of the 16 rows (four 16-byte copies a lane,
    // each warp instruction covering four whole 128-byte row pieces) and its
    // 32 scale bytes (one copy a lane), then one commit.  Rows past O are
    // zero-filled without being read.
    auto issue = [&](int stage, int tau) {
        uint8_t* st = wring + stage * kWarpStage;
        if (tau < ntiles) {
            const int64_t r0 = (tile0 + tau) * kTileRows;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int row = 4 * k + (lane >> 3), piece = lane & 7;
                const bool in = r0 + row < O;
                const uint8_t* src = a.W + (in ? (r0 + row) * a.rowbytes + nib_off + 16 * piece : 0);
                cp_async16(st + row * kNibStride + 16 * piece, src, in ? 16u : 0u);
            }
            {
                const int row = lane >> 1, piece = lane & 1;
                const bool in = r0 + row < O;
                const uint8_t* src = a.W + (in ? (r0 + row) * a.rowbytes + sc_off + 16 * piece : 0);
                cp_async16(st + kTileRows * kNibStride + row * kScStride + 16 * piece, src, in ? 16u : 0u);
            }
        }
        cp_async_commit();   // one group per call, empty or not, so that the wait count is fixed
    };

    if (threadIdx.x == 0) {
        mbar_init(xbar, 1);
        *abort_sh = 0;
        fence_barrier_init();
    }
    __syncthreads();
    pdl_trigger();
    // The weights do not depend on the preceding kernel: the warp's first
    // tiles are requested before the dependency wait.
    if (worker) {
#pragma unroll
        for (int k = 0; k < kSegStages; ++k) issue(k, slot + k * nslots);
    }
    pdl_wait();

    // ---- the CTA's activation blocks (N rows x cq chunks of 272 bytes) land
    // in the partial-sum area with one bulk copy per vector, then each lane
    // builds its fragments from there (as in the plain-layout kernel).
    uint8_t* xsm = reinterpret_cast<uint8_t*>(part);
    const int xrow_sm = wmax * kChunkBlocks * 34 + 16;
    if (threadIdx.x == 0) {
        const uint32_t bytes = static_cast<uint32_t>(cq * kChunkBlocks * 34);
        mbar_arrive_expect_tx(xbar, bytes * static_cast<uint32_t>(a.N));
        for (int n = 0; n < a.N; ++n)
            bulk_g2s_plain(xsm + n * xrow_sm,
                           a.xq + static_cast<int64_t>(n) * a.nb * 34 + static_cast<int64_t>(ch0) * kChunkBlocks * 34,
                           bytes, xbar);
    }
    if (!__all_sync(0xffffffffu, mbar_wait(xbar, 0)) && lane == 0) {
        atomicOr(&g_flags_small_n_seg, FLAG_TIMEOUT);
        *abort_sh = 1;
    }
    uint32_t xlo[kChunkBlocks], xhi[kChunkBlocks], xd[kChunkBlocks];
#pragma unroll
    for (int b = 0; b < kChunkBlocks; ++b) {
        xlo[b] = xhi[b] = xd[b] = 0;
        if (worker && g < a.N) {
            const unsigned short* h =
                reinterpret_cast<const unsigned short*>(xsm + g * xrow_sm + (wl * kChunkBlocks + b) * 34);
            xd[b] = h[0];
            xlo[b] = static_cast<uint32_t>(h[1 + 2 * t]) | (static_cast<uint32_t>(h[2 + 2 * t]) << 16);
            xhi[b] = static_cast<uint32_t>(h[9 + 2 * t]) | (static_cast<uint32_t>(h[10 + 2 * t]) << 16);
        }
    }
    __syncthreads();   // the activation area becomes the partial-sum area
    XBlock xs[kChunkBlocks];
#pragma unroll
    for (int b = 0; b < kChunkBlocks; ++b) {
        const uint32_t lo = xlo[b], hi = xhi[b];
        xs[b].b[0] = act_pair(lo, 0x4240u, false);
        xs[b].b[1] = act_pair(lo, 0x4341u, false);
        xs[b].b[2] = act_pair(hi, 0x4240u, true);
        xs[b].b[3] = act_pair(hi, 0x4341u, true);
        int slo = __dp4a(static_cast<int>(lo), 0x01010101, 0);
        int shi = __dp4a(static_cast<int>(hi), 0x01010101, 0);
        slo += __shfl_xor_sync(0xffffffffu, slo, 1);
        shi += __shfl_xor_sync(0xffffffffu, shi, 1);
        slo += __shfl_xor_sync(0xffffffffu, slo, 2);
        shi += __shfl_xor_sync(0xffffffffu, shi, 2);
        const float mg = static_cast<float>(-1032 * slo - 72 * shi);
        XTab e;
        e.m0 = __shfl_sync(0xffffffffu, mg, 8 * t);
        e.m1 = __shfl_sync(0xffffffffu, mg, 8 * t + 4);
        e.dx0 = half_bits_to_float(__shfl_sync(0xffffffffu, xd[b], 8 * t));
        e.dx1 = half_bits_to_float(__shfl_sync(0xffffffffu, xd[b], 8 * t + 4));
        if (g == 0) tab[b * 4 + t] = e;
    }
    __syncwarp();

    const bool ok = *abort_sh == 0;   // the same in every warp after the barrier above

    int stage = 0;    // the stage of this warp's next tile: its tile count modulo kSegStages
    for (int beta = 0; beta < nbatch; ++beta) {
        for (int j = 0; j < bt / nslots; ++j) {
            const int tb = j * nslots + slot;          // tile within the batch
            const int tau = beta * bt + tb;            // tile within the cluster's rows
            if (tau >= ntiles) break;
            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (worker) {
                cp_async_wait<kSegStages - 1>();       // this lane's copies of the tile have landed
                __syncwarp();                          // and every lane's
                const uint8_t* st = wring + stage * kWarpStage;
                if (ok) {
                    float is[kChunkBlocks][4];
                    staged_block_step<0>(st, g, t, hs, xs[0], tab, acc, is[0]);
                    staged_block_step<1>(st, g, t, hs, xs[1], tab, acc, is[1]);
                    staged_block_step<2>(st, g, t, hs, xs[2], tab, acc, is[2]);
                    staged_block_step<3>(st, g, t, hs, xs[3], tab, acc, is[3]);
                    staged_block_step<4>(st, g, t, hs, xs[4], tab, acc, is[4]);
                    staged_block_step<5>(st, g, t, hs, xs[5], tab, acc, is[5]);
                    staged_block_step<6>(st, g, t, hs, xs[6], tab, acc, is[6]);
                    staged_block_step<7>(st, g, t, hs, xs[7], tab, acc, is[7]);
                    if (kDebug) {
                        const int64_t rt = (tile0 + tau) * kTileRows;
#pragma unroll
                        for (int b = 0; b < kChunkBlocks; ++b)
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int64_t row = rt + g + 8 * (i >> 1);
                                const int col = 2 * t + (i & 1);
                                if (row < O && col < a.N)
                                    a.dbg[(col * O + row) * a.nb + chunk * kChunkBlocks + b] =
                                        static_cast<int32_t>(is[b][i]);
                            }
                    }
                }
                __syncwarp();                          // every lane is done with the stage
                issue(stage, tau + kSegStages * nslots);
                stage = stage + 1 == kSegStages ? 0 : stage + 1;
            }
            if (worker)
                *reinterpret_cast<float4*>(part + (tb * wmax + wl) * 128 + lane * 4) =
                    make_float4(acc[0], acc[1], acc[2], acc[3]);
        }
        __syncthreads();
        // ---- batch reduction.  Index e of a tile's 128 partials = lane * 4 + i
        // of the writing lane: row g + 8 (i >> 1), column 2t + (i & 1).
        const int tiles_here = min(bt, ntiles - beta * bt);
        const int64_t rbase = (tile0 + static_cast<int64_t>(beta) * bt) * kTileRows;
        if (kDebug) {
            __syncthreads();
        } else if (!kCluster) {
            for (int e = threadIdx.x; e < tiles_here * 128; e += blockDim.x) {
                const int tb = e >> 7, l = (e >> 2) & 31, i = e & 3;
                const int col = 2 * (l & 3) + (i & 1);
                const int64_t row = rbase + tb * kTileRows + (l >> 2) + 8 * (i >> 1);
                if (col >= a.N || row >= O) continue;
                const float* src = part + tb * wmax * 128 + (e & 127);
                float v = src[0];
                for (int w = 1; w < cq; ++w) v = __fadd_rn(v, src[w * 128]);
                a.y[col * a.ldy + row] = v;
            }
            __syncthreads();   // partials read before the next batch overwrites them
        } else {
            // clusters imply one slot
            float* lb = loc + (beta & 1) * bt * 128;
            for (int e = threadIdx.x; e < tiles_here * 128; e += blockDim.x) {
                const float* src = part + (e >> 7) * wmax * 128 + (e & 127);
                float v = src[0];
                for (int w = 1; w < cq; ++w) v = __fadd_rn(v, src[w * 128]);
                lb[e] = v;
            }
            __syncwarp();
            cluster_sync();
            const int share = (tiles_here * 128 + csize - 1) / csize;
            const int e0 = rank * share;
            const int e1 = min(tiles_here * 128, e0 + share);
            for (int e = e0 + static_cast<int>(threadIdx.x); e < e1; e += blockDim.x) {
                const int tb = e >> 7, l = (e >> 2) & 31, i = e & 3;
                const int col = 2 * (l & 3) + (i & 1);
                const int64_t row = rbase + tb * kTileRows + (l >> 2) + 8 * (i >> 1);
                if (col >= a.N || row >= O) continue;
                float v = ld_cluster(lb + e, 0);
                for (int q = 1; q < csize; ++q) v = __fadd_rn(v, ld_cluster(lb + e, static_cast<uint32_t>(q)));
                a.y[col * a.ldy + row] = v;
            }
        }
    }
    // Copies still in flight (none unless a warp stopped early) land before
    // the CTA may exit; after a timeout, wait (bounded) for the activation copy.
    cp_async_wait<0>();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_sh != 0) mbar_wait(xbar, 0);
    __syncwarp();
    // No CTA leaves while the others of its cluster may still read its shared memory.
    if (kCluster) cluster_sync();
}

std::mutex g_seg_mutex;
std::map<std::tuple<int, bool, int, int, size_t>, int> g_seg_max_clusters;

size_t seg_smem_bytes(const SArgs& a) {
    return kSHeadBytes + kSTabBytes + kSRingBytes + static_cast<size_t>(a.part_floats) * sizeof(float) +
           (a.csize > 1 ? 2 * static_cast<size_t>(a.bt) * 128 * sizeof(float) : 0);
}

template <bool kDebug, bool kCluster>
int seg_max_clusters(int csize, int warps, size_t smem, int sms) {
    std::lock_guard<std::mutex> lock(g_seg_mutex);
    const DeviceInfo dev = device_info();
    if (dev.device < 0) return -1;
    if (ensure_smem_limit(reinterpret_cast<const void*>(small_n_seg_kernel<kDebug, kCluster>), dev.smem_optin) != cudaSuccess)
        return -1;
    if (!kCluster) return sms;
    // the occupancy answer depends on the device, so the record is kept per device
    const auto key = std::make_tuple(dev.device, kDebug, csize, warps, smem);
    auto it = g_seg_max_clusters.find(key);
    if (it != g_seg_max_clusters.end()) return it->second;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(csize * (sms / csize)));
    cfg.blockDim = dim3(static_cast<unsigned>(warps * 32));
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(csize);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, small_n_seg_kernel<kDebug, kCluster>, &cfg) != cudaSuccess || n < 1)
        return -1;
    g_seg_max_clusters[key] = n;
    return n;
}

template <bool kDebug, bool kCluster>
cudaError_t launch_small_n_seg(const SArgs& a, int warps, size_t smem, int sms, int64_t O, cudaStream_t stream) {
    const int maxcl = seg_max_clusters<kDebug, kCluster>(a.csize, warps, smem, sms);
    if (maxcl < 1) return cudaErrorInvalidConfiguration;
    const int64_t tiles = (O + kTileRows - 1) / kTileRows;
    const int ncl = static_cast<int>(std::min<int64_t>(maxcl, tiles));
    return launch_cluster(small_n_seg_kernel<kDebug, kCluster>, dim3(static_cast<unsigned>(ncl * a.csize)),
                          dim3(static_cast<unsigned>(warps * 32)), smem, stream, !kDebug, kCluster ? a.csize : 1, a);
}

}  // namespace

// N = 3..8 vectors on the segment layout (N = 1, 2 have their own kernels).
int small_n_seg_launch(const void* W, const void* xq, float* y, int64_t ldy, int64_t O, int64_t K, int64_t N,
                       cudaStream_t stream, int32_t* dbg) {
    if (!W || !xq || (!y && !dbg)) return QDG_EINVAL;
    if (O <= 0 || K <= 0 || N < 1 || N > 8) return QDG_EINVAL;
    if (!dbg && ldy < O) return QDG_EINVAL;
    if (K % 256 != 0 || K > 32768 || O >= (int64_t(1) << 31) - kTileRows) return QDG_ESHAPE;
    if (!aligned(W, 16) || !aligned(xq, 16) || (y && !aligned(y, 4))) return QDG_EALIGN;
    const DeviceInfo dev = device_info();
    if (dev.device < 0) return QDG_ECUDA;
    SArgs a;
    a.W = static_cast<const uint8_t*>(W);
    a.xq = static_cast<const uint8_t*>(xq);
    a.y = y;
    a.dbg = dbg;
    a.ldy = ldy;
    a.O = O;
    a.nb = static_cast<int>(K / 32);
    a.nseg = (a.nb + 63) / 64;
    a.rlast = a.nb - 64 * (a.nseg - 1);
    a.rowbytes = static_cast<int64_t>(kSegBytes) * (a.nseg - 1) + 16 * a.rlast + 128;
    a.N = static_cast<int>(N);
    a.chunks = static_cast<int>(K / 256);
    a.csize = (a.chunks + kMaxWarps - 1) / kMaxWarps;
    a.wmax = (a.chunks + a.csize - 1) / a.csize;
    a.nslots = kMaxWarps / a.wmax;
    a.bt = kSegBatchTiles * a.nslots;
    a.part_floats = std::max(a.bt * a.wmax * 128, 8 * (a.wmax * kChunkBlocks * 34 + 16) / 4);
    if (a.csize > kMaxCluster) return QDG_ECUDA;
    if (dev.smem_optin < seg_smem_bytes(a)) return QDG_ECUDA;
    const int warps = a.wmax * a.nslots;
    const size_t smem = seg_smem_bytes(a);
    cudaError_t e;
    if (dbg)
        e = a.csize > 1 ? launch_small_n_seg<true, true>(a, warps, smem, dev.sms, O, stream)
                        : launch_small_n_seg<true, false>(a, warps, smem, dev.sms, O, stream);
    else
        e = a.csize > 1 ? launch_small_n_seg<false, true>(a, warps, smem, dev.sms, O, stream)
                        : launch_small_n_seg<false, false>(a, warps, smem, dev.sms, O, stream);
    if (e != cudaSuccess) return QDG_ECUDA;
    count_launch(2);
    return QDG_OK;
}

unsigned flags_read_clear_small_n_seg(cudaStream_t stream) {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_flags_small_n_seg, sizeof(v), 0, cudaMemcpyDeviceToHost, stream) !=
        cudaSuccess)
        return ~0u;
    if (cudaMemcpyToSymbolAsync(g_flags_small_n_seg, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream) !=
        cudaSuccess)
        return ~0u;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return ~0u;
    return v;
}

}  // namespace qdg
