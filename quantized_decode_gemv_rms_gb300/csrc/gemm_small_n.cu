// gemm_small_n.cu -- Q4_0 x Q8_0 product for 1..8 activation vectors that
// share one pass over W (speculative / parallel decode: the "vector case" of
// the quantized matrix-vector route [GGML: Backend abstraction and hardware
// acceleration, section "CUDA: mmvq, mmq, cublas -- three matrix paths"]).
//
// Still bound by the weight stream, but N dot products per weight make the
// integer work N times larger than at N = 1, so the exact per-block sums are
// formed by the warp-level fp16 MMA m16n8k16 (fp32 accumulation): 16 rows x
// 8 columns x 16 elements per instruction.  The integer MMA forms of sm_103a
// issue eight times slower than this one, and dp4a would need 64 operations
// per weight block at N = 8.  The operands hold integers exactly in fp16:
//   * low nibbles n become 1024 + n with one LOP3 ((v & 0x000F000F) |
//     0x64006400); high nibbles stay in place and become 1024 + 16 n
//     ((v & 0x00F000F0) | 0x64006400), so a 32-bit word of 8 nibbles costs
//     one shift and four LOP3s;
//   * the activation codes that meet low nibbles enter as q_x, those that
//     meet high nibbles as q_x / 16 (exact in fp16); every product is then the
//     integer (1024 + n) q_x or (64 + n) q_x, and every partial sum an integer
//     of magnitude below 2^24, exact in fp32;
//   * sum((n - 8) q_x) = D - 1032 S_lo - 72 S_hi, with S_lo, S_hi the sums of
//     the block's first and last 16 activation codes, added in fp32 (exact).
// The order of the 32 elements inside an MMA is free as long as A and B use
// the same one: a lane's 32-bit word t of a Q4_0 block holds elements
// 4t..4t+3 (low nibbles) and 16+4t..16+4t+3 (high nibbles); the first MMA of
// a block takes the low nibbles, the second the high ones, and the lane's
// activation fragments are built in that order once, at kernel start.
//
// Work split: a warp owns a chunk of 8 consecutive blocks of K (256
// elements) and keeps the activation fragments, scales and corrections of
// those blocks for all N columns in registers.  The CTA streams its row
// tiles (32 rows x all of its chunks) through a ring of shared-memory
// stages, one 3-D tensor copy (TMA) per tile that lands each chunk as its own
// 32 x 144-byte slab (row stride 144 bytes: conflict-free fragment loads);
// the last warp done with a stage refills it.  Each warp accumulates
// d_w * d_x * isum in fp32 for its 32 rows x 8 columns (two MMA row groups
// share a tile's waits, refill and partial-sum stores, and each block's
// activation fragments and column table).  A CTA holds up to 16 chunks (K <= 4096); for
// larger K a thread-block cluster of ceil(K / 4096) CTAs splits K, and the
// per-chunk partials are combined in a fixed order: first across the CTA's
// warps in shared memory, then across the cluster's CTAs through distributed
// shared memory.  No workspace, no atomics: results are deterministic.
// Every wait is bounded; a timeout sets a flag, the warp stops computing,
// waits for its copies in flight and leaves with the others.
#include "common.cuh"
#include "small_n.cuh"
#include "tma.cuh"

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

namespace qdg {

static __device__ unsigned g_flags_small_n;

namespace {

constexpr int kChunkBytes = kChunkBlocks * 18;        // 144 bytes of a row per chunk, a multiple of 16
constexpr int kRows = 2 * kTileRows;                  // rows of a tile: two MMA row groups share its bookkeeping
constexpr int kUnitBytes = kRows * kChunkBytes;       // 4608 bytes per ring slot (36 x 128)
constexpr int kPartTile = kRows * 8;                  // partial sums of one tile and warp: 32 rows x 8 columns
constexpr int kBatchTilesPerSlot = 4;                 // row tiles per slot and batch of partial sums

static_assert(kChunkBytes % 16 == 0 && kUnitBytes % 128 == 0, "tensor-copy alignment");

// Word t of the nibbles of block b in a staged row (row start 16-byte aligned):
// the block starts at 18b, its nibbles at 18b + 2, so the word is 4-byte
// aligned for odd b and straddles two aligned words for even b.
template <int kB>
__device__ __forceinline__ uint32_t nibble_word(const uint8_t* row, int t) {
    if (kB & 1) return *reinterpret_cast<const uint32_t*>(row + 18 * kB + 2 + 4 * t);
    const uint32_t* p = reinterpret_cast<const uint32_t*>(row + 18 * kB + 4 * t);
    return bytes_2_to_5(p[0], p[1]);
}

struct Args {
    CUtensorMap wmap;   // W as [chunk][row][144 bytes]; box = 32 rows x wmax chunks
    const uint8_t* xq;
    float* y;
    int32_t* dbg;
    int64_t ldy;
    int64_t O;
    int nb;        // K / 32
    int N;
    int chunks;    // K / 256
    int csize;     // CTAs per cluster
    int wmax;      // chunk warps per CTA (largest share of the cluster's CTAs)
    int nslots;    // row tiles in flight per CTA (warps = wmax * nslots)
    int bt;        // row tiles per batch of partial sums (a multiple of nslots)
    int stages;    // tile stages in the ring
    int part_floats;   // partial-sum area: bt * wmax * 128 floats, and room for the staged activations
};

// One block of the warp's chunk for the tile's 32 rows: rows g, g + 8 (ra, rb)
// and g + 16, g + 24 (rc, rd), each pair one m16 MMA row group; the
// activation fragments and the column table serve both.
template <int kB>
__device__ __forceinline__ void block_step(const uint8_t* ra, const uint8_t* rb, const uint8_t* rc, const uint8_t* rd,
                                           int t, const XBlock& x, const XTab* tab, float (&acc)[8],
                                           float (&isum)[8]) {
    const XTab e = tab[kB * 4 + t];
    const uint8_t* rows[4] = {ra, rb, rc, rd};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t w0 = nibble_word<kB>(rows[2 * h], t);
        const uint32_t w1 = nibble_word<kB>(rows[2 * h + 1], t);
        const uint32_t v0 = w0 >> 8, v1 = w1 >> 8;
        const unsigned short dw0 = *reinterpret_cast<const unsigned short*>(rows[2 * h] + 18 * kB);
        const unsigned short dw1 = *reinterpret_cast<const unsigned short*>(rows[2 * h + 1] + 18 * kB);
        float d0, d1, d2, d3;
        // first MMA: low nibbles of bytes (0, 2) and (1, 3), rows g and g + 8
        // of the group; second MMA: high nibbles of the same bytes (x 16),
        // activations / 16; plus the columns' corrections: d = the exact
        // block sums of columns 2t, 2t + 1 for the two rows
        hmma2(d0, d1, d2, d3, lo_pair(w0), lo_pair(w1), lo_pair(v0), lo_pair(v1), x.b[0], x.b[1], hi_pair(w0),
              hi_pair(w1), hi_pair(v0), hi_pair(v1), x.b[2], x.b[3]);
        // acc += (d_w * d_x) * isum; the scale product is exact in fp32
        fadd2(d0, d1, e.m0, e.m1);
        fadd2(d2, d3, e.m0, e.m1);
        const float dwa = half_bits_to_float(dw0), dwb = half_bits_to_float(dw1);
        float s0, s1, s2, s3;
        fmul2(s0, s1, dwa, dwa, e.dx0, e.dx1);
        fmul2(s2, s3, dwb, dwb, e.dx0, e.dx1);
        ffma2(acc[4 * h], acc[4 * h + 1], s0, s1, d0, d1);
        ffma2(acc[4 * h + 2], acc[4 * h + 3], s2, s3, d2, d3);
        isum[4 * h] = d0;
        isum[4 * h + 1] = d1;
        isum[4 * h + 2] = d2;
        isum[4 * h + 3] = d3;
    }
}

// Shared memory: [mbarriers][counters][pad], the per-warp tables, then the
// stage ring, the batch partials and (cluster case) the per-CTA partials.
constexpr int kMaxStages = 32;
constexpr int kHeadBytes = 512;
constexpr int kTabBytes = kMaxWarps * kChunkBlocks * 4 * 16;   // 8 KB

template <bool kDebug, bool kCluster>
__global__ void __launch_bounds__(kMaxWarps * 32, 1) small_n_kernel(const __grid_constant__ Args a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;
    const int t = lane & 3;
    const int wmax = a.wmax;
    const int nslots = a.nslots;
    const int bt = a.bt;
    const int S = a.stages;
    const int stage_bytes = wmax * kUnitBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);                     // [S]
    int* cnt = reinterpret_cast<int*>(smem + kMaxStages * sizeof(uint64_t)); // [S] consumer arrivals
    int* issued_sh = cnt + kMaxStages;                                       // tiles issued so far
    volatile int* abort_sh = issued_sh + 1;                                  // a wait gave up
    uint64_t* xbar = full + kMaxStages - 1;                                  // activation copies (S < kMaxStages)
    XTab* tab = reinterpret_cast<XTab*>(smem + kHeadBytes) + warp * kChunkBlocks * 4;   // [8 blocks][4]
    uint8_t* ring = smem + kHeadBytes + kTabBytes;
    float* part = reinterpret_cast<float*>(ring + S * stage_bytes);          // [bt][wmax][kPartTile]
    float* loc = part + a.part_floats;                                       // [2][bt * kPartTile], cluster case

    const int csize = kCluster ? a.csize : 1;
    const int rank = kCluster ? static_cast<int>(cluster_rank()) : 0;
    const int ncl = static_cast<int>(gridDim.x) / csize;
    const int cid = static_cast<int>(blockIdx.x) / csize;
    const int64_t O = a.O;
    // the cluster's row tiles [tile0, tile0 + ntiles); rows past O read as zero
    const int64_t tiles = (O + kRows - 1) / kRows;
    const int64_t tile0 = static_cast<int64_t>(cid) * tiles / ncl;
    const int ntiles = static_cast<int>(static_cast<int64_t>(cid + 1) * tiles / ncl - tile0);
    const int nbatch = (ntiles + bt - 1) / bt;

    // this CTA's chunks of K, and this warp's chunk and row slot
    const int ch0 = rank * a.chunks / csize;
    const int cq = (rank + 1) * a.chunks / csize - ch0;
    const int wl = warp % wmax;
    const int slot = warp / wmax;
    const bool worker = wl < cq;
    const int chunk = ch0 + wl;

    // Tile tau of the cluster's rows goes to stage s = tau % S; one tensor copy
    // brings the 32 rows x wmax chunks of the CTA (chunk slabs of 32 x 144 B).
    auto issue = [&](int s, int tau) {
        mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(stage_bytes));
        tma_load_3d(ring + s * stage_bytes, &a.wmap, 0, static_cast<int>((tile0 + tau) * kRows), ch0, &full[s]);
    };
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            cnt[i] = 0;
        }
        mbar_init(xbar, 1);
        *abort_sh = 0;
        fence_barrier_init();
    }
    __syncthreads();
    pdl_trigger();
    const int n0 = ntiles < S ? ntiles : S;
    pdl_wait();

    // ---- the CTA's activation blocks (N rows x cq chunks of 272 bytes) land
    // in the partial-sum area (sized for 8 rows) with one bulk copy per row,
    // issued before the weight tiles so that they do not queue behind them;
    // then each lane builds its fragments from there.
    uint8_t* xsm = reinterpret_cast<uint8_t*>(part);   // [N][wmax * 272 + 16]
    const int xrow_sm = wmax * kChunkBlocks * 34 + 16;  // padded: the 8 rows of a quad's loads hit 8 banks
    if (threadIdx.x == 0) {
        const uint32_t bytes = static_cast<uint32_t>(cq * kChunkBlocks * 34);
        mbar_arrive_expect_tx(xbar, bytes * static_cast<uint32_t>(a.N));
        for (int n = 0; n < a.N; ++n)
            bulk_g2s_plain(xsm + n * xrow_sm,
                           a.xq + static_cast<int64_t>(n) * a.nb * 34 + static_cast<int64_t>(ch0) * kChunkBlocks * 34,
                           bytes, xbar);
        for (int tau = 0; tau < n0; ++tau) issue(tau, tau);
        *issued_sh = n0;
    }
    if (!__all_sync(0xffffffffu, mbar_wait(xbar, 0)) && lane == 0) {
        atomicOr(&g_flags_small_n, FLAG_TIMEOUT);
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
        xs[b].b[0] = act_pair(lo, 0x4240u, false);   // elements 4t, 4t + 2
        xs[b].b[1] = act_pair(lo, 0x4341u, false);   // elements 4t + 1, 4t + 3
        xs[b].b[2] = act_pair(hi, 0x4240u, true);    // elements 16 + 4t, 16 + 4t + 2, divided by 16
        xs[b].b[3] = act_pair(hi, 0x4341u, true);
        int slo = __dp4a(static_cast<int>(lo), 0x01010101, 0);
        int shi = __dp4a(static_cast<int>(hi), 0x01010101, 0);
        slo += __shfl_xor_sync(0xffffffffu, slo, 1);
        shi += __shfl_xor_sync(0xffffffffu, shi, 1);
        slo += __shfl_xor_sync(0xffffffffu, slo, 2);
        shi += __shfl_xor_sync(0xffffffffu, shi, 2);
        const float mg = static_cast<float>(-1032 * slo - 72 * shi);   // of column g, exact
        XTab e;
        e.m0 = __shfl_sync(0xffffffffu, mg, 8 * t);
        e.m1 = __shfl_sync(0xffffffffu, mg, 8 * t + 4);
        e.dx0 = half_bits_to_float(__shfl_sync(0xffffffffu, xd[b], 8 * t));
        e.dx1 = half_bits_to_float(__shfl_sync(0xffffffffu, xd[b], 8 * t + 4));
        if (g == 0) tab[b * 4 + t] = e;
    }
    __syncwarp();

    bool ok = true;   // false once a wait gave up: stop computing, keep the barrier schedule
    int s = slot;     // stage of this warp's next tile, tau % S (slot < nslots <= S)
    uint32_t ph = 0;  // and its phase parity, (tau / S) & 1
    for (int beta = 0; beta < nbatch; ++beta) {
        for (int j = 0; j < bt / nslots; ++j) {
            const int tb = j * nslots + slot;          // tile within the batch
            const int tau = beta * bt + tb;            // tile within the cluster's rows
            if (tau >= ntiles) break;
            float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
            if (worker && ok) {
                ok = *abort_sh == 0 && __all_sync(0xffffffffu, mbar_wait(&full[s], ph));
                if (!ok && lane == 0) {
                    atomicOr(&g_flags_small_n, FLAG_TIMEOUT);
                    *abort_sh = 1;
                }
            }
            if (worker && ok) {
                const uint8_t* ra = ring + s * stage_bytes + wl * kUnitBytes + g * kChunkBytes;
                const uint8_t* rb = ra + 8 * kChunkBytes;
                const uint8_t* rc = ra + 16 * kChunkBytes;
                const uint8_t* rd = ra + 24 * kChunkBytes;
                float is[kChunkBlocks][8];
                block_step<0>(ra, rb, rc, rd, t, xs[0], tab, acc, is[0]);
                block_step<1>(ra, rb, rc, rd, t, xs[1], tab, acc, is[1]);
                block_step<2>(ra, rb, rc, rd, t, xs[2], tab, acc, is[2]);
                block_step<3>(ra, rb, rc, rd, t, xs[3], tab, acc, is[3]);
                block_step<4>(ra, rb, rc, rd, t, xs[4], tab, acc, is[4]);
                block_step<5>(ra, rb, rc, rd, t, xs[5], tab, acc, is[5]);
                block_step<6>(ra, rb, rc, rd, t, xs[6], tab, acc, is[6]);
                block_step<7>(ra, rb, rc, rd, t, xs[7], tab, acc, is[7]);
                if (kDebug) {
                    const int64_t rt = (tile0 + tau) * kRows;
#pragma unroll
                    for (int b = 0; b < kChunkBlocks; ++b)
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int64_t row = rt + g + 8 * (i >> 1);
                            const int col = 2 * t + (i & 1);
                            if (row < O && col < a.N)
                                a.dbg[(col * O + row) * a.nb + chunk * kChunkBlocks + b] = static_cast<int32_t>(is[b][i]);
                        }
                }
                // The warp is done with its slab of the stage: every value read
                // from it was consumed by the MMAs above.  The last of the
                // CTA's cq warps refills the stage with tile tau + S.
                __syncwarp();
                if (lane == 0 && atomicAdd(&cnt[s], 1) == cq - 1) {
                    cnt[s] = 0;
                    if (tau + S < ntiles && *abort_sh == 0) {
                        issue(s, tau + S);
                        atomicMax(issued_sh, tau + S + 1);
                    }
                }
                __syncwarp();
            }
            if (worker) {
                float4* dst = reinterpret_cast<float4*>(part + (tb * wmax + wl) * kPartTile + lane * 8);
                dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
                dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
            }
            s += nslots;
            if (s >= S) {
                s -= S;
                ph ^= 1u;
            }
        }
        __syncthreads();
        // ---- batch reduction.  Index e of a tile's 256 partials = lane * 8 + i
        // of the writing lane: row g + 8 (i >> 1), column 2t + (i & 1).
        const int tiles_here = min(bt, ntiles - beta * bt);
        const int64_t rbase = (tile0 + static_cast<int64_t>(beta) * bt) * kRows;
        if (kDebug) {
            __syncthreads();
        } else if (!kCluster) {
            for (int e = threadIdx.x; e < tiles_here * kPartTile; e += blockDim.x) {
                const int tb = e >> 8, l = (e >> 3) & 31, i = e & 7;
                const int col = 2 * (l & 3) + (i & 1);
                const int64_t row = rbase + tb * kRows + (l >> 2) + 8 * (i >> 1);
                if (col >= a.N || row >= O) continue;
                const float* src = part + tb * wmax * kPartTile + (e & 255);
                float v = src[0];
                for (int w = 1; w < cq; ++w) v = __fadd_rn(v, src[w * kPartTile]);
                a.y[col * a.ldy + row] = v;
            }
            __syncthreads();   // partials read before the next batch overwrites them
        } else {
            // clusters imply one slot
            float* lb = loc + (beta & 1) * bt * kPartTile;
            for (int e = threadIdx.x; e < tiles_here * kPartTile; e += blockDim.x) {
                const float* src = part + (e >> 8) * wmax * kPartTile + (e & 255);
                float v = src[0];
                for (int w = 1; w < cq; ++w) v = __fadd_rn(v, src[w * kPartTile]);
                lb[e] = v;
            }
            __syncwarp();
            cluster_sync();
            const int per = (tiles_here * kPartTile + csize - 1) / csize;
            const int e0 = rank * per;
            const int e1 = min(tiles_here * kPartTile, e0 + per);
            for (int e = e0 + static_cast<int>(threadIdx.x); e < e1; e += blockDim.x) {
                const int tb = e >> 8, l = (e >> 3) & 31, i = e & 7;
                const int col = 2 * (l & 3) + (i & 1);
                const int64_t row = rbase + tb * kRows + (l >> 2) + 8 * (i >> 1);
                if (col >= a.N || row >= O) continue;
                float v = ld_cluster(lb + e, 0);
                for (int q = 1; q < csize; ++q) v = __fadd_rn(v, ld_cluster(lb + e, static_cast<uint32_t>(q)));
                a.y[col * a.ldy + row] = v;
            }
        }
    }
    // After a timeout: wait (bounded) for the copies of the last S tiles issued.
    __syncthreads();
    if (threadIdx.x == 0 && *abort_sh != 0) {
        mbar_wait(xbar, 0);
        const int n = *reinterpret_cast<volatile int*>(issued_sh);
        for (int tau = (n - S > 0 ? n - S : 0); tau < n; ++tau) mbar_wait(&full[tau % S], (tau / S) & 1);
    }
    __syncwarp();
    // No CTA leaves while the others of its cluster may still read its shared memory.
    if (kCluster) cluster_sync();
}

std::mutex g_mutex;
std::map<std::tuple<int, bool, int, int, size_t>, int> g_max_clusters;

size_t smem_bytes(const Args& a) {
    const size_t stage = static_cast<size_t>(a.wmax) * kUnitBytes;
    return kHeadBytes + kTabBytes + a.stages * stage + static_cast<size_t>(a.part_floats) * sizeof(float) +
           (a.csize > 1 ? 2 * static_cast<size_t>(a.bt) * kPartTile * sizeof(float) : 0);
}

template <bool kDebug, bool kCluster>
int max_clusters(int csize, int warps, size_t smem, int sms) {
    std::lock_guard<std::mutex> lock(g_mutex);
    const DeviceInfo dev = device_info();
    if (dev.device < 0) return -1;
    if (ensure_smem_limit(reinterpret_cast<const void*>(small_n_kernel<kDebug, kCluster>), dev.smem_optin) != cudaSuccess)
        return -1;
    if (!kCluster) return sms;
    // the occupancy answer depends on the device, so the record is kept per device
    const auto key = std::make_tuple(dev.device, kDebug, csize, warps, smem);
    auto it = g_max_clusters.find(key);
    if (it != g_max_clusters.end()) return it->second;
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
    if (cudaOccupancyMaxActiveClusters(&n, small_n_kernel<kDebug, kCluster>, &cfg) != cudaSuccess || n < 1)
        return -1;
    g_max_clusters[key] = n;
    return n;
}

template <bool kDebug, bool kCluster>
cudaError_t launch_small_n(const Args& a, int warps, size_t smem, int sms, int64_t O, cudaStream_t stream) {
    const int maxcl = max_clusters<kDebug, kCluster>(a.csize, warps, smem, sms);
    if (maxcl < 1) return cudaErrorInvalidConfiguration;
    const int64_t tiles = (O + kRows - 1) / kRows;
    const int ncl = static_cast<int>(std::min<int64_t>(maxcl, tiles));
    return launch_cluster(small_n_kernel<kDebug, kCluster>, dim3(static_cast<unsigned>(ncl * a.csize)),
                          dim3(static_cast<unsigned>(warps * 32)), smem, stream, !kDebug, kCluster ? a.csize : 1, a);
}

}  // namespace

int small_n_launch(const void* W, const void* xq, float* y, int64_t ldy, int64_t O, int64_t K, int64_t N,
                   cudaStream_t stream, int32_t* dbg) {
    if (!W || !xq || (!y && !dbg)) return QDG_EINVAL;
    if (O <= 0 || K <= 0 || N < 1 || N > 8) return QDG_EINVAL;
    if (!dbg && ldy < O) return QDG_EINVAL;
    if (K % 256 != 0 || K > 32768 || O >= (int64_t(1) << 31) - kRows) return QDG_ESHAPE;
    if (!aligned(W, 16) || !aligned(xq, 16) || (y && !aligned(y, 4))) return QDG_EALIGN;
    const DeviceInfo dev = device_info();
    if (dev.device < 0) return QDG_ECUDA;
    Args a;
    a.xq = static_cast<const uint8_t*>(xq);
    a.y = y;
    a.dbg = dbg;
    a.ldy = ldy;
    a.O = O;
    a.nb = static_cast<int>(K / 32);
    a.N = static_cast<int>(N);
    a.chunks = static_cast<int>(K / 256);
    a.csize = (a.chunks + kMaxWarps - 1) / kMaxWarps;
    a.wmax = (a.chunks + a.csize - 1) / a.csize;
    a.nslots = kMaxWarps / a.wmax;
    // kBatchTilesPerSlot row tiles per slot and batch of partial sums; the rest of shared
    // memory holds as many tile stages as fit (at least two).
    a.bt = kBatchTilesPerSlot * a.nslots;
    // the partial-sum area first receives the activations: N x wmax chunks x 272 bytes
    a.part_floats = std::max(a.bt * a.wmax * kPartTile, 8 * (a.wmax * kChunkBlocks * 34 + 16) / 4);
    if (a.csize > kMaxCluster) return QDG_ECUDA;
    a.stages = 0;
    const size_t fixed = smem_bytes(a);
    const size_t stage = static_cast<size_t>(a.wmax) * kUnitBytes;
    if (dev.smem_optin < fixed + 2 * stage) return QDG_ECUDA;
    a.stages = static_cast<int>(std::min<size_t>(kMaxStages - 1, (dev.smem_optin - fixed) / stage));
    const int warps = a.wmax * a.nslots;
    const size_t smem = smem_bytes(a);
    if (!encode_row_segments(&a.wmap, W, static_cast<int64_t>(a.nb) * 18, O, kChunkBytes, kRows, a.wmax))
        return QDG_ECUDA;
    cudaError_t e;
    if (dbg)
        e = a.csize > 1 ? launch_small_n<true, true>(a, warps, smem, dev.sms, O, stream)
                        : launch_small_n<true, false>(a, warps, smem, dev.sms, O, stream);
    else
        e = a.csize > 1 ? launch_small_n<false, true>(a, warps, smem, dev.sms, O, stream)
                        : launch_small_n<false, false>(a, warps, smem, dev.sms, O, stream);
    if (e != cudaSuccess) return QDG_ECUDA;
    count_launch(2);
    return QDG_OK;
}

unsigned flags_read_clear_small_n(cudaStream_t stream) {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_flags_small_n, sizeof(v), 0, cudaMemcpyDeviceToHost, stream) !=
        cudaSuccess)
        return ~0u;
    if (cudaMemcpyToSymbolAsync(g_flags_small_n, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream) !=
        cudaSuccess)
        return ~0u;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return ~0u;
    return v;
}

}  // namespace qdg

extern "C" int q4_0_q8_0_gemm_small_n(const void* W, const void* xq, float* y, int64_t ldy, int64_t O, int64_t K,
                                      int64_t N, qdg_stream_t stream) {
    if (!y) return QDG_EINVAL;
    return qdg::small_n_launch(W, xq, y, ldy, O, K, N, reinterpret_cast<cudaStream_t>(stream), nullptr);
}
