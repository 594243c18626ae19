// small_n.cuh -- pieces shared by the small-N (N <= 8) products on the plain
// Q4_0 layout (gemm_small_n.cu) and on the segment layout
// (gemm_small_n_seg.cu): the fp16 warp-MMA form of the exact block sums, the
// activation fragments and the cluster helpers.  The arithmetic is described
// at the top of gemm_small_n.cu.
#pragma once
#include "common.cuh"

namespace qdg {
namespace {

constexpr int kMaxWarps = 16;
constexpr int kChunkBlocks = 8;                       // blocks of one row owned by a warp
constexpr int kTileRows = 16;                         // rows of one MMA
constexpr int kMaxCluster = 8;
constexpr uint32_t kLoNib = 0x000F000Fu;
constexpr uint32_t kHiNib = 0x00F000F0u;
constexpr uint32_t kMagic = 0x64006400u;              // fp16 1024.0 in both halves

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Load a float from the shared memory of CTA `rank` of this cluster, at the
// offset that `p` has in this CTA.
__device__ __forceinline__ float ld_cluster(const float* p, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// Bits (0..3, 16..19) -> fp16 pair (1024 + n0, 1024 + n1); bits (4..7, 20..23)
// -> (1024 + 16 n0, 1024 + 16 n1).
__device__ __forceinline__ uint32_t lo_pair(uint32_t v) { return (v & kLoNib) | kMagic; }
__device__ __forceinline__ uint32_t hi_pair(uint32_t v) { return (v & kHiNib) | kMagic; }


// D = A * B (C = 0), m16n8k16, fp16 operands, fp32 accumulation; then D += A2 * B2.
__device__ __forceinline__ void hmma2(float& d0, float& d1, float& d2, float& d3, uint32_t a0, uint32_t a1,
                                      uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1, uint32_t e0, uint32_t e1,
                                      uint32_t e2, uint32_t e3, uint32_t f0, uint32_t f1) {
    asm volatile(
        "{\n\t.reg .f32 z;\n\tmov.f32 z, 0f00000000;\n\t"
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {z,z,z,z};\n\t"
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%10,%11,%12,%13}, {%14,%15}, "
        "{%0,%1,%2,%3};\n\t}"
        : "=&f"(d0), "=&f"(d1), "=&f"(d2), "=&f"(d3)
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "r"(e0), "r"(e1), "r"(e2), "r"(e3), "r"(f0),
          "r"(f1));
}

// (d0, d1) += (b0, b1), packed fp32x2.
__device__ __forceinline__ void fadd2(float& d0, float& d1, float b0, float b1) {
    asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%0, %1};\n\tmov.b64 b, {%2, %3};\n\t"
        "add.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}" : "+f"(d0), "+f"(d1) : "f"(b0), "f"(b1));
}

// Per lane and block, in registers: fp16 activation fragments of column g.
struct XBlock {
    uint32_t b[4];
};
// Per warp, block and t, in shared memory (read as one 16-byte vector): the
// corrections -1032 S_lo - 72 S_hi of columns 2t and 2t + 1, and their
// scales d_x in fp32.
struct XTab {
    float m0, m1;
    float dx0, dx1;
};

// fp16 pairs from the int8 codes of bytes (0, 2) or (1, 3) of v: x, or x / 16.
__device__ __forceinline__ uint32_t act_pair(uint32_t v, uint32_t sel, bool div16) {
    // (x + 128) as the low byte of an fp16 with exponent 2^10: 1152 + x
    const uint32_t h = __byte_perm(v ^ 0x80808080u, 0x64646464u, sel);
    uint32_t r;
    if (div16)   // (1152 + x) / 16 - 72 = x / 16, one rounding of an exact value
        asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(h), "r"(0x2C002C00u), "r"(0xD480D480u));
    else         // (1152 + x) - 1152
        asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0xE480E480u));
    return r;
}

}  // namespace
}  // namespace qdg
