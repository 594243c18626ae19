// quantize.cu -- the fused RMS_NORM + MUL(gamma) [+ ADD] -> Q8_0 activation
// kernel and the load-time fp32 -> Q4_0 weight quantizer.
//
// RMS_NORM followed by MUL is the pattern whose fusion the Metal backend
// lost, costing about 5% of token-generation speed [llama.cpp b10909: Metal
// backend fusion-table refactor, introduction]; here the two ops and the Q8_0
// quantization the Q4 x Q8 products need [GGML: Backend abstraction and
// hardware acceleration, section "Metal and Vulkan"] are a single pass.
// Epsilon is added to the mean square, inside the square root [llama.cpp
// b10981, section "NPU cacheless encoder models and norm optimisation"].
#include "common.cuh"

namespace qdg {

static __device__ unsigned g_flags_quantize;

namespace {

constexpr int kNormThreads = 256;     // the fixed reduction order is defined over 256 lanes
// Q8_0 blocks quantized by one CTA: one per warp.  A block is a dependent
// chain of about 380 SM cycles (the five-step maximum alone about 135,
// measured on GB300), so a warp with four blocks spent about 1.5 us on a
// decode-step boundary; more CTAs with one block a warp cut that to one chain.
constexpr int kBlocksPerCta = 8;
constexpr int kStageMax = 8192;       // vectors up to this length are read for the norm in one wave of loads
constexpr int kStagePer = kStageMax / 4 / kNormThreads;   // 16-byte loads per thread in that wave

// Grid: (vectors * splits).  Every CTA of a vector recomputes the vector's
// sum of squares in the library's fixed order (so all CTAs agree bit for
// bit), then quantizes its own slice of kBlocksPerCta blocks.
//   Sum of squares: thread j sums x_i^2 for i = j (mod 256) with an fma chain
//   in ascending i; each warp combines with an xor butterfly (16,8,4,2,1);
//   the 8 warp totals combine as ((w0+w1)+(w2+w3))+((w4+w5)+(w6+w7)).  A
//   16-byte aligned vector of up to kStageMax elements is first read whole,
//   in one wave of 16-byte loads, into shared memory (the chains are the same).
//   Quantization: warp w takes blocks w, w+8, ... of the slice, lane l
//   element 32b+l.
//   add (optional): v = (x*s)*gamma + a, one fp32 addition after the MUL
//   (the RMS_NORM+MUL+ADD pattern), a = add + n*ldadd (ldadd 0: broadcast).
__global__ void __launch_bounds__(kNormThreads)
qnorm_q8_kernel(const float* __restrict__ x, int64_t ldx, const float* __restrict__ gamma,
                const float* __restrict__ add, int64_t ldadd, float eps, int K, int splits,
                uint8_t* __restrict__ xq) {
    // Let the next kernel (the product that reads xq) launch at once: it only
    // touches its weights before its own dependency wait, so its CTAs take
    // their SMs as the previous product's CTAs leave and stream weights while
    // this kernel waits and quantizes.  Measured on GB300, triggering here
    // instead of after the statistic took the 8B-shaped decode step from 86.2
    // to 80.5 us and the 1B-shaped step from 19.3 to 16.4 us (per-CTA timer
    // stamps: the product's CTAs started 0.5 us after this kernel ended, and
    // the memory system idled through each boundary).
    pdl_trigger();
    pdl_wait();
    const int64_t n = blockIdx.x / splits;
    const int split = blockIdx.x - static_cast<int>(n * splits);
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const float* xn = x + n * ldx;
    const float* an = add != nullptr ? add + n * ldadd : nullptr;
    const int nb = K >> 5;
    const int b0 = split * kBlocksPerCta;
    const int b1 = min(nb, b0 + kBlocksPerCta);

    // Issue this CTA's slice loads first; they overlap the reduction below.
    constexpr int kPer = kBlocksPerCta / (kNormThreads / 32);
    float xv[kPer], gv[kPer], av[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int b = b0 + warp + u * (kNormThreads / 32);
        xv[u] = b < b1 ? __ldg(xn + (b << 5) + lane) : 0.0f;
        gv[u] = (gamma != nullptr && b < b1) ? __ldg(gamma + (b << 5) + lane) : 1.0f;
        av[u] = (an != nullptr && b < b1) ? __ldg(an + (b << 5) + lane) : 0.0f;
    }

    float s = 1.0f;
    if (gamma != nullptr) {
        __shared__ float wsum[kNormThreads / 32];
        __shared__ __align__(16) float xs[kStageMax];
        float acc = 0.0f;
        if (K <= kStageMax && (reinterpret_cast<uintptr_t>(xn) & 15) == 0) {
            // the whole vector in one wave of 16-byte loads (one memory round
            // trip), staged in shared memory; then each chain in order
            const int k4 = K >> 2;
            float4 t[kStagePer];
#pragma unroll
            for (int u = 0; u < kStagePer; ++u) {
                const int i = tid + u * kNormThreads;
                if (i < k4) t[u] = __ldg(reinterpret_cast<const float4*>(xn) + i);
            }
#pragma unroll
            for (int u = 0; u < kStagePer; ++u) {
                const int i = tid + u * kNormThreads;
                if (i < k4) reinterpret_cast<float4*>(xs)[i] = t[u];
            }
            __syncthreads();
            for (int i = tid; i < K; i += kNormThreads) acc = __fmaf_rn(xs[i], xs[i], acc);
        } else {
            for (int i0 = tid; i0 < K; i0 += kNormThreads * 8) {
                float v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int i = i0 + u * kNormThreads;
                    v[u] = i < K ? __ldg(xn + i) : 0.0f;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (i0 + u * kNormThreads < K) acc = __fmaf_rn(v[u], v[u], acc);
            }
        }
        acc = warp_sum(acc);
        if (lane == 0) wsum[warp] = acc;
        __syncthreads();
        const float ss = __fadd_rn(__fadd_rn(__fadd_rn(wsum[0], wsum[1]), __fadd_rn(wsum[2], wsum[3])),
                                   __fadd_rn(__fadd_rn(wsum[4], wsum[5]), __fadd_rn(wsum[6], wsum[7])));
        const float mean = __fdiv_rn(ss, static_cast<float>(K));
        s = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
    }

    uint8_t* out = xq + n * nb * 34;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int b = b0 + warp + u * (kNormThreads / 32);
        if (b >= b1) break;
        float v = xv[u];
        if (gamma != nullptr) v = __fmul_rn(__fmul_rn(v, s), gv[u]);
        if (an != nullptr) v = __fadd_rn(v, av[u]);
        float amax = fabsf(v);
#pragma unroll
        for (int h = 16; h >= 1; h >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, h));
        const float d = __fdiv_rn(amax, 127.0f);
        int q = 0;
        if (d != 0.0f) {
            float r = roundf(__fdiv_rn(v, d));
            r = fminf(fmaxf(r, -127.0f), 127.0f);
            q = static_cast<int>(r);
        }
        uint8_t* blk = out + static_cast<int64_t>(b) * 34;
        if (lane == 0) {
            const __half dh = __float2half_rn(d);
            *reinterpret_cast<unsigned short*>(blk) = __half_as_ushort(dh);
            if (__hisinf(dh)) atomicOr(&g_flags_quantize, FLAG_OVERFLOW);
        }
        blk[2 + lane] = static_cast<uint8_t>(static_cast<int8_t>(q));
    }
}

// One thread per Q4_0 block.
__global__ void quantize_q4_0_kernel(const float* __restrict__ w, int64_t ldw, int64_t O, int K,
                                     uint8_t* __restrict__ Wq) {
    const int nb = K >> 5;
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= O * nb) return;
    const int64_t row = idx / nb;
    const int b = static_cast<int>(idx - row * nb);
    const float* v = w + row * ldw + (b << 5);
    float vals[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) vals[j] = __ldg(v + j);
    float amax = 0.0f, m = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        if (fabsf(vals[j]) > amax) {
            amax = fabsf(vals[j]);
            m = vals[j];
        }
    }
    const float d = __fdiv_rn(m, -8.0f);
    int q[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        if (d == 0.0f) {
            q[j] = 8;
        } else {
            const float t = __fadd_rn(__fdiv_rn(vals[j], d), 8.5f);
            const int qi = static_cast<int>(t);
            q[j] = qi > 15 ? 15 : (qi < 0 ? 0 : qi);
        }
    }
    unsigned short* dst = reinterpret_cast<unsigned short*>(Wq + idx * 18);
    dst[0] = __half_as_ushort(__float2half_rn(d));
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
        const unsigned lo = static_cast<unsigned>(q[j] | (q[j + 16] << 4));
        const unsigned hi = static_cast<unsigned>(q[j + 1] | (q[j + 17] << 4));
        dst[1 + j / 2] = static_cast<unsigned short>(lo | (hi << 8));
    }
}

// Q4_K weight quantization, one thread per 256-weight super-block (load
// time, not the decode path).  The library's plain reading of the k-quant
// recipe, every step one IEEE fp32 operation in this order:
//   sub-block j: lo, hi = min, max of its 32 weights; mn_j = -lo if lo < 0
//   else 0; a_j = (hi + mn_j) / 15;  D = max_j a_j / 63, Dm = max_j mn_j / 63,
//   stored d = fp16(D), dmin = fp16(Dm) (nearest even), dd, ddm their values;
//   sc_j = round(a_j / dd), m_j = round(mn_j / ddm) (halves away from zero,
//   0 when the divisor is 0), clamped to 0..63;  q = round((w + ddm m_j) /
//   (dd sc_j)) clamped to 0..15, 0 when dd sc_j is 0.
// Layout of the 144 bytes: d, dmin, twelve scale bytes (j < 4: s[j] = sc_j
// plus the top two bits of sc_{j+4} in bits 6-7, s[j+4] = m_j plus those of
// m_{j+4}; s[j+8] = low nibbles of sc_{j+4} and m_{j+4}), then code byte
// 16 + 32p + i = element i of sub-block 2p (low nibble) and 2p+1 (high).
__device__ __forceinline__ int round_clamp(float v, int hi) {
    const int q = static_cast<int>(roundf(v));
    return q < 0 ? 0 : (q > hi ? hi : q);
}

__global__ void quantize_q4_k_kernel(const float* __restrict__ w, int64_t ldw, int64_t O, int K,
                                     uint8_t* __restrict__ Wq) {
    const int nsb = K >> 8;
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= O * nsb) return;
    const int64_t row = idx / nsb;
    const int sbi = static_cast<int>(idx - row * nsb);
    const float* v = w + row * ldw + (static_cast<int64_t>(sbi) << 8);
    float a[8], mn[8], amax = 0.0f, mnmax = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float lo = __ldg(v + 32 * j), hi = lo;
        for (int i = 1; i < 32; ++i) {
            const float t = __ldg(v + 32 * j + i);
            if (t < lo) lo = t;
            if (t > hi) hi = t;
        }
        mn[j] = lo < 0.0f ? -lo : 0.0f;
        a[j] = __fdiv_rn(__fadd_rn(hi, mn[j]), 15.0f);
        if (a[j] > amax) amax = a[j];
        if (mn[j] > mnmax) mnmax = mn[j];
    }
    const __half dh = __float2half_rn(__fdiv_rn(amax, 63.0f));
    const __half dmh = __float2half_rn(__fdiv_rn(mnmax, 63.0f));
    const float dd = __half2float(dh), ddm = __half2float(dmh);
    int sc[8], m[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        sc[j] = dd > 0.0f ? round_clamp(__fdiv_rn(a[j], dd), 63) : 0;
        m[j] = ddm > 0.0f ? round_clamp(__fdiv_rn(mn[j], ddm), 63) : 0;
    }
    uint32_t out[36];
    out[0] = static_cast<uint32_t>(__half_as_ushort(dh)) | (static_cast<uint32_t>(__half_as_ushort(dmh)) << 16);
    uint8_t s[12];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        s[j] = static_cast<uint8_t>((sc[j] & 63) | ((sc[j + 4] >> 4) << 6));
        s[j + 4] = static_cast<uint8_t>((m[j] & 63) | ((m[j + 4] >> 4) << 6));
        s[j + 8] = static_cast<uint8_t>((sc[j + 4] & 15) | ((m[j + 4] & 15) << 4));
    }
#pragma unroll
    for (int k = 0; k < 3; ++k)
        out[1 + k] = static_cast<uint32_t>(s[4 * k]) | (static_cast<uint32_t>(s[4 * k + 1]) << 8) |
                     (static_cast<uint32_t>(s[4 * k + 2]) << 16) | (static_cast<uint32_t>(s[4 * k + 3]) << 24);
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const float step0 = __fmul_rn(dd, static_cast<float>(sc[2 * p]));
        const float off0 = __fmul_rn(ddm, static_cast<float>(m[2 * p]));
        const float step1 = __fmul_rn(dd, static_cast<float>(sc[2 * p + 1]));
        const float off1 = __fmul_rn(ddm, static_cast<float>(m[2 * p + 1]));
        for (int i4 = 0; i4 < 8; ++i4) {
            uint32_t word = 0;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = 4 * i4 + u;
                int q0 = 0, q1 = 0;
                if (step0 > 0.0f)
                    q0 = round_clamp(__fdiv_rn(__fadd_rn(__ldg(v + 64 * p + i), off0), step0), 15);
                if (step1 > 0.0f)
                    q1 = round_clamp(__fdiv_rn(__fadd_rn(__ldg(v + 64 * p + 32 + i), off1), step1), 15);
                word |= static_cast<uint32_t>(q0 | (q1 << 4)) << (8 * u);
            }
            out[4 + 8 * p + i4] = word;
        }
    }
    uint32_t* dst = reinterpret_cast<uint32_t*>(Wq + idx * 144);
#pragma unroll
    for (int k = 0; k < 36; ++k) dst[k] = out[k];
}

// One thread per Q5_K super-block (176 bytes: the Q4_K header, 32 bytes of
// top bits, 128 bytes of low four bits), the Q4_K steps with 31 code steps
// per sub-block, each one IEEE fp32 operation (the same bytes as the
// library's reference quantizer).
__global__ void quantize_q5_k_kernel(const float* __restrict__ w, int64_t ldw, int64_t O, int K,
                                     uint8_t* __restrict__ Wq) {
    const int nsb = K >> 8;
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= O * nsb) return;
    const int64_t row = idx / nsb;
    const int sbi = static_cast<int>(idx - row * nsb);
    const float* v = w + row * ldw + (static_cast<int64_t>(sbi) << 8);
    float a[8], mn[8], amax = 0.0f, mnmax = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float lo = __ldg(v + 32 * j), hi = lo;
        for (int i = 1; i < 32; ++i) {
            const float t = __ldg(v + 32 * j + i);
            if (t < lo) lo = t;
            if (t > hi) hi = t;
        }
        mn[j] = lo < 0.0f ? -lo : 0.0f;
        a[j] = __fdiv_rn(__fadd_rn(hi, mn[j]), 31.0f);
        if (a[j] > amax) amax = a[j];
        if (mn[j] > mnmax) mnmax = mn[j];
    }
    const __half dh = __float2half_rn(__fdiv_rn(amax, 63.0f));
    const __half dmh = __float2half_rn(__fdiv_rn(mnmax, 63.0f));
    const float dd = __half2float(dh), ddm = __half2float(dmh);
    int sc[8], m[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        sc[j] = dd > 0.0f ? round_clamp(__fdiv_rn(a[j], dd), 63) : 0;
        m[j] = ddm > 0.0f ? round_clamp(__fdiv_rn(mn[j], ddm), 63) : 0;
    }
    uint32_t out[44];
    out[0] = static_cast<uint32_t>(__half_as_ushort(dh)) | (static_cast<uint32_t>(__half_as_ushort(dmh)) << 16);
    uint8_t s[12];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        s[j] = static_cast<uint8_t>((sc[j] & 63) | ((sc[j + 4] >> 4) << 6));
        s[j + 4] = static_cast<uint8_t>((m[j] & 63) | ((m[j + 4] >> 4) << 6));
        s[j + 8] = static_cast<uint8_t>((sc[j + 4] & 15) | ((m[j + 4] & 15) << 4));
    }
#pragma unroll
    for (int k = 0; k < 3; ++k)
        out[1 + k] = static_cast<uint32_t>(s[4 * k]) | (static_cast<uint32_t>(s[4 * k + 1]) << 8) |
                     (static_cast<uint32_t>(s[4 * k + 2]) << 16) | (static_cast<uint32_t>(s[4 * k + 3]) << 24);
    uint32_t qh[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) qh[k] = 0u;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const float step0 = __fmul_rn(dd, static_cast<float>(sc[2 * p]));
        const float off0 = __fmul_rn(ddm, static_cast<float>(m[2 * p]));
        const float step1 = __fmul_rn(dd, static_cast<float>(sc[2 * p + 1]));
        const float off1 = __fmul_rn(ddm, static_cast<float>(m[2 * p + 1]));
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
            uint32_t word = 0, top = 0;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = 4 * i4 + u;
                int q0 = 0, q1 = 0;
                if (step0 > 0.0f)
                    q0 = round_clamp(__fdiv_rn(__fadd_rn(__ldg(v + 64 * p + i), off0), step0), 31);
                if (step1 > 0.0f)
                    q1 = round_clamp(__fdiv_rn(__fadd_rn(__ldg(v + 64 * p + 32 + i), off1), step1), 31);
                word |= static_cast<uint32_t>((q0 & 15) | ((q1 & 15) << 4)) << (8 * u);
                top |= static_cast<uint32_t>(((q0 >> 4) << (2 * p)) | ((q1 >> 4) << (2 * p + 1))) << (8 * u);
            }
            out[12 + 8 * p + i4] = word;
            qh[i4] |= top;
        }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) out[4 + k] = qh[k];
    uint32_t* dst = reinterpret_cast<uint32_t*>(Wq + idx * 176);
#pragma unroll
    for (int k = 0; k < 44; ++k) dst[k] = out[k];
}

}  // namespace

unsigned flags_read_clear_quantize(cudaStream_t stream) {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_flags_quantize, sizeof(v), 0, cudaMemcpyDeviceToHost, stream) !=
        cudaSuccess)
        return ~0u;
    if (cudaMemcpyToSymbolAsync(g_flags_quantize, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream) !=
        cudaSuccess)
        return ~0u;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return ~0u;
    return v;
}

}  // namespace qdg

using namespace qdg;

namespace {

int qnorm_launch(const float* x, int64_t ldx, const float* gamma, const float* add, int64_t ldadd, float eps,
                 int64_t K, int64_t N, void* xq, qdg_stream_t stream) {
    if (!x || !xq) return QDG_EINVAL;
    if (K <= 0 || N <= 0 || ldx < K) return QDG_EINVAL;
    if (add && ldadd != 0 && ldadd < K) return QDG_EINVAL;
    if (!(eps >= 0.0f) || std::isinf(eps)) return QDG_EINVAL;
    if (K % 32 != 0 || K > (1 << 20)) return QDG_ESHAPE;
    const int splits = static_cast<int>((K / 32 + kBlocksPerCta - 1) / kBlocksPerCta);
    if (N * splits > 0x7fffffff) return QDG_ESHAPE;
    if (!aligned(x, 4) || !aligned(xq, 2) || (gamma && !aligned(gamma, 4)) || (add && !aligned(add, 4)))
        return QDG_EALIGN;
    cudaError_t e = launch(qnorm_q8_kernel, dim3(static_cast<unsigned>(N * splits)), dim3(kNormThreads), 0,
                           reinterpret_cast<cudaStream_t>(stream), true, x, ldx, gamma, add, add ? ldadd : int64_t(0),
                           eps, static_cast<int>(K), splits, static_cast<uint8_t*>(xq));
    if (e != cudaSuccess) return QDG_ECUDA;
    count_launch(0);
    return QDG_OK;
}

}  // namespace

extern "C" int qnorm_quantize_q8_0(const float* x, int64_t ldx, const float* gamma, float eps, int64_t K, int64_t N,
                                   void* xq, qdg_stream_t stream) {
    return qnorm_launch(x, ldx, gamma, nullptr, 0, eps, K, N, xq, stream);
}

extern "C" int qnorm_add_quantize_q8_0(const float* x, int64_t ldx, const float* gamma, const float* add,
                                       int64_t ldadd, float eps, int64_t K, int64_t N, void* xq,
                                       qdg_stream_t stream) {
    if (!add) return QDG_EINVAL;
    return qnorm_launch(x, ldx, gamma, add, ldadd, eps, K, N, xq, stream);
}

extern "C" int quantize_q4_0(const float* w, int64_t ldw, int64_t O, int64_t K, void* Wq, qdg_stream_t stream) {
    if (!w || !Wq) return QDG_EINVAL;
    if (O <= 0 || K <= 0 || ldw < K) return QDG_EINVAL;
    if (K % 32 != 0 || K > (1 << 20)) return QDG_ESHAPE;
    if (!aligned(w, 4) || !aligned(Wq, 2)) return QDG_EALIGN;
    const int64_t blocks = O * (K / 32);
    const int threads = 256;
    const int64_t grid = (blocks + threads - 1) / threads;
    if (grid > 0x7fffffff) return QDG_ESHAPE;
    cudaError_t e = launch(quantize_q4_0_kernel, dim3(static_cast<unsigned>(grid)), dim3(threads), 0,
                           reinterpret_cast<cudaStream_t>(stream), false, w, ldw, O, static_cast<int>(K),
                           static_cast<uint8_t*>(Wq));
    if (e != cudaSuccess) return QDG_ECUDA;
    count_launch(4);
    return QDG_OK;
}

extern "C" int quantize_q4_k(const float* w, int64_t ldw, int64_t O, int64_t K, void* Wq, qdg_stream_t stream) {
    if (!w || !Wq) return QDG_EINVAL;
    if (O <= 0 || K <= 0 || ldw < K) return QDG_EINVAL;
    if (K % 256 != 0 || K > (1 << 20)) return QDG_ESHAPE;
    if (!aligned(w, 4) || !aligned(Wq, 4)) return QDG_EALIGN;
    const int64_t sbs = O * (K / 256);
    const int threads = 128;
    const int64_t grid = (sbs + threads - 1) / threads;
    if (grid > 0x7fffffff) return QDG_ESHAPE;
    cudaError_t e = launch(quantize_q4_k_kernel, dim3(static_cast<unsigned>(grid)), dim3(threads), 0,
                           reinterpret_cast<cudaStream_t>(stream), false, w, ldw, O, static_cast<int>(K),
                           static_cast<uint8_t*>(Wq));
    if (e != cudaSuccess) return QDG_ECUDA;
    count_launch(4);
    return QDG_OK;
}

extern "C" int quantize_q5_k(const float* w, int64_t ldw, int64_t O, int64_t K, void* Wq, qdg_stream_t stream) {
    if (!w || !Wq) return QDG_EINVAL;
    if (O <= 0 || K <= 0 || ldw < K) return QDG_EINVAL;
    if (K % 256 != 0 || K > (1 << 20)) return QDG_ESHAPE;
    if (!aligned(w, 4) || !aligned(Wq, 4)) return QDG_EALIGN;
    const int64_t sbs = O * (K / 256);
    const int threads = 128;
    const int64_t grid = (sbs + threads - 1) / threads;
    if (grid > 0x7fffffff) return QDG_ESHAPE;
    cudaError_t e = launch(quantize_q5_k_kernel, dim3(static_cast<unsigned>(grid)), dim3(threads), 0,
                           reinterpret_cast<cudaStream_t>(stream), false, w, ldw, O, static_cast<int>(K),
                           static_cast<uint8_t*>(Wq));
    if (e != cudaSuccess) return QDG_ECUDA;
    count_launch(4);
    return QDG_OK;
}
