/*
 * qdg.h -- C ABI of the GB300 (sm_103a) quantized decode GEMV library.
 *
 * What the library computes.  A decode step multiplies each projection's
 * quantized weight matrix by one activation vector; prefill multiplies it by
 * many.  Batch-1 decode goes down the quantized matrix-vector route ("mmvq"),
 * longer batches down the quantized matrix-matrix route ("mmq")  [GGML:
 * Backend abstraction and hardware acceleration, section "CUDA: mmvq, mmq,
 * cublas -- three matrix paths", shape-dispatch table].  Weights are Q4,
 * activations Q8 on every backend  [same page, sections "Metal and Vulkan"
 * and "How hardware choice maps onto the stack"].  The activation is first
 * RMS-normalised and multiplied by gamma (RMS_NORM + MUL), a pair the Metal
 * backend runs as one fused kernel; losing that fusion cost about 5% of
 * token-generation speed  [llama.cpp b10909: Metal backend fusion-table
 * refactor, introduction].  Here the norm, the MUL and the Q8_0 quantization
 * are one kernel, and the quantized products are three more.
 *
 * Formats (32-element blocks, little-endian, packed, no padding):
 *   Q4_0 block (18 bytes): uint16 fp16 scale d; uint8 qs[16].  Byte j holds
 *     element j in its low nibble and element j+16 in its high nibble; the
 *     value of element i is d * (q_i - 8), q_i in 0..15.
 *   Q8_0 block (34 bytes): uint16 fp16 scale d; int8 q[32]; value d * q_i.
 *   A Q4_0 matrix of O rows and K columns is row-major: row o holds its K/32
 *   blocks contiguously (o * K/32 * 18 bytes from the base).  N Q8_0 vectors
 *   are stored one after another, K/32 blocks each.
 *
 * Output.  y[n][o] = sum over blocks b of d_w(o,b) * d_x(n,b) * isum(n,o,b)
 *   with the exact integer block sum isum = sum_j (q_w - 8) * q_x, computed in
 *   fp32 from exact products; the result agrees with the exact value within
 *   1e-5 * sum_b |d_w d_x isum|.
 *
 * Conventions for every entry point:
 *   - Pointers named x, gamma, xq, W, y, w, isum are DEVICE pointers owned by
 *     the caller; the library never frees or keeps them and allocates no
 *     device memory.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  Arguments are validated on the host before anything
 *     is launched; a rejected call launches nothing and returns a negative
 *     status.  QDG_ECUDA reports a failed launch (cudaGetLastError).
 *   - Device-side problems (a bounded wait that gave up, a Q8_0 scale that
 *     overflowed fp16) set a flag on the device; qdg_device_status() reports
 *     and clears it.
 *   - No entry point is thread-safe against concurrent qdg_set_option calls.
 */
#ifndef QDG_H
#define QDG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define QDG_API __attribute__((visibility("default")))
#else
#define QDG_API
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* qdg_stream_t;

enum qdg_status {
    QDG_OK = 0,
    QDG_EINVAL = -1,    /* null pointer, non-positive size, N out of range, bad option */
    QDG_EALIGN = -2,    /* a pointer or a leading dimension breaks the required alignment */
    QDG_ESHAPE = -3,    /* K not a multiple of 32 (256 for the products) or beyond a stated maximum */
    QDG_ECUDA = -4,     /* a CUDA runtime call failed */
    QDG_ETIMEOUT = -5,  /* a bounded device-side wait gave up (from qdg_device_status) */
    QDG_EOVERFLOW = -6  /* a Q8_0 scale exceeded the fp16 range (from qdg_device_status) */
};

/*
 * qnorm_quantize_q8_0 -- fused RMS_NORM + MUL(gamma) + Q8_0 quantization.
 *   [llama.cpp b10909, introduction and section "CI and related fixes"
 *   (the RMS_NORM+MUL pattern); llama.cpp b10981, section "NPU cacheless
 *   encoder models and norm optimisation" (epsilon kept where GGML puts it)]
 *
 * x      [N][ldx] fp32, vector n at x + n*ldx (ldx >= K; 4-byte aligned).
 * gamma  [K] fp32, or NULL for plain quantization (no norm: v = x).
 * eps    >= 0, added to the mean square inside the square root.
 * K      multiple of 32, 32 <= K <= 1048576.   N >= 1.
 * xq     [N][K/32] Q8_0 blocks (2-byte aligned).
 * With gamma: s = 1/sqrt(sum(x^2)/K + eps), v_i = (x_i*s)*gamma_i, each an
 * IEEE fp32 operation; the sum of squares uses this library's fixed order
 * (256 strided fused multiply-add chains, then pairwise trees), so results
 * are bit-reproducible.  Per block: d = max|v|/127, q = round(v/d) (halves
 * away from zero), stored d = fp16(d) rounded to nearest even; d = 0 stores
 * q = 0.  A block whose d exceeds the fp16 range stores an infinite scale
 * and sets QDG_EOVERFLOW on the device.
 */
QDG_API int qnorm_quantize_q8_0(const float* x, int64_t ldx, const float* gamma, float eps,
                        int64_t K, int64_t N, void* xq, qdg_stream_t stream);

/*
 * qnorm_add_quantize_q8_0 -- fused RMS_NORM + MUL(gamma) + ADD + Q8_0
 * quantization  [llama.cpp b10909, section "CI and related fixes" (the
 * RMS_NORM+MUL+ADD fusion pattern)].
 *
 * As qnorm_quantize_q8_0, with v_i = (x_i*s)*gamma_i + a_i (or x_i + a_i
 * when gamma is NULL): one IEEE fp32 addition after the products.  The RMS
 * statistic is over x alone.
 * add    fp32 addend, 4-byte aligned: vector n uses add + n*ldadd; ldadd = 0
 *        uses the same K values for every vector, otherwise ldadd >= K.
 * Errors: QDG_EINVAL also for a NULL add or 0 < ldadd < K.
 */
QDG_API int qnorm_add_quantize_q8_0(const float* x, int64_t ldx, const float* gamma,
                                    const float* add, int64_t ldadd, float eps, int64_t K,
                                    int64_t N, void* xq, qdg_stream_t stream);

/*
 * q4_0_q8_0_gemv -- y = W * x for one Q8_0 vector (batch-1 decode, the
 * "mmvq" route)  [GGML: Backend abstraction and hardware acceleration,
 * section "CUDA: mmvq, mmq, cublas -- three matrix paths"].
 *
 * W   [O][K/32] Q4_0, 16-byte aligned.      xq  [K/32] Q8_0, 4-byte aligned.
 * y   [O] fp32, 4-byte aligned (overwritten).
 * K   multiple of 256, 256 <= K <= 32768.   1 <= O < 2^31.
 * W is streamed once from HBM with 16-byte loads issued several row
 * segments ahead; the result is deterministic (fixed reduction order).
 */
QDG_API int q4_0_q8_0_gemv(const void* W, const void* xq, float* y, int64_t O, int64_t K,
                   qdg_stream_t stream);

/*
 * q4_0_q8_0_gemv_group -- q4_0_q8_0_gemv for up to 4 matrices that read the
 * same Q8_0 vector (a decode layer's q, k and v; its gate and up), in one
 * launch: y[g] = W[g] * x.  W, y, O are host arrays of `count` (1..4) entries:
 * device pointers W[g] ([O[g]][K/32] Q4_0, 16-byte aligned), y[g] ([O[g]]
 * fp32), row counts O[g] >= 1; all matrices have the same K (multiple of 256,
 * <= 32768).  Results are bit-identical to one q4_0_q8_0_gemv per matrix.
 */
QDG_API int q4_0_q8_0_gemv_group(const void* const* W, float* const* y, const int64_t* O, int count,
                                 const void* xq, int64_t K, qdg_stream_t stream);

/*
 * q4_0_gemv_rmsnorm -- the fused decode route: RMS_NORM + MUL(gamma) + Q8_0
 * quantization + Q4_0 x Q8_0 GEMV in one kernel.  The norm/MUL pair is the
 * pattern whose fusion the Metal backend lost (about 5% of token generation)
 *   [llama.cpp b10909, introduction]; here the quantization and the product
 *   join it, so a decode projection is a single launch.
 *
 * W      [O][K/32] Q4_0, 16-byte aligned.
 * x      [K] fp32, 16-byte aligned.   gamma [K] fp32, 16-byte aligned, or NULL
 *        for plain quantization.   eps >= 0 (inside the square root).
 * y      [O] fp32 (overwritten).
 * xq_out [K/32] Q8_0 or NULL: if given, receives the quantized activations.
 * K      multiple of 256, 256 <= K <= 16384 (x and gamma are staged in
 *        shared memory).
 * The quantized activations are bit-identical to qnorm_quantize_q8_0's and y
 * is bit-identical to q4_0_q8_0_gemv on them.  Every CTA recomputes the
 * norm and the quantization (the vector is small and L2-resident) while its
 * first weight segments are already in flight.
 */
QDG_API int q4_0_gemv_rmsnorm(const void* W, const float* x, const float* gamma, float eps, float* y,
                              int64_t O, int64_t K, void* xq_out, qdg_stream_t stream);

/*
 * q4_0_gemv_rmsnorm_group -- the fused route for up to 4 projections that
 * read the same activation (a decode layer's q, k and v; its gate and up):
 * one launch normalises and quantizes x once per CTA and streams the rows of
 * all the matrices, y[g] = W[g] * Q8_0(RMSNorm(x) * gamma).
 *
 * W, y, O   host arrays of `count` entries (1..4): device pointers W[g]
 *           ([O[g]][K/32] Q4_0, 16-byte aligned) and y[g] ([O[g]] fp32), and
 *           row counts O[g] >= 1.  All matrices have the same K.
 * Other arguments as q4_0_gemv_rmsnorm.  Results are bit-identical to
 * q4_0_gemv_rmsnorm called once per matrix.
 */
QDG_API int q4_0_gemv_rmsnorm_group(const void* const* W, float* const* y, const int64_t* O, int count,
                                    const float* x, const float* gamma, float eps, int64_t K, void* xq_out,
                                    qdg_stream_t stream);

/*
 * q4_0_q8_0_gemm_small_n -- Y = W * X for 1 <= N <= 8 Q8_0 vectors sharing
 * one pass over W (speculative / parallel decode; the "vector case" of the
 * mmvq route)  [same page and section].
 *
 * W   [O][K/32] Q4_0, 16-byte aligned.   xq  [N][K/32] Q8_0, 16-byte aligned.
 * y   [N][ldy] fp32: output vector n at y + n*ldy, ldy >= O.
 * K   multiple of 256, 256 <= K <= 32768.   1 <= N <= 8.
 * The exact per-block integer sums are formed on the warp-level fp16 MMA
 * (integer codes held exactly in fp16, fp32 accumulation) and scaled per
 * block in fp32.  For K > 4096 the kernel runs as thread-block clusters of
 * ceil(K/4096) CTAs that split K and combine their partial sums in a fixed
 * order through distributed shared memory: no workspace, deterministic
 * results.
 */
QDG_API int q4_0_q8_0_gemm_small_n(const void* W, const void* xq, float* y, int64_t ldy,
                           int64_t O, int64_t K, int64_t N, qdg_stream_t stream);

/*
 * q4_0_q8_0_gemm -- Y = W * X for T tokens (prefill, the "mmq" route)
 *   [same page and section: quantized matrices other than the vector case go
 *   to mmq; long prefill batches keep it busy].
 *
 * W   [O][K/32] Q4_0, 16-byte aligned.   xq  [T][K/32] Q8_0, 16-byte aligned.
 * y   [T][ldy] fp32: the output for token t at y + t*ldy, ldy >= O.
 * K   multiple of 256, 256 <= K <= 65536.   1 <= O, T <= 2^30.
 * workspace: device memory of at least q4_0_q8_0_gemm_workspace_bytes(K, T)
 *   bytes, 16-byte aligned, owned by the caller; contents need no
 *   initialisation and are overwritten.  Two calls that overlap on the GPU
 *   must not share a workspace.
 * Two kernels: the first converts each activation block once into the
 * tensor-core operand form (fp16 codes, fp32 scale) in the workspace; the
 * second forms the exact per-block integer sums on the fifth-generation
 * tensor cores (tcgen05.mma, fp16 operands holding the integer codes
 * exactly, fp32 accumulation in tensor memory) and scales them per block on
 * the CUDA cores.  Every output tile is owned by one CTA, so results are
 * deterministic.
 * Errors: QDG_EINVAL (null pointer, sizes, workspace too small), QDG_ESHAPE,
 * QDG_EALIGN, QDG_ECUDA (launch).
 */
QDG_API int q4_0_q8_0_gemm(const void* W, const void* xq, float* y, int64_t ldy,
                           int64_t O, int64_t K, int64_t T, void* workspace,
                           int64_t workspace_bytes, qdg_stream_t stream);

/*
 * q4_0_q8_0_gemm_workspace_bytes -- workspace size for q4_0_q8_0_gemm:
 * ceil(T/128) * (K/32) * 8704 bytes (one converted activation record per
 * 128-token tile and block).  Negative status for invalid K or T.
 */
QDG_API int64_t q4_0_q8_0_gemm_workspace_bytes(int64_t K, int64_t T);

/*
 * q4_0_q8_0_gemm_workspace_size -- the same figure with the argument list
 * (O, K, T) of the product itself; O does not change it (O < 1 gives
 * QDG_EINVAL, O > 2^30 QDG_ESHAPE, as the product would).
 */
QDG_API int64_t q4_0_q8_0_gemm_workspace_size(int64_t O, int64_t K, int64_t T);

/*
 * q4_0_q8_0_gemm_static -- q4_0_q8_0_gemm without a caller workspace and
 * without any device allocation.  The pages have no counterpart: this is a
 * library convenience for callers that cannot allocate device memory, such
 * as a plug-in whose host program owns every byte of the GPU through its
 * own pool, or code that runs where cudaMalloc is not permitted (inside a
 * stream capture, or under a fixed memory budget).
 * Its scratch is a 16 MiB array in the library's device memory (held by
 * every GPU that loads the library until the process exits), so the
 * problem must satisfy q4_0_q8_0_gemm_workspace_bytes(K, T) <= 16 MiB
 * (e.g. T <= 1920 tokens at K = 4096, T <= 512 at K = 14336); larger ones
 * return QDG_ESHAPE.  The first call on a device looks up the array's
 * address on that device (make it before any stream capture); the address
 * is kept for the life of the process, so after cudaDeviceReset the library
 * must be unloaded and loaded again before this entry is used.  Nothing
 * needs to start at zero.  All calls share the array: calls that overlap on
 * the GPU race.  Other arguments and errors as q4_0_q8_0_gemm.
 */
QDG_API int q4_0_q8_0_gemm_static(const void* W, const void* xq, float* y, int64_t ldy,
                                  int64_t O, int64_t K, int64_t T, qdg_stream_t stream);

/*
 * quantize_q4_0 -- weight preparation: fp32 [O][ldw] -> Q4_0 [O][K/32].
 * Per block: m = the element of largest magnitude (the first one on ties),
 * d = m / -8 in fp32, q = min(15, floor(w/d + 8.5)), stored d = fp16(d); an
 * all-zero block stores d = 0 and q = 8.  Runs once at load time, not on the
 * decode path.  K multiple of 32, ldw >= K; Wq 2-byte aligned.
 */
QDG_API int quantize_q4_0(const float* w, int64_t ldw, int64_t O, int64_t K, void* Wq,
                  qdg_stream_t stream);

/*
 * q8_0_q8_0_gemv -- y = W * x with Q8_0 weights: the stack's conversion step
 * picks the weight type (Q4_K or Q8_0) and every back end's matrix kernels
 * must know each type [GGML: Backend abstraction and hardware acceleration,
 * sections "How one production call lands on the hardware" and "Metal and
 * Vulkan"].  W [O][K/32] Q8_0 blocks (34 bytes: fp16 d, 32 int8 codes; made,
 * for example, by qnorm_quantize_q8_0 with gamma = NULL), 16-byte aligned.
 * xq [K/32] Q8_0, 4-byte aligned.  y [O] fp32 (overwritten).  K multiple of
 * 256, <= 32768; 1 <= O < 2^31.  Per block the exact integer sum of code
 * products, scaled by d_w * d_x; deterministic.  8.5 bits per weight are
 * streamed, so it takes about 1.9x the time of the Q4_0 product.
 */
QDG_API int q8_0_q8_0_gemv(const void* W, const void* xq, float* y, int64_t O, int64_t K,
                           qdg_stream_t stream);

/* q8_0_q8_0_gemv for up to 4 Q8_0 matrices reading one Q8_0 vector, in one
 * launch (argument rules as q4_0_q8_0_gemv_group). */
QDG_API int q8_0_q8_0_gemv_group(const void* const* W, float* const* y, const int64_t* O, int count,
                                 const void* xq, int64_t K, qdg_stream_t stream);

/*
 * quantize_q4_k -- weight preparation: fp32 [O][ldw] -> Q4_K [O][K/256]
 * super-blocks (format under q4_k_q8_0_gemv below).  The library's plain
 * reading of the k-quant recipe (the pages name Q4_K but give no
 * quantizer): per 32-weight sub-block j, mn_j = max(0, -min w) and
 * a_j = (max w + mn_j) / 15; d = fp16(max_j a_j / 63), dmin =
 * fp16(max_j mn_j / 63); sc_j = round(a_j / d), m_j = round(mn_j / dmin)
 * clamped to 0..63; q = round((w + dmin m_j) / (d sc_j)) clamped to 0..15
 * (halves away from zero; 0 where a divisor is 0); each step one IEEE fp32
 * operation.  Load time, not the decode path.  K multiple of 256,
 * ldw >= K; w and Wq 4-byte aligned.
 */
QDG_API int quantize_q4_k(const float* w, int64_t ldw, int64_t O, int64_t K, void* Wq,
                          qdg_stream_t stream);

/*
 * q4_k_q8_0_gemv -- y = W * x with Q4_K weights, the other weight type the
 * conversion step picks [GGML: Backend abstraction and hardware
 * acceleration, sections "How one production call lands on the hardware"
 * and "Metal and Vulkan"].  The pages give no block format; the library
 * reads Q4_K as GGML's 256-weight k-quant super-block of 144 bytes:
 *   bytes 0-1 fp16 d, bytes 2-3 fp16 dmin, bytes 4-15 s[0..11] packing
 *   eight 6-bit sub-block scales sc_j and mins m_j (j < 4: sc_j = s[j] & 63,
 *   m_j = s[j+4] & 63; j >= 4: sc_j = (s[j+4] & 15) + 16 (s[j-4] >> 6),
 *   m_j = (s[j+4] >> 4) + 16 (s[j] >> 6)), bytes 16-143 the codes: byte
 *   16 + 32p + i holds element i of sub-block 2p (low nibble) and of
 *   sub-block 2p+1 (high nibble).  Weight = d sc_j q - dmin m_j, q in 0..15.
 * W [O][K/256] super-blocks (row = 18 K/32 bytes, as Q4_0), 16-byte aligned.
 * xq [K/32] Q8_0, 4-byte aligned: each Q8_0 block meets one 32-weight
 * sub-block.  y [O] fp32 (overwritten).  K multiple of 256, <= 32768;
 * 1 <= O < 2^31.  Per sub-block the exact integer sums isum = sum q q_x and
 * xsum = sum q_x, then d_x (d sc isum - dmin m xsum) in fp32; results agree
 * with the exact value within 1e-5 * sum |d_x d sc isum| + |d_x dmin m xsum|.
 * Deterministic.  4.5 bits per weight; a super-block is nine 16-byte words,
 * so lanes load their codes and headers straight into registers (the
 * row/segment split of q4_0s_q8_0_gemv, no repack needed).
 */
QDG_API int q4_k_q8_0_gemv(const void* W, const void* xq, float* y, int64_t O, int64_t K,
                           qdg_stream_t stream);

/* q4_k_q8_0_gemv for up to 4 Q4_K matrices reading one Q8_0 vector, in one
 * launch (argument rules as q4_0_q8_0_gemv_group). */
QDG_API int q4_k_q8_0_gemv_group(const void* const* W, float* const* y, const int64_t* O, int count,
                                 const void* xq, int64_t K, qdg_stream_t stream);

/*
 * quantize_q5_k -- weight preparation: fp32 [O][ldw] -> Q5_K [O][K/256]
 * super-blocks (format under q5_k_q8_0_gemv below).  The steps of
 * quantize_q4_k with 31 code steps per sub-block: a_j = (max w + mn_j) / 31,
 * q = round((w + dmin m_j) / (d sc_j)) clamped to 0..31; each step one IEEE
 * fp32 operation.  Load time.  K multiple of 256, ldw >= K; w and Wq 4-byte
 * aligned.
 */
QDG_API int quantize_q5_k(const float* w, int64_t ldw, int64_t O, int64_t K, void* Wq,
                          qdg_stream_t stream);

/*
 * q5_k_q8_0_gemv -- y = W * x with Q5_K weights, the 5-bit k-quant the pages
 * name beside Q4_K [llama.cpp b10981: OpenVINO backend optimises stateful
 * decode and GPU MoE inference, section "GPU MoE, env vars"].  No format on
 * the pages; the library reads Q5_K as GGML's 256-weight super-block of 176
 * bytes: bytes 0-15 as Q4_K (fp16 d, fp16 dmin, the twelve packed bytes of
 * 6-bit scales sc_j and mins m_j), bytes 16-47 qh[0..31] (bit j of qh[i] is
 * the top bit, value 16, of element i of sub-block j), bytes 48-175 the low
 * four bits placed as the Q4_K codes (byte 48 + 32p + i: element i of
 * sub-block 2p in the low nibble, of 2p+1 in the high nibble).  Weight =
 * d sc_j q - dmin m_j, q in 0..31.  W [O][K/256 * 176 bytes], 16-byte
 * aligned; xq [K/32] Q8_0, 2-byte aligned; y [O] fp32.  K multiple of 256,
 * <= 32768; 1 <= O < 2^31.  Exact sub-block sums isum = sum q q_x and
 * xsum = sum q_x, then d_x (d sc isum - dmin m xsum) in fp32 (tolerance as
 * q4_k_q8_0_gemv).  Deterministic.  5.5 bits per weight; the kernel of
 * q4_k_q8_0_gemv with each lane also loading its super-block's qh bytes.
 */
QDG_API int q5_k_q8_0_gemv(const void* W, const void* xq, float* y, int64_t O, int64_t K,
                           qdg_stream_t stream);

/* q5_k_q8_0_gemv for up to 4 Q5_K matrices reading one Q8_0 vector, in one
 * launch (argument rules as q4_0_q8_0_gemv_group). */
QDG_API int q5_k_q8_0_gemv_group(const void* const* W, float* const* y, const int64_t* O, int count,
                                 const void* xq, int64_t K, qdg_stream_t stream);

/*
 * Segment layout of Q4_0 weights (load-time repack).  GGML's CPU back end
 * rearranges Q4 weights once, when they are loaded, for its own kernels
 * [GGML: Backend abstraction and hardware acceleration, section "How build
 * switches become runtime capabilities", build-option table,
 * GGML_CPU_REPACK]; the pages give no layout.  This library's GPU layout
 * keeps each row contiguous and splits it into segments of 64 blocks:
 * segment s starts at byte 1152*s and holds the 16 nibble bytes of each of
 * its r blocks (block 64s+i at byte 16*i, bytes as in the Q4_0 block), then
 * 32 little-endian words, word l = fp16 scale of block 64s+l (low half) and
 * of block 64s+32+l (high half), 0 where that block does not exist.
 * Row bytes = 1152*(nseg-1) + 16*r_last + 128 (18*K/32 when 2048 divides K).
 * Every product of this layout gives the same exact block sums as the plain
 * layout; rows of several matrices that read one input (gate and up) may be
 * repacked into one buffer back to back and multiplied as one matrix.
 */

/* Bytes of one row in the segment layout; QDG_EINVAL (K <= 0) or QDG_ESHAPE
 * (K not a multiple of 256 or above 32768). */
QDG_API int64_t q4_0_seg_row_bytes(int64_t K);

/*
 * q4_0_repack_seg -- W [O][K/32] Q4_0 (2-byte aligned) -> Wr [O][row bytes]
 * in the segment layout (16-byte aligned, caller-owned, not overlapping W).
 * A byte rearrangement, bit-exact; runs once at load time.  K multiple of
 * 256, <= 32768.  Asynchronous on `stream`.
 */
QDG_API int q4_0_repack_seg(const void* W, void* Wr, int64_t O, int64_t K, qdg_stream_t stream);

/*
 * q4_0s_q8_0_gemv -- q4_0_q8_0_gemv on weights in the segment layout.
 * Wr  [O][q4_0_seg_row_bytes(K)], 16-byte aligned.  xq [K/32] Q8_0, 2-byte
 * aligned.  y [O] fp32 (overwritten).  K multiple of 256, <= 32768;
 * 1 <= O < 2^31.  Each lane reads its blocks' nibbles with 16-byte loads and
 * their scales with one 4-byte load, issued four row segments ahead, straight
 * into registers; deterministic (fixed reduction order).
 */
QDG_API int q4_0s_q8_0_gemv(const void* Wr, const void* xq, float* y, int64_t O, int64_t K,
                            qdg_stream_t stream);

/*
 * q4_0s_q8_0_gemv_group -- q4_0s_q8_0_gemv for up to 4 segment-layout
 * matrices reading one Q8_0 vector, in one launch (argument rules as
 * q4_0_q8_0_gemv_group).  Bit-identical to one call per matrix.
 */
QDG_API int q4_0s_q8_0_gemv_group(const void* const* Wr, float* const* y, const int64_t* O, int count,
                                  const void* xq, int64_t K, qdg_stream_t stream);

/*
 * q4_0s_q8_0_gemm_small_n -- the small-N product on the segment layout for
 * N = 1..8 vectors sharing one pass over W (speculative / parallel decode).
 * N = 1 is q4_0s_q8_0_gemv.  At N = 2 each block's nibbles are unpacked once
 * and dotted with both vectors by dp4a.  At N = 3, 4 with K <= 16384 a lane
 * owns one block of a half-segment and keeps that block of every vector in
 * registers; the exact block sums come from dp4a, eight rows in flight per
 * warp.  Otherwise (N = 5..8, or K > 16384) the exact block sums come from
 * the fp16 warp MMA as in q4_0_q8_0_gemm_small_n (same arithmetic and order,
 * bit-identical), each warp staging its own tiles with cp.async; for
 * K > 4096 a thread-block cluster of ceil(K/4096) CTAs splits K.
 * Wr [O][q4_0_seg_row_bytes(K)], 16-byte aligned; xq: N Q8_0 vectors of K/32
 * blocks back to back (16-byte aligned for N >= 3, 2-byte aligned for
 * N <= 2); y: [N][ldy] fp32, ldy >= O.
 * K multiple of 256, <= 32768; 1 <= O < 2^31.  Deterministic (fixed
 * reduction order).  QDG_EINVAL for N outside 1..8.
 */
QDG_API int q4_0s_q8_0_gemm_small_n(const void* Wr, const void* xq, float* y, int64_t ldy, int64_t O,
                                    int64_t K, int64_t N, qdg_stream_t stream);

/*
 * q4_0s_gemv_rmsnorm_group -- the fused route on the segment layout: for up
 * to 4 matrices Wr[g] (segment layout, [O[g]] rows) that share the input x,
 * one launch runs RMS_NORM + MUL by gamma + Q8_0 quantization of x and the
 * products y[g] = Wr[g] * xq  [llama.cpp b10909: Metal backend fusion-table
 * refactor, introduction (RMS_NORM+MUL); GGML: Backend abstraction and
 * hardware acceleration, section "CUDA: mmvq, mmq, cublas -- three matrix
 * paths"].  Every CTA quantizes the whole vector with the arithmetic and the
 * summation order of qnorm_quantize_q8_0, so xq (optionally copied to xq_out,
 * [K/32] Q8_0, 4-byte aligned) is bit-identical to it and y equals
 * q4_0s_q8_0_gemv_group on that xq.  x, gamma: fp32 [K], 16-byte aligned;
 * gamma = NULL quantizes x without a norm.  K multiple of 256, <= 16384
 * (x and gamma are staged whole in shared memory).
 */
QDG_API int q4_0s_gemv_rmsnorm_group(const void* const* Wr, float* const* y, const int64_t* O, int count,
                                     const float* x, const float* gamma, float eps, int64_t K, void* xq_out,
                                     qdg_stream_t stream);

/*
 * q4_0s_gemv_chain -- the stages of a decode step in one launch.  Stage g
 * quantizes its input (RMS_NORM * gamma -> Q8_0, or plain Q8_0 when gamma is
 * NULL; the arithmetic of qnorm_quantize_q8_0, so the Q8_0 vector is the
 * same bit for bit) and multiplies it by up to four matrices in the segment
 * layout (q4_0_repack_seg), as q4_0s_q8_0_gemv_group does.  Stage g+1 reads
 * its input only after every output of stage g is written, so a stage may
 * read what an earlier stage wrote (its x may be an earlier stage's y).
 *   [RMS_NORM+MUL as one fused step: llama.cpp b10909: Metal backend
 *   fusion-table refactor, introduction and section "CI and related fixes";
 *   batch-1 decode on the quantized matrix-vector route: GGML: Backend
 *   abstraction and hardware acceleration, section "CUDA: mmvq, mmq,
 *   cublas -- three matrix paths"]
 * The pages describe the separate kernels; running a step's stages as one
 * persistent launch (cooperative: one CTA per SM, all resident, meeting at a
 * device-wide barrier between stages) is this library's GB300 design: it
 * removes the launch and grid-completion gaps at every stage boundary.
 *
 * stages   host array of nstages (1..8) stage descriptions:
 *   x        fp32 [K] input, 16-byte aligned.
 *   gamma    fp32 [K], 16-byte aligned, or NULL (no norm).
 *   xq_out   Q8_0 [K/32] copy of the stage's quantized input, or NULL.
 *   K        multiple of 256, 256 <= K <= 16384.
 *   count    matrices that read this input, 1..4; W[i] segment-layout
 *            weights of O[i] rows (16-byte aligned), y[i] fp32 [O[i]]
 *            (4-byte aligned); sum of O[i] < 2^30.
 * eps      epsilon of the norm (>= 0), added to the mean square inside the root.
 * workspace  device memory of q4_0s_gemv_chain_workspace_bytes() bytes,
 *          16-byte aligned, zeroed once before its first use: the stage
 *          barriers' arrival counters (64 bytes, left zero by every launch)
 *          and the image of a stage's quantized input.  Launches that may run
 *          at the same time need separate workspaces.  After a QDG_ETIMEOUT
 *          report it must be zeroed again.
 * Errors: QDG_EINVAL, QDG_ESHAPE, QDG_EALIGN as the single calls;
 * QDG_ECUDA if the cooperative launch is refused.  Results are
 * deterministic: every output row is summed in a fixed order.
 */
typedef struct {
    const float* x;
    const float* gamma;
    void* xq_out;
    int64_t K;
    int count;
    const void* W[4];
    float* y[4];
    int64_t O[4];
} qdg_chain_stage;

QDG_API int64_t q4_0s_gemv_chain_workspace_bytes(void);
QDG_API int q4_0s_gemv_chain(const qdg_chain_stage* stages, int nstages, float eps, void* workspace,
                             qdg_stream_t stream);

/*
 * qdg_device_status -- synchronise `stream`, then read and clear the device
 * flags of every kernel of this library on the current device.  Returns
 * QDG_OK, QDG_ETIMEOUT (a bounded wait gave up; that call's output is
 * incomplete), QDG_EOVERFLOW, or QDG_ECUDA.
 */
QDG_API int qdg_device_status(qdg_stream_t stream);

/* Human-readable text for a status code (static storage). */
QDG_API const char* qdg_status_string(int status);

/*
 * Options (process-wide).  QDG_OPT_PDL = 1 launches the decode kernels with
 * programmatic dependent launch: a kernel may start streaming W while the
 * previous kernel on the stream is still running, and waits for it before
 * reading activations or writing outputs.  Enable it only when W is not
 * written by the kernel launched immediately before on the same stream.
 * Default 0.  Returns QDG_EINVAL for an unknown option.
 */
enum qdg_option { QDG_OPT_PDL = 1 };
QDG_API int qdg_set_option(int option, int64_t value);

/*
 * qdg_stage_copy -- copy `bytes` bytes from src to dst with a kernel on
 * `stream`: the host <-> device move of a decode step's input vectors and
 * outputs.  Either pointer may be device memory or pinned host memory that is
 * mapped into the device's address space (memory from cudaHostAlloc, or
 * PyTorch's pin_memory(), on a unified-address system); the kernel reaches
 * host memory over the CPU-GPU link, so no copy engine is involved and, with
 * QDG_OPT_PDL set, the copy stays in the chain of dependent launches (the
 * kernel waits for the preceding grid before it touches either buffer, and
 * the next kernel may launch while it runs).
 *   dst, src  16-byte aligned, non-overlapping; caller-owned.
 *   bytes     a multiple of 16 (0: nothing launched).
 * Errors: QDG_EINVAL for a null pointer, negative size, overlapping ranges,
 * or a pointer the device cannot reach (pageable host memory); QDG_EALIGN
 * for an unaligned pointer or size; QDG_ECUDA if the launch fails.
 * Asynchronous: dst is complete when the stream reaches the copy's end.
 */
QDG_API int qdg_stage_copy(void* dst, const void* src, int64_t bytes, qdg_stream_t stream);

/*
 * qdg_launch_count -- number of kernels this library has launched in this
 * process, per kernel: which = 0 qnorm/quantize, 1 gemv, 2 small-N, 3 gemm,
 * 4 weight quantize, 5 fused norm+gemv, 6 segment-layout gemv, 7 repack,
 * 8 Q8_0-weight gemv, 9 fused norm+gemv on the segment layout, 10 staging copy,
 * 11 decode-step chain, 12 Q4_K-weight gemv, 13 three/four-vector segment-layout
 * small-N, 14 Q5_K-weight gemv, -1 total.  Lets a caller check
 * that the fused kernel is the one that ran.
 */
QDG_API int64_t qdg_launch_count(int which);

/*
 * qdg_debug_block_sums -- test hook.  Runs the production inner loop of one
 * product path and writes the exact per-block integer sums
 * isum[n][o][b] = sum_j (q_w - 8) * q_x  (int32 [N][O][K/32]) instead of y.
 * path: 0 = gemv (N must be 1), 1 = small-N, 2 = prefill gemm (N = T tokens),
 * 3 = segment-layout gemv (W in the segment layout, N must be 1),
 * 4 = Q8_0-weight gemv (W in Q8_0 blocks, N must be 1), 5 = segment-layout
 * small-N (W in the segment layout, N = 1..8), 6 = Q4_K-weight gemv (W in
 * Q4_K super-blocks, N must be 1; isum = sum q q_x per 32-weight sub-block),
 * 7 = Q5_K-weight gemv (W in Q5_K super-blocks, N must be 1; isum as for 6).
 * Same argument rules as the corresponding entry point.
 */
QDG_API int qdg_debug_block_sums(const void* W, const void* xq, int32_t* isum, int64_t O,
                         int64_t K, int64_t N, int path, qdg_stream_t stream);

/*
 * qdg_debug_timeout_probe -- test hook for failure detection.  Launches one
 * kernel that waits on a barrier nothing will complete; its bounded wait
 * gives up after about two seconds, sets the timeout flag and returns, so a
 * following qdg_device_status() reports QDG_ETIMEOUT and the context stays
 * usable.  Faults nothing.
 */
QDG_API int qdg_debug_timeout_probe(qdg_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QDG_H */
