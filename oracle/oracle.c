/*
 * oracle.c -- plain scalar CPU oracle for the quantized decode GEMV path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant with the CUDA library: every routine below is a
 * direct, slow restatement of what the method computes, in plain loops,
 * compiled with -O2 -ffp-contract=off so that every fp32 operation rounds
 * exactly once, where written.
 *
 * What the method computes (sources, by page title and section):
 *  - Decode multiplies a quantized weight matrix by one activation vector
 *    ("mmvq"), prefill by many ("mmq")  [GGML: Backend abstraction and
 *    hardware acceleration, section "CUDA: mmvq, mmq, cublas -- three matrix
 *    paths", shape-dispatch table].
 *  - The arithmetic convention is Q4 weights x Q8 activations on every
 *    backend  [same page, sections "Metal and Vulkan" and "How hardware choice
 *    maps onto the stack"].
 *  - The activation entering a projection is the output of RMS_NORM followed
 *    by MUL with a weight vector gamma, a pattern the Metal backend fuses
 *    [llama.cpp b10909: Metal backend fusion-table refactor, fixes ~5% token
 *    generation regression, introduction and section "CI and related fixes"].
 *  - The norm's epsilon sits where GGML puts it: added to the mean square,
 *    inside the square root  [llama.cpp b10981: OpenVINO backend optimises
 *    stateful decode and GPU MoE inference, section "NPU cacheless encoder
 *    models and norm optimisation"].
 *
 * Block formats (the library's reading of the Q4/Q8 convention; 32-element
 * blocks, little-endian):
 *  Q4_0 block, 18 bytes: fp16 scale d, then 16 bytes; byte j holds element j
 *       in its low nibble and element j+16 in its high nibble; value of
 *       element = d * (q - 8), q in 0..15.
 *  Q8_0 block, 34 bytes: fp16 scale d, then 32 int8 q; value = d * q.
 *
 * Parity pins: every function here is checked in tests/test_oracle_pins.py
 * against values the mathematics fixes (IEEE binary16 encodings from numpy,
 * closed forms, round-trip bounds, exact rational brute force on tiny
 * shapes, special blocks).  The bitwise summation order of the RMS statistic
 * is a convention of this library (fixed below); its value is pinned to the
 * fp64 definition within a few ulp.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <fenv.h>

#define QK 32

/* ---------------------------------------------------------------------- */
/* IEEE 754 binary16 <-> binary32, from the format's definition.           */
/* ---------------------------------------------------------------------- */

float orc_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);     /* (1 + m/1024) * 2^(e-15) */
    return (float)(sign ? -v : v);
}

/* Round to nearest, ties to even; overflow to infinity. */
uint16_t orc_f32_to_f16(float f)
{
    uint16_t sign = signbit(f) ? 0x8000u : 0u;
    if (isnan(f))
        return (uint16_t)(sign | 0x7E00u);
    double a = fabs((double)f);
    /* 65520 is the midpoint between the largest finite value 65504 and 2^16;
       ties go to the even significand, which is the (infinite) 2^16. */
    if (a >= 65520.0)
        return (uint16_t)(sign | 0x7C00u);
    if (a == 0.0)
        return sign;
    int e2;
    frexp(a, &e2);                  /* a = f * 2^e2, f in [0.5, 1) */
    int ex = e2 - 1;                /* floor(log2 a) */
    if (ex < -14)
        ex = -14;                   /* subnormal range has quantum 2^-24 */
    double quantum = ldexp(1.0, ex - 10);
    double n = a / quantum;         /* exact: division by a power of two */
    int old = fegetround();
    fesetround(FE_TONEAREST);
    double r = nearbyint(n);        /* ties to even */
    fesetround(old);
    long ri = (long)r;
    if (ex == -14 && ri < 1024)
        return (uint16_t)(sign | (uint16_t)ri);           /* subnormal (or min normal reached below) */
    if (ri == 2048) {               /* rounding carried into the next binade */
        ri = 1024;
        ex += 1;
    }
    if (ex + 15 >= 31)
        return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (uint16_t)((ex + 15) << 10) | (uint16_t)(ri - 1024));
}

static uint16_t rd_u16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void wr_u16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)(v & 0xFF); p[1] = (uint8_t)(v >> 8); }

/* ---------------------------------------------------------------------- */
/* Q4_0 weight quantization (input preparation).                           */
/* Per block: m = the element of largest magnitude (first one on ties),     */
/* d = m / -8 (fp32), q = min(15, floor(w/d + 8.5)), stored d = fp16(d).    */
/* An all-zero block stores d = 0 and q = 8 everywhere.                     */
/* ---------------------------------------------------------------------- */
void orc_quantize_q4_0(const float* w, int64_t rows, int64_t K, uint8_t* out)
{
    const int64_t nb = K / QK;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const float* v = w + r * K + b * QK;
            uint8_t* blk = out + (r * nb + b) * 18;
            float amax = 0.0f, m = 0.0f;
            for (int j = 0; j < QK; ++j) {
                if (fabsf(v[j]) > amax) {
                    amax = fabsf(v[j]);
                    m = v[j];
                }
            }
            float d = m / -8.0f;
            int q[QK];
            for (int j = 0; j < QK; ++j) {
                if (d == 0.0f) {
                    q[j] = 8;
                } else {
                    float t = v[j] / d;
                    t = t + 8.5f;
                    int qi = (int)t;            /* t >= 0.5 here, so this is floor */
                    q[j] = qi > 15 ? 15 : (qi < 0 ? 0 : qi);
                }
            }
            wr_u16(blk, orc_f32_to_f16(d));
            for (int j = 0; j < 16; ++j)
                blk[2 + j] = (uint8_t)(q[j] | (q[j + 16] << 4));
        }
    }
}

/* ---------------------------------------------------------------------- */
/* Segment layout of Q4_0 rows.  A weight row is rearranged once, at load   */
/* time, for the way the GPU reads it -- the GPU counterpart of the CPU back */
/* end's load-time repack of Q4 weights  [GGML: Backend abstraction and     */
/* hardware acceleration, section "How build switches become runtime        */
/* capabilities", build-option table, GGML_CPU_REPACK].  The pages name the */
/* repack but not a layout; this one is the library's:                      */
/*   a row of nb = K/32 blocks (K a multiple of 256) is cut into segments of */
/*   64 blocks; the last segment holds r = nb - 64*(nseg-1) blocks.          */
/*   Segment s starts at byte 1152*s and holds 16*r_s + 128 bytes:          */
/*     bytes 16*i .. 16*i+15: the 16 nibble bytes of block 64*s+i, as in    */
/*       the Q4_0 block;                                                    */
/*     then 32 little-endian 32-bit words; word l holds the fp16 scale of    */
/*       block 64*s+l in its low half and that of block 64*s+32+l in its    */
/*       high half; a half whose block does not exist is 0.                 */
/*   Row bytes = 1152*(nseg-1) + 16*r_last + 128 (= 18*nb when 64 divides nb). */
/* ---------------------------------------------------------------------- */
int64_t orc_q4_0_seg_row_bytes(int64_t K)
{
    const int64_t nb = K / QK;
    const int64_t nseg = (nb + 63) / 64;
    const int64_t r_last = nb - 64 * (nseg - 1);
    return 1152 * (nseg - 1) + 16 * r_last + 128;
}

void orc_repack_q4_0_seg(const uint8_t* W, int64_t O, int64_t K, uint8_t* out)
{
    const int64_t nb = K / QK;
    const int64_t nseg = (nb + 63) / 64;
    const int64_t rb = orc_q4_0_seg_row_bytes(K);
    for (int64_t o = 0; o < O; ++o) {
        const uint8_t* row = W + o * nb * 18;
        uint8_t* dst = out + o * rb;
        for (int64_t s = 0; s < nseg; ++s) {
            const int64_t first = 64 * s;
            const int64_t r = (nb - first < 64) ? nb - first : 64;
            uint8_t* seg = dst + 1152 * s;
            for (int64_t i = 0; i < r; ++i)
                memcpy(seg + 16 * i, row + (first + i) * 18 + 2, 16);
            uint8_t* words = seg + 16 * r;
            for (int l = 0; l < 32; ++l) {
                uint16_t lo = 0, hi = 0;
                if (l < r)
                    lo = rd_u16(row + (first + l) * 18);
                if (32 + l < r)
                    hi = rd_u16(row + (first + 32 + l) * 18);
                wr_u16(words + 4 * l, lo);
                wr_u16(words + 4 * l + 2, hi);
            }
        }
    }
}

/* Element j (0..31) of a Q4_0 block, as the code q in 0..15. */
static int q4_code(const uint8_t* blk, int j)
{
    uint8_t byte = blk[2 + (j & 15)];
    return j < 16 ? (byte & 0x0F) : (byte >> 4);
}

/* ---------------------------------------------------------------------- */
/* RMS statistic s = 1 / sqrt(mean(x^2) + eps)  (fp32).                     */
/*                                                                          */
/* fp32 sums depend on their order, and bit-exact quantized activations     */
/* need one fixed order.  This library fixes it as follows:                 */
/*   partial[j], j = 0..255: x_i^2 accumulated with fused multiply-add over */
/*     i = j, j+256, j+512, ... in ascending order, starting from 0;        */
/*   the 256 partials form 8 groups of 32; within a group, five rounds of   */
/*     pairwise sums t[l] <- t[l] + t[l xor h] for h = 16, 8, 4, 2, 1 leave  */
/*     the group total in t[0];                                             */
/*   ss = ((g0+g1)+(g2+g3)) + ((g4+g5)+(g6+g7));                             */
/*   mean = ss / K, s = 1 / sqrt(mean + eps), each one IEEE fp32 operation. */
/* ---------------------------------------------------------------------- */
float orc_rms_scale(const float* x, int64_t K, float eps)
{
    float partial[256];
    for (int j = 0; j < 256; ++j) {
        float acc = 0.0f;
        for (int64_t i = j; i < K; i += 256)
            acc = fmaf(x[i], x[i], acc);
        partial[j] = acc;
    }
    float g[8];
    for (int grp = 0; grp < 8; ++grp) {
        float t[32], u[32];
        for (int l = 0; l < 32; ++l)
            t[l] = partial[grp * 32 + l];
        for (int h = 16; h >= 1; h >>= 1) {
            for (int l = 0; l < 32; ++l)
                u[l] = t[l] + t[l ^ h];
            for (int l = 0; l < 32; ++l)
                t[l] = u[l];
        }
        g[grp] = t[0];
    }
    float ss = ((g[0] + g[1]) + (g[2] + g[3])) + ((g[4] + g[5]) + (g[6] + g[7]));
    float mean = ss / (float)K;
    float denom = sqrtf(mean + eps);
    return 1.0f / denom;
}

/* ---------------------------------------------------------------------- */
/* Activation -> Q8_0, optionally through RMS_NORM then MUL by gamma, and  */
/* optionally an ADD after them (the RMS_NORM+MUL+ADD fusion pattern of     */
/* [llama.cpp b10909: Metal backend fusion-table refactor, "CI and related  */
/* fixes"]):                                                                */
/*  gamma != NULL: v_i = (x_i * s) * gamma_i   (two fp32 products, in that   */
/*                 order: normalise, then multiply)                         */
/*  gamma == NULL: v_i = x_i (plain quantization, no norm)                   */
/*  add != NULL:   v_i = v_i + a_i, one fp32 addition after the above, with  */
/*                 a = add + n * ldadd for vector n (ldadd 0: one addend     */
/*                 for every vector); the norm statistic is over x alone.   */
/* Per block: amax = max |v|, d = amax / 127 (fp32), q = round(v / d) with   */
/* halves away from zero, clamped to [-127, 127]; d == 0 gives q = 0; the   */
/* stored scale is fp16(d), round to nearest even.                          */
/* x is [N][ldx] (row n = one vector); xq is [N][K/32] blocks.              */
/* ---------------------------------------------------------------------- */
void orc_quantize_q8_0_add(const float* x, int64_t ldx, const float* gamma, const float* add, int64_t ldadd,
                           float eps, int64_t K, int64_t N, uint8_t* xq)
{
    const int64_t nb = K / QK;
    for (int64_t n = 0; n < N; ++n) {
        const float* xn = x + n * ldx;
        const float* an = add ? add + n * ldadd : NULL;
        float s = gamma ? orc_rms_scale(xn, K, eps) : 1.0f;
        for (int64_t b = 0; b < nb; ++b) {
            float v[QK];
            for (int j = 0; j < QK; ++j) {
                int64_t i = b * QK + j;
                if (gamma) {
                    float t = xn[i] * s;
                    v[j] = t * gamma[i];
                } else {
                    v[j] = xn[i];
                }
                if (an)
                    v[j] = v[j] + an[i];
            }
            float amax = 0.0f;
            for (int j = 0; j < QK; ++j)
                if (fabsf(v[j]) > amax)
                    amax = fabsf(v[j]);
            float d = amax / 127.0f;
            uint8_t* blk = xq + (n * nb + b) * 34;
            wr_u16(blk, orc_f32_to_f16(d));
            for (int j = 0; j < QK; ++j) {
                int q = 0;
                if (d != 0.0f) {
                    float r = roundf(v[j] / d);
                    if (r > 127.0f) r = 127.0f;
                    if (r < -127.0f) r = -127.0f;
                    q = (int)r;
                }
                blk[2 + j] = (uint8_t)(int8_t)q;
            }
        }
    }
}

void orc_quantize_q8_0(const float* x, int64_t ldx, const float* gamma, float eps,
                       int64_t K, int64_t N, uint8_t* xq)
{
    orc_quantize_q8_0_add(x, ldx, gamma, NULL, 0, eps, K, N, xq);
}

/* ---------------------------------------------------------------------- */
/* Exact per-block integer sums isum[n][o][b] = sum_j (qw_j - 8) * qx_j.     */
/* ---------------------------------------------------------------------- */
void orc_block_sums(const uint8_t* W, const uint8_t* xq, int64_t O, int64_t K, int64_t N,
                    int32_t* isum)
{
    const int64_t nb = K / QK;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t o = 0; o < O; ++o)
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t* wb = W + (o * nb + b) * 18;
                const uint8_t* xb = xq + (n * nb + b) * 34;
                int32_t acc = 0;
                for (int j = 0; j < QK; ++j)
                    acc += (q4_code(wb, j) - 8) * (int32_t)(int8_t)xb[2 + j];
                isum[(n * O + o) * nb + b] = acc;
            }
}

/* ---------------------------------------------------------------------- */
/* Reference product: dequantize both operands and take the dot product in  */
/* fp64:  y[n][o] = sum_b sum_j (d_w * (qw_j - 8)) * (d_x * qx_j).           */
/* Each term is exact in fp64 (11+4 by 11+8 significant bits), so y64 is     */
/* the exact value up to fp64 summation rounding; y32 = (float)y64.          */
/* S[n][o] = sum_b |d_w * d_x * isum_b| is the magnitude that scales the     */
/* output tolerance.                                                        */
/* rows: optional list of nrows row indices to evaluate (NULL = all O).     */
/* Outputs are [N][nrows].                                                  */
/* ---------------------------------------------------------------------- */
void orc_matvec(const uint8_t* W, const uint8_t* xq, int64_t O, int64_t K, int64_t N,
                const int64_t* rows, int64_t nrows, float* y32, double* y64, double* S)
{
    const int64_t nb = K / QK;
    if (!rows)
        nrows = O;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t t = 0; t < nrows; ++t) {
            int64_t o = rows ? rows[t] : t;
            double acc = 0.0, mag = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t* wb = W + (o * nb + b) * 18;
                const uint8_t* xb = xq + (n * nb + b) * 34;
                double dw = (double)orc_f16_to_f32(rd_u16(wb));
                double dx = (double)orc_f16_to_f32(rd_u16(xb));
                double blk = 0.0;
                int64_t isum = 0;
                for (int j = 0; j < QK; ++j) {
                    double wv = dw * (double)(q4_code(wb, j) - 8);
                    double xv = dx * (double)(int8_t)xb[2 + j];
                    blk += wv * xv;
                    isum += (int64_t)(q4_code(wb, j) - 8) * (int64_t)(int8_t)xb[2 + j];
                }
                acc += blk;
                mag += fabs(dw * dx * (double)isum);
            }
            if (y32) y32[n * nrows + t] = (float)acc;
            if (y64) y64[n * nrows + t] = acc;
            if (S) S[n * nrows + t] = mag;
        }
    }
}

/* ---------------------------------------------------------------------- */
/* Q8_0 weights.  The stack's conversion step picks the weight type, Q4_K or */
/* Q8_0, and every back end's kernels must know each type  [GGML: Backend    */
/* abstraction and hardware acceleration, sections "How one production call */
/* lands on the hardware" and "Metal and Vulkan"].  A Q8_0 weight row is K/32 */
/* Q8_0 blocks (the activation format above, made by the same quantizer with */
/* no norm); the product takes per block the exact integer sum               */
/* isum = sum_j qw_j * qx_j (both signed) and y = sum_b d_w * d_x * isum_b.   */
/* ---------------------------------------------------------------------- */
void orc_block_sums_q8w(const uint8_t* W, const uint8_t* xq, int64_t O, int64_t K, int64_t N,
                        int32_t* isum)
{
    const int64_t nb = K / QK;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t o = 0; o < O; ++o)
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t* wb = W + (o * nb + b) * 34;
                const uint8_t* xb = xq + (n * nb + b) * 34;
                int32_t acc = 0;
                for (int j = 0; j < QK; ++j)
                    acc += (int32_t)(int8_t)wb[2 + j] * (int32_t)(int8_t)xb[2 + j];
                isum[(n * O + o) * nb + b] = acc;
            }
}

/* Reference product for Q8_0 weights, as orc_matvec: dequantize both operands */
/* and take the dot product in fp64 (every term exact); S as there.            */
void orc_matvec_q8w(const uint8_t* W, const uint8_t* xq, int64_t O, int64_t K, int64_t N,
                    const int64_t* rows, int64_t nrows, float* y32, double* y64, double* S)
{
    const int64_t nb = K / QK;
    if (!rows)
        nrows = O;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t t = 0; t < nrows; ++t) {
            int64_t o = rows ? rows[t] : t;
            double acc = 0.0, mag = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t* wb = W + (o * nb + b) * 34;
                const uint8_t* xb = xq + (n * nb + b) * 34;
                double dw = (double)orc_f16_to_f32(rd_u16(wb));
                double dx = (double)orc_f16_to_f32(rd_u16(xb));
                double blk = 0.0;
                int64_t isum = 0;
                for (int j = 0; j < QK; ++j) {
                    double wv = dw * (double)(int8_t)wb[2 + j];
                    double xv = dx * (double)(int8_t)xb[2 + j];
                    blk += wv * xv;
                    isum += (int64_t)(int8_t)wb[2 + j] * (int64_t)(int8_t)xb[2 + j];
                }
                acc += blk;
                mag += fabs(dw * dx * (double)isum);
            }
            if (y32) y32[n * nrows + t] = (float)acc;
            if (y64) y64[n * nrows + t] = acc;
            if (S) S[n * nrows + t] = mag;
        }
    }
}

/* ---------------------------------------------------------------------- */
/* Q4_K weights.  The conversion step picks Q4_K for weights [GGML: Backend */
/* abstraction and hardware acceleration, section "How one production call */
/* lands on the hardware"], but the pages give no block format.  The        */
/* library reads it as GGML's k-quant super-block of 256 weights (8 sub-     */
/* blocks of 32), 144 bytes:                                                */
/*   bytes 0-1   fp16 d    (multiplies the sub-block scales)                */
/*   bytes 2-3   fp16 dmin (multiplies the sub-block mins)                  */
/*   bytes 4-15  s[0..11]: eight 6-bit scales sc_j and eight 6-bit mins m_j: */
/*                 j < 4:  sc_j = s[j] & 63,          m_j = s[j+4] & 63      */
/*                 j >= 4: sc_j = (s[j+4] & 15) + 16 * (s[j-4] >> 6),        */
/*                         m_j  = (s[j+4] >> 4) + 16 * (s[j] >> 6)           */
/*   bytes 16-143: codes; byte 16 + 32p + i holds element i of sub-block 2p  */
/*                 in its low nibble and element i of sub-block 2p+1 in its  */
/*                 high nibble (p = 0..3, i = 0..31).                        */
/*   Element i of sub-block j = d * sc_j * q - dmin * m_j, q in 0..15.       */
/* A row of K weights (K a multiple of 256) is K/256 super-blocks.          */
/* ---------------------------------------------------------------------- */
static void q4k_scale_min(const uint8_t* blk, int j, int* sc, int* m)
{
    const uint8_t* s = blk + 4;
    if (j < 4) {
        *sc = s[j] & 63;
        *m = s[j + 4] & 63;
    } else {
        *sc = (s[j + 4] & 15) + 16 * (s[j - 4] >> 6);
        *m = (s[j + 4] >> 4) + 16 * (s[j] >> 6);
    }
}

/* Code q (0..15) of element e (0..255) of a super-block. */
static int q4k_code(const uint8_t* blk, int e)
{
    int j = e / 32, i = e % 32;
    uint8_t byte = blk[16 + 32 * (j / 2) + i];
    return (j % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
}

static int round_half_away_clamp(float v, int lo, int hi)
{
    float r = roundf(v);
    int q = (int)r;
    return q < lo ? lo : (q > hi ? hi : q);
}

/* Q4_K quantization (input preparation; the library's plain reading of the   */
/* k-quant recipe, all fp32 operations):                                      */
/*   sub-block j: lo = min w, hi = max w; mn_j = -lo if lo < 0 else 0;        */
/*     a_j = (hi + mn_j) / 15 (the code step);                                */
/*   D = max_j a_j / 63, Dm = max_j mn_j / 63; stored d = fp16(D),            */
/*     dmin = fp16(Dm); dd, ddm = their fp32 values;                          */
/*   sc_j = round(a_j / dd), m_j = round(mn_j / ddm) (0 when the divisor is 0), */
/*     halves away from zero, clamped to 0..63;                              */
/*   q = round((w + ddm*m_j) / (dd*sc_j)) clamped to 0..15 (0 when the step   */
/*     dd*sc_j is 0).                                                         */
void orc_quantize_q4_k(const float* w, int64_t rows, int64_t K, uint8_t* out)
{
    const int64_t nsb = K / 256;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t sb = 0; sb < nsb; ++sb) {
            const float* v = w + r * K + sb * 256;
            uint8_t* blk = out + (r * nsb + sb) * 144;
            float a[8], mn[8], amax = 0.0f, mnmax = 0.0f;
            for (int j = 0; j < 8; ++j) {
                float lo = v[32 * j], hi = v[32 * j];
                for (int i = 1; i < 32; ++i) {
                    if (v[32 * j + i] < lo) lo = v[32 * j + i];
                    if (v[32 * j + i] > hi) hi = v[32 * j + i];
                }
                mn[j] = lo < 0.0f ? -lo : 0.0f;
                a[j] = (hi + mn[j]) / 15.0f;
                if (a[j] > amax) amax = a[j];
                if (mn[j] > mnmax) mnmax = mn[j];
            }
            uint16_t dh = orc_f32_to_f16(amax / 63.0f), dmh = orc_f32_to_f16(mnmax / 63.0f);
            float dd = orc_f16_to_f32(dh), ddm = orc_f16_to_f32(dmh);
            int sc[8], m[8];
            for (int j = 0; j < 8; ++j) {
                sc[j] = dd > 0.0f ? round_half_away_clamp(a[j] / dd, 0, 63) : 0;
                m[j] = ddm > 0.0f ? round_half_away_clamp(mn[j] / ddm, 0, 63) : 0;
            }
            memset(blk, 0, 144);
            wr_u16(blk, dh);
            wr_u16(blk + 2, dmh);
            uint8_t* s = blk + 4;
            for (int j = 0; j < 4; ++j) {
                s[j] = (uint8_t)((sc[j] & 63) | ((sc[j + 4] >> 4) << 6));
                s[j + 4] = (uint8_t)((m[j] & 63) | ((m[j + 4] >> 4) << 6));
                s[j + 8] = (uint8_t)((sc[j + 4] & 15) | ((m[j + 4] & 15) << 4));
            }
            for (int j = 0; j < 8; ++j) {
                float step = dd * (float)sc[j];
                float off = ddm * (float)m[j];
                for (int i = 0; i < 32; ++i) {
                    int q = 0;
                    if (step > 0.0f) {
                        float t = v[32 * j + i] + off;
                        q = round_half_away_clamp(t / step, 0, 15);
                    }
                    uint8_t* byte = blk + 16 + 32 * (j / 2) + i;
                    *byte = (uint8_t)((j % 2 == 0) ? ((*byte & 0xF0) | q) : ((*byte & 0x0F) | (q << 4)));
                }
            }
        }
    }
}

/* Dequantized weights in fp64 (every value d*sc*q - dmin*m is exact there). */
void orc_dequantize_q4_k(const uint8_t* W, int64_t rows, int64_t K, double* out)
{
    const int64_t nsb = K / 256;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t sb = 0; sb < nsb; ++sb) {
            const uint8_t* blk = W + (r * nsb + sb) * 144;
            double d = (double)orc_f16_to_f32(rd_u16(blk)), dmin = (double)orc_f16_to_f32(rd_u16(blk + 2));
            for (int e = 0; e < 256; ++e) {
                int sc, m;
                q4k_scale_min(blk, e / 32, &sc, &m);
                out[r * K + sb * 256 + e] = d * (double)sc * (double)q4k_code(blk, e) - dmin * (double)m;
            }
        }
}

/* Exact integer sums per 32-weight sub-block (= per Q8_0 block of the      */
/* activations): isum[n][o][b] = sum_i q_i * qx_i (codes 0..15 times int8).  */
void orc_block_sums_q4k(const uint8_t* W, const uint8_t* xq, int64_t O, int64_t K, int64_t N, int32_t* isum)
{
    const int64_t nb = K / QK, nsb = K / 256;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t o = 0; o < O; ++o)
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t* blk = W + (o * nsb + b / 8) * 144;
                const uint8_t* xb = xq + (n * nb + b) * 34;
                int32_t acc = 0;
                for (int i = 0; i < QK; ++i)
                    acc += q4k_code(blk, (int)(b % 8) * 32 + i) * (int32_t)(int8_t)xb[2 + i];
                isum[(n * O + o) * nb + b] = acc;
            }
}

/* Reference product for Q4_K weights: dequantize both operands, dot product */
/* in fp64.  S[n][o] = sum over sub-blocks b of                             */
/*   |d_x * d * sc_b * isum_b| + |d_x * dmin * m_b * xsum_b|                 */
/* (xsum_b = sum of the activation codes), the magnitude of the two terms    */
/* each sub-block contributes; it scales the output tolerance.              */
void orc_matvec_q4k(const uint8_t* W, const uint8_t* xq, int64_t O, int64_t K, int64_t N,
                    const int64_t* rows, int64_t nrows, float* y32, double* y64, double* S)
{
    const int64_t nb = K / QK, nsb = K / 256;
    if (!rows)
        nrows = O;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t t = 0; t < nrows; ++t) {
            int64_t o = rows ? rows[t] : t;
            double acc = 0.0, mag = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t* blk = W + (o * nsb + b / 8) * 144;
                const uint8_t* xb = xq + (n * nb + b) * 34;
                double d = (double)orc_f16_to_f32(rd_u16(blk)), dmin = (double)orc_f16_to_f32(rd_u16(blk + 2));
                double dx = (double)orc_f16_to_f32(rd_u16(xb));
                int sc, m;
                q4k_scale_min(blk, (int)(b % 8), &sc, &m);
                double sub = 0.0;
                int64_t isum = 0, xsum = 0;
                for (int i = 0; i < QK; ++i) {
                    int q = q4k_code(blk, (int)(b % 8) * 32 + i);
                    int qx = (int8_t)xb[2 + i];
                    double wv = d * (double)sc * (double)q - dmin * (double)m;
                    sub += wv * (dx * (double)qx);
                    isum += (int64_t)q * qx;
                    xsum += qx;
                }
                acc += sub;
                mag += fabs(dx * d * (double)sc * (double)isum) + fabs(dx * dmin * (double)m * (double)xsum);
            }
            if (y32) y32[n * nrows + t] = (float)acc;
            if (y64) y64[n * nrows + t] = acc;
            if (S) S[n * nrows + t] = mag;
        }
    }
}

/* ---------------------------------------------------------------------- */
/* Q5_K weights.  The pages name Q5_K beside Q4_K (the GPU MoE tests compare */
/* Q4_K/Q5_K results [llama.cpp b10981: OpenVINO backend optimises stateful */
/* decode and GPU MoE inference, section "GPU MoE, env vars"]) but give no  */
/* format.  The library reads it as GGML's 5-bit k-quant super-block of 256  */
/* weights (8 sub-blocks of 32), 176 bytes:                                 */
/*   bytes 0-15    as in Q4_K: fp16 d, fp16 dmin, the twelve bytes of 6-bit  */
/*                 scales sc_j and mins m_j (same packing);                 */
/*   bytes 16-47   qh[0..31]: bit j of qh[i] is the top bit (value 16) of    */
/*                 element i of sub-block j;                                */
/*   bytes 48-175  the low four bits, placed as the Q4_K codes: byte         */
/*                 48 + 32p + i holds element i of sub-block 2p in its low   */
/*                 nibble and element i of sub-block 2p+1 in its high one.   */
/*   Element i of sub-block j = d * sc_j * q - dmin * m_j, q in 0..31.       */
/* ---------------------------------------------------------------------- */
static int q5k_code(const uint8_t* blk, int e)
{
    int sub = e / 32, i = e % 32;
    uint8_t low4 = blk[48 + 32 * (sub / 2) + i];
    int lo = (sub % 2 == 0) ? (low4 & 0x0F) : (low4 >> 4);
    return lo + 16 * ((blk[16 + i] >> sub) & 1);
}

/* Q5_K quantization: the Q4_K recipe above with 31 code steps per sub-block */
/* (a_j = (hi + mn_j) / 31; q clamped to 0..31), every step one fp32         */
/* operation.                                                               */
void orc_quantize_q5_k(const float* w, int64_t rows, int64_t K, uint8_t* out)
{
    const int64_t nsb = K / 256;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t sb = 0; sb < nsb; ++sb) {
            const float* v = w + r * K + sb * 256;
            uint8_t* blk = out + (r * nsb + sb) * 176;
            float step5[8], off5[8], a5[8], mn5[8], amax5 = 0.0f, mnmax5 = 0.0f;
            for (int j = 0; j < 8; ++j) {
                float lo = v[32 * j], hi = v[32 * j];
                for (int i = 1; i < 32; ++i) {
                    if (v[32 * j + i] < lo) lo = v[32 * j + i];
                    if (v[32 * j + i] > hi) hi = v[32 * j + i];
                }
                mn5[j] = lo < 0.0f ? -lo : 0.0f;
                a5[j] = (hi + mn5[j]) / 31.0f;
                if (a5[j] > amax5) amax5 = a5[j];
                if (mn5[j] > mnmax5) mnmax5 = mn5[j];
            }
            uint16_t dh = orc_f32_to_f16(amax5 / 63.0f), dmh = orc_f32_to_f16(mnmax5 / 63.0f);
            float dd = orc_f16_to_f32(dh), ddm = orc_f16_to_f32(dmh);
            int sc5[8], m5[8];
            for (int j = 0; j < 8; ++j) {
                sc5[j] = dd > 0.0f ? round_half_away_clamp(a5[j] / dd, 0, 63) : 0;
                m5[j] = ddm > 0.0f ? round_half_away_clamp(mn5[j] / ddm, 0, 63) : 0;
                step5[j] = dd * (float)sc5[j];
                off5[j] = ddm * (float)m5[j];
            }
            memset(blk, 0, 176);
            wr_u16(blk, dh);
            wr_u16(blk + 2, dmh);
            uint8_t* s = blk + 4;
            for (int j = 0; j < 4; ++j) {
                s[j] = (uint8_t)((sc5[j] & 63) | ((sc5[j + 4] >> 4) << 6));
                s[j + 4] = (uint8_t)((m5[j] & 63) | ((m5[j + 4] >> 4) << 6));
                s[j + 8] = (uint8_t)((sc5[j + 4] & 15) | ((m5[j + 4] & 15) << 4));
            }
            for (int j = 0; j < 8; ++j) {
                for (int i = 0; i < 32; ++i) {
                    int q5 = 0;
                    if (step5[j] > 0.0f)
                        q5 = round_half_away_clamp((v[32 * j + i] + off5[j]) / step5[j], 0, 31);
                    uint8_t* low = blk + 48 + 32 * (j / 2) + i;
                    *low = (uint8_t)((j % 2 == 0) ? ((*low & 0xF0) | (q5 & 15)) : ((*low & 0x0F) | ((q5 & 15) << 4)));
                    blk[16 + i] = (uint8_t)(blk[16 + i] | ((q5 >> 4) << j));
                }
            }
        }
    }
}

/* Dequantized Q5_K weights in fp64 (exact there). */
void orc_dequantize_q5_k(const uint8_t* W, int64_t rows, int64_t K, double* out)
{
    const int64_t nsb = K / 256;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t sb = 0; sb < nsb; ++sb) {
            const uint8_t* blk = W + (r * nsb + sb) * 176;
            const double dd = (double)orc_f16_to_f32(rd_u16(blk));
            const double ddmin = (double)orc_f16_to_f32(rd_u16(blk + 2));
            for (int e = 0; e < 256; ++e) {
                int scale, mins;
                q4k_scale_min(blk, e / 32, &scale, &mins);
                out[r * K + sb * 256 + e] = dd * (double)scale * (double)q5k_code(blk, e) - ddmin * (double)mins;
            }
        }
}

/* Exact integer sums per 32-weight sub-block: sum_i q_i * qx_i (codes      */
/* 0..31 times int8).                                                        */
void orc_block_sums_q5k(const uint8_t* W, const uint8_t* xq, int64_t O, int64_t K, int64_t N, int32_t* isum)
{
    const int64_t nb = K / QK, nsb = K / 256;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t o = 0; o < O; ++o)
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t* sblk = W + (o * nsb + b / 8) * 176;
                const uint8_t* xblk = xq + (n * nb + b) * 34;
                int32_t total = 0;
                for (int i = 0; i < QK; ++i)
                    total += q5k_code(sblk, (int)(b % 8) * 32 + i) * (int32_t)(int8_t)xblk[2 + i];
                isum[(n * O + o) * nb + b] = total;
            }
}

/* Reference product for Q5_K weights, as orc_matvec_q4k: fp64 dot product  */
/* of the dequantized operands; S = sum over sub-blocks of                  */
/* |d_x d sc isum| + |d_x dmin m xsum|.                                      */
void orc_matvec_q5k(const uint8_t* W, const uint8_t* xq, int64_t O, int64_t K, int64_t N,
                    const int64_t* rows, int64_t nrows, float* y32, double* y64, double* S)
{
    const int64_t nb = K / QK, nsb = K / 256;
    if (!rows)
        nrows = O;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t t = 0; t < nrows; ++t) {
            int64_t o = rows ? rows[t] : t;
            double total = 0.0, bound = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t* sblk = W + (o * nsb + b / 8) * 176;
                const uint8_t* xblk = xq + (n * nb + b) * 34;
                const double dd = (double)orc_f16_to_f32(rd_u16(sblk));
                const double ddmin = (double)orc_f16_to_f32(rd_u16(sblk + 2));
                const double dx = (double)orc_f16_to_f32(rd_u16(xblk));
                int scale, mins;
                q4k_scale_min(sblk, (int)(b % 8), &scale, &mins);
                double part = 0.0;
                int64_t qsum = 0, xsum = 0;
                for (int i = 0; i < QK; ++i) {
                    const int q5 = q5k_code(sblk, (int)(b % 8) * 32 + i);
                    const int qx = (int8_t)xblk[2 + i];
                    part += (dd * (double)scale * (double)q5 - ddmin * (double)mins) * (dx * (double)qx);
                    qsum += (int64_t)q5 * qx;
                    xsum += qx;
                }
                total += part;
                bound += fabs(dx * dd * (double)scale * (double)qsum) + fabs(dx * ddmin * (double)mins * (double)xsum);
            }
            if (y32) y32[n * nrows + t] = (float)total;
            if (y64) y64[n * nrows + t] = total;
            if (S) S[n * nrows + t] = bound;
        }
    }
}
