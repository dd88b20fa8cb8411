/*
 * CPU oracle for the quantized-weight prefill GEMM.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this library.  The CUDA path never links, calls or reads it, and it
 * shares no code, header, table or constant with the CUDA path.
 *
 * What it computes is the plain definition of the method:
 *   1. decode every stored number exactly (IEEE binary16 / bfloat16 -> double),
 *   2. dequantize each weight exactly in double precision,
 *   3. y[m][n] = sum_k x[m][k] * w[n][k] with a naive double loop, and the
 *      companion magnitude a[m][n] = sum_k |x[m][k] * w[n][k]| used by the
 *      error bound |y_gpu - y| <= 1e-3 * a + 1e-5.
 *
 * Sources (web pages, by title and section):
 *  - "The dequant scratch round-trip is ZINC's last RDNA4 prefill tax",
 *    section "The two passes hiding inside one matmul": a Q4_K weight costs
 *    0.5625 byte, i.e. 144 bytes per 256-weight super-block.
 *  - "How ZINC's RDNA4 batched prefill went from 42 to 208 tok/s", section
 *    "The fix: K-parallel batched DMMV": each decoded stripe is
 *    factor * q - bias, and the low and high nibbles of one byte are 32
 *    elements apart (by0/by1 and q0_lo/q0_hi).
 *  - The GGML Q4_K block named by the workload definition: fp16 d, fp16
 *    dmin, 12 bytes of packed 6-bit scales[8]/mins[8], 128 bytes of nibbles;
 *    w = d * sc_j * q - dmin * m_j.  The bit packing of the 6-bit values is
 *    GGML's (not printed on the pages): values 0..3 are the low six bits of
 *    bytes 0..3 (scales) and 4..7 (mins); values 4..7 take their low four
 *    bits from bytes 8..11 (scale: low nibble, min: high nibble) and their
 *    top two bits from the top two bits of bytes 0..3 (scales) and 4..7
 *    (mins).
 *  - "[ROCm][Perf] W4A16: packed fp16 prefill dequant", section "1. Packed
 *    fp16 dequant": an int32 holds val[2p] at bits 4p..4p+3 and val[2p+1] at
 *    bits 16+4p..19+4p (p = 0..3); w = s * (q - zp); section "2." keeps a
 *    K-block inside one quantisation group (groups run along K); the
 *    measurements table and "Duplicate-work check" name a symmetric variant
 *    without zero points (read here as zp = 8).
 *  - "How ZINC's RDNA4 batched prefill went from 42 to 208 tok/s", sections
 *    "Bug 2: Q6_K had a gate but no dispatcher" and "What changed": Q4_K_M
 *    checkpoints keep ffn_down and attn_v in Q6_K, and the batched path needs
 *    a Q6_K kernel beside the Q4_K one.  The pages name the format but do not
 *    print it; the oracle follows the GGML Q6_K block (parity partly
 *    unpinned): 256 weights in 210 bytes -- ql[128] (low four bits), qh[64]
 *    (high two bits), int8 scales[16] (one per 16 weights), fp16 d last;
 *    w = d * scale * (q - 32) with q the 6-bit code.
 *  - "The dequant scratch round-trip is ZINC's last RDNA4 prefill tax",
 *    section "What removing it was worth": the DP4a path quantizes the
 *    activations first (Q8_1: 8-bit codes per block of 32 with a scale) and
 *    multiplies them, still packed, with the 4-bit weights.  The pages give no
 *    rounding rule; the one taken here (GGML's Q8_1 rule, with the scale kept
 *    in fp32 and an exact integer block sum) is in oracle_q8_quantize.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_SHAPE (-1)
#define ORACLE_ERR_NONFINITE (-2)
#define ORACLE_ERR_RANGE (-3)

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);              /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);  /* (1 + f/2^10) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_bf16_to_double(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 255;
    int f = b & 127;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);             /* subnormal: f * 2^-126 * 2^-7 */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + f), e - 134);  /* (1 + f/2^7) * 2^(e-127) */
    return sign ? -v : v;
}

int oracle_half_array_to_double(const uint16_t *src, int64_t n, double *dst)
{
    int status = ORACLE_OK;
    for (int64_t i = 0; i < n; ++i) {
        dst[i] = oracle_half_to_double(src[i]);
        if (!isfinite(dst[i]))
            status = ORACLE_ERR_NONFINITE;  /* flagged; the value is still written */
    }
    return status;
}

int oracle_bf16_array_to_double(const uint16_t *src, int64_t n, double *dst)
{
    int status = ORACLE_OK;
    for (int64_t i = 0; i < n; ++i) {
        dst[i] = oracle_bf16_to_double(src[i]);
        if (!isfinite(dst[i]))
            status = ORACLE_ERR_NONFINITE;  /* flagged; the value is still written */
    }
    return status;
}

/* The 6-bit scale sc_j and min m_j of sub-block j (0..7) from the 12 packed bytes. */
void oracle_q4k_scale_min(const uint8_t *s, int j, int *sc, int *m)
{
    if (j < 4) {
        *sc = s[j] & 63;
        *m = s[j + 4] & 63;
    } else {
        *sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
        *m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

/*
 * Dequantize N rows of K weights stored as GGML Q4_K super-blocks
 * (row n, super-block b at byte offset (n*(K/256) + b) * 144) into w[N][K].
 */
int oracle_q4k_dequant(const uint8_t *blocks, int64_t N, int64_t K, double *w)
{
    if (N < 0 || K < 0 || K % 256 != 0)
        return ORACLE_ERR_SHAPE;
    const int64_t nb = K / 256;
    int status = ORACLE_OK;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t *blk = blocks + (n * nb + b) * 144;
            double d = oracle_half_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
            double dmin = oracle_half_to_double((uint16_t)(blk[2] | (blk[3] << 8)));
            if (!isfinite(d) || !isfinite(dmin)) {
                status = ORACLE_ERR_NONFINITE;
                continue;
            }
            const uint8_t *s = blk + 4;
            const uint8_t *qs = blk + 16;
            double *row = w + n * K + b * 256;
            for (int c = 0; c < 4; ++c) {
                int sc_lo, m_lo, sc_hi, m_hi;
                oracle_q4k_scale_min(s, 2 * c, &sc_lo, &m_lo);
                oracle_q4k_scale_min(s, 2 * c + 1, &sc_hi, &m_hi);
                for (int l = 0; l < 32; ++l) {
                    int q_lo = qs[32 * c + l] & 15;  /* element 64c + l,      sub-block 2c   */
                    int q_hi = qs[32 * c + l] >> 4;  /* element 64c + 32 + l, sub-block 2c+1 */
                    row[64 * c + l] = d * sc_lo * q_lo - dmin * m_lo;
                    row[64 * c + 32 + l] = d * sc_hi * q_hi - dmin * m_hi;
                }
            }
        }
    }
    return status;
}

/*
 * The 6-bit code of element e (0..255) of one GGML Q6_K block.  The block is
 * two halves of 128 elements; in half h, element 32*j + l (j = 0..3,
 * l = 0..31) takes its low four bits from byte 64*h + l + 32*(j % 2) of ql
 * (the low nibble for j < 2, the high nibble for j >= 2) and its high two
 * bits from bits 2j..2j+1 of byte 32*h + l of qh.
 */
int oracle_q6k_code(const uint8_t *blk, int e)
{
    const uint8_t *ql = blk, *qh = blk + 128;
    int h = e / 128, j = (e % 128) / 32, l = e % 32;
    int lo_byte = ql[64 * h + l + 32 * (j % 2)];
    int lo = (j < 2) ? (lo_byte & 15) : (lo_byte >> 4);
    int hi = (qh[32 * h + l] >> (2 * j)) & 3;
    return lo | (hi << 4);
}

/*
 * Dequantize N rows of K weights stored as GGML Q6_K blocks (row n, block b
 * at byte offset (n*(K/256) + b) * 210) into w[N][K]: element e of a block is
 * d * scales[e / 16] * (q_e - 32).
 */
int oracle_q6k_dequant(const uint8_t *blocks, int64_t N, int64_t K, double *w)
{
    if (N < 0 || K < 0 || K % 256 != 0)
        return ORACLE_ERR_SHAPE;
    const int64_t nb = K / 256;
    int status = ORACLE_OK;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t *blk = blocks + (n * nb + b) * 210;
            const int8_t *scales = (const int8_t *)(blk + 192);
            double d = oracle_half_to_double((uint16_t)(blk[208] | (blk[209] << 8)));
            if (!isfinite(d)) {
                status = ORACLE_ERR_NONFINITE;
                continue;
            }
            double *row = w + n * K + b * 256;
            for (int e = 0; e < 256; ++e)
                row[e] = d * (double)scales[e / 16] * (double)(oracle_q6k_code(blk, e) - 32);
        }
    }
    return status;
}

/*
 * Dequantize group-wise 4-bit weights: wq[N][K/8] int32 words in the
 * interleaved order, scales[N][K/group] fp16 bits, zeros[N][K/group] in 0..15
 * (asymmetric), or zeros == NULL for the symmetric form, whose zero point is
 * the middle code 8 (the pages name a symmetric path with no zero points;
 * centring the unsigned 4-bit code at 8 is the reading taken here).
 */
int oracle_w4a16_dequant(const uint32_t *wq, const uint16_t *scales, const uint8_t *zeros,
                         int64_t N, int64_t K, int64_t group, double *w)
{
    if (N < 0 || K < 0 || group <= 0 || K % 8 != 0 || K % group != 0)
        return ORACLE_ERR_SHAPE;
    const int64_t ng = K / group;
    int status = ORACLE_OK;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t i = 0; i < K / 8; ++i) {
            uint32_t word = wq[n * (K / 8) + i];
            for (int t = 0; t < 8; ++t) {
                int p = t / 2;
                int shift = (t % 2 == 0) ? 4 * p : 16 + 4 * p;
                int q = (int)((word >> shift) & 15u);
                int64_t k = 8 * i + t;
                int64_t g = k / group;
                double s = oracle_half_to_double(scales[n * ng + g]);
                int z = zeros ? zeros[n * ng + g] : 8;
                if (!isfinite(s))
                    status = ORACLE_ERR_NONFINITE;
                if (z > 15)
                    status = ORACLE_ERR_RANGE;
                w[n * K + k] = s * (double)(q - z);
            }
        }
    }
    return status;
}

/*
 * The two terms of every Q4_K weight, w = a - b with a = d * sc_j * q and
 * b = dmin * m_j (both exact in double), for the error bound of products whose
 * arithmetic keeps the terms apart.  Same layout and checks as oracle_q4k_dequant.
 */
int oracle_q4k_terms(const uint8_t *blocks, int64_t N, int64_t K, double *a, double *b)
{
    if (N < 0 || K < 0 || K % 256 != 0)
        return ORACLE_ERR_SHAPE;
    const int64_t nb = K / 256;
    int status = ORACLE_OK;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t blk_i = 0; blk_i < nb; ++blk_i) {
            const uint8_t *blk = blocks + (n * nb + blk_i) * 144;
            double d = oracle_half_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
            double dmin = oracle_half_to_double((uint16_t)(blk[2] | (blk[3] << 8)));
            if (!isfinite(d) || !isfinite(dmin)) {
                status = ORACLE_ERR_NONFINITE;
                continue;
            }
            for (int e = 0; e < 256; ++e) {
                int c = e / 64, hi = (e % 64) / 32, l = e % 32;
                int sc, m;
                oracle_q4k_scale_min(blk + 4, 2 * c + hi, &sc, &m);
                int qv = hi ? (blk[16 + 32 * c + l] >> 4) : (blk[16 + 32 * c + l] & 15);
                a[n * K + blk_i * 256 + e] = d * sc * qv;
                b[n * K + blk_i * 256 + e] = dmin * m;
            }
        }
    }
    return status;
}

/*
 * Activation quantization: each token row of x ([M][K] bfloat16 bits) is cut
 * into blocks of 32 along K.  Block j of row m gets
 *     d = RN32(amax / 127),  amax = the largest |x| of the block (exact in fp32),
 *     q = round-half-away-from-zero(RN32(x * RN32(1 / d)))  (q = 0 when d == 0),
 *     s = the sum of the block's 32 codes (exact),
 * every step in IEEE single precision, as written (GGML's Q8_1 rule; the scale
 * is kept in fp32 rather than rounded to fp16, and the sum as an integer).
 * q[M][K] int8, d[M][K/32] fp32, s[M][K/32] int32.  A non-finite x is rejected.
 */
int oracle_q8_quantize(const uint16_t *x, int64_t M, int64_t K, int8_t *q, float *d, int32_t *s)
{
    if (M < 0 || K < 0 || K % 32 != 0)
        return ORACLE_ERR_SHAPE;
    for (int64_t i = 0; i < M * K; ++i)
        if (!isfinite(oracle_bf16_to_double(x[i])))
            return ORACLE_ERR_NONFINITE;
    const int64_t nbk = K / 32;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t j = 0; j < nbk; ++j) {
            const uint16_t *xb = x + m * K + 32 * j;
            float v[32];
            float amax = 0.0f;
            for (int l = 0; l < 32; ++l) {
                v[l] = (float)oracle_bf16_to_double(xb[l]);  /* exact: bfloat16 is a subset of fp32 */
                if (fabsf(v[l]) > amax)
                    amax = fabsf(v[l]);
            }
            const float dj = amax / 127.0f;
            const float id = dj != 0.0f ? 1.0f / dj : 0.0f;
            int32_t sum = 0;
            for (int l = 0; l < 32; ++l) {
                const float t = v[l] * id;
                const int qi = (int)roundf(t);
                q[m * K + 32 * j + l] = (int8_t)qi;
                sum += qi;
            }
            d[m * nbk + j] = dj;
            s[m * nbk + j] = sum;
        }
    }
    return ORACLE_OK;
}

/*
 * y[m][n] = sum_k x[m][k] * w[n][k];  a[m][n] = sum_k |x[m][k] * w[n][k]|.
 * x is [M][K], w is [N][K], y and a are [M][N]; a may be NULL.
 */
int oracle_gemm(const double *x, const double *w, int64_t M, int64_t N, int64_t K,
                double *y, double *a)
{
    if (M < 0 || N < 0 || K < 0)
        return ORACLE_ERR_SHAPE;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        const double *wr = w + n * K;
        for (int64_t m = 0; m < M; ++m) {
            const double *xr = x + m * K;
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = xr[k] * wr[k];
                acc += p;
                mag += fabs(p);
            }
            y[m * N + n] = acc;
            if (a)
                a[m * N + n] = mag;
        }
    }
    return ORACLE_OK;
}

/* Number of threads the parallel loops above use (1 when built without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
