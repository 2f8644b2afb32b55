/*
 * qmm_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow CPU oracle for the fused-dequantisation quantized matmul.
 * It exists so that the CUDA library can be checked against something
 * obviously correct; nothing on the product path may load it.  Only tests,
 * the smoke check and the benchmark's CPU-baseline leg call it.
 *
 * What it computes (and why this is the right definition):
 *   "Building a Rust Inference Engine That Matches Llama.cpp", sections
 *   "What Ferrox actually is" and "Where the wins came from": quantized
 *   weights are never expanded into a full-precision buffer; the dequant
 *   math happens inline as part of the dot product.  Fusing changes where
 *   the arithmetic happens, not what it is, so the oracle is the plain
 *   definition: decode every weight to its exact real value, then take the
 *   dot product, accumulating in fp64.
 *
 *   The pages name the formats ("Frink Inference: the Rust alternative to
 *   llama.cpp", section "Where llama.cpp is still ahead": Q8_0 and the
 *   K-quants, activations kept in f32) but do not print their layouts.  The
 *   layouts below are the GGUF block formats:
 *     Q4_K super-block, 144 bytes, 256 weights:
 *       [0..1] d (binary16) [2..3] dmin (binary16)
 *       [4..15] twelve bytes holding eight 6-bit scales and eight 6-bit mins
 *       [16..143] 128 bytes of 4-bit quants.
 *       Weight i: chunk c = i/64, l = i%64; l<32 -> low nibble of qs[32c+l]
 *       in sub-block 2c, l>=32 -> high nibble of qs[32c+l-32] in sub-block
 *       2c+1.  w = d*sc_j*q - dmin*m_j.
 *     Q8_0 block, 34 bytes, 32 weights: [0..1] d (binary16), then 32 int8;
 *       w = d*q.
 *   The further formats of the next step ("Frink Inference: the Rust
 *   alternative to llama.cpp", sections "Where llama.cpp is still ahead" --
 *   IQ4_NL -- and "Where Frink is already better than llama.cpp" -- the
 *   other K-quants, written byte-identically), also GGUF block formats:
 *     Q5_K super-block, 176 bytes, 256 weights: d, dmin (binary16), the
 *       twelve scale/min bytes of Q4_K, qh[32] (fifth bits), qs[128] (low
 *       four bits, in the Q4_K nibble order).  Weight i: chunk c = i/64,
 *       l = i%64; the fifth bit is bit (2c + (l >= 32)) of qh[l % 32].
 *       w = d*sc_j*q - dmin*m_j with q in 0..31.
 *     Q6_K super-block, 210 bytes, 256 weights: ql[128] (low four bits),
 *       qh[64] (high two bits), sixteen int8 scales, d (binary16).  Weight
 *       i: half n = i/128, r = i%128, quarter t = r/32, l = r%32; the low
 *       bits are nibble (t >= 2) of ql[64n + 32*(t & 1) + l], the high bits
 *       are bits 2t..2t+1 of qh[32n + l]; q = low | high << 4 (0..63);
 *       w = d * scale[i/16] * (q - 32).
 *     IQ4_NL block, 18 bytes, 32 weights: d (binary16), qs[16]; weight j
 *       (j < 16) is the low nibble of qs[j], weight 16+j the high nibble;
 *       w = d * T[q] with the non-uniform 16-entry table T below.
 *   Every value is little-endian.
 *
 * Every function returns 0 on success and a negative number on a bad
 * argument.  No function allocates more than it frees before returning.
 * Compiled with -std=c11 -ffp-contract=off so the fp64 arithmetic is
 * evaluated as written (no fused multiply-add contraction).
 */
#include <stdint.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_Q8_0 8
#define OR_Q4_K 12
#define OR_Q5_K 13
#define OR_Q6_K 14
#define OR_IQ4_NL 20

/* The IQ4_NL code book: the value of each 4-bit code before the block
 * scale (GGUF IQ4_NL format definition).  Parity unpinned: no source here
 * prints these sixteen values; the tests pin their structure only. */
static const int iq4nl_table[16] = {-127, -104, -83, -65, -49, -35, -22, -10,
                                    1,    13,   25,  38,  53,  69,  89,  113};

/* ---------------------------------------------------------------------- */
/* Scalar decoders                                                         */
/* ---------------------------------------------------------------------- */

/* IEEE 754 binary16 -> double, from the format's definition: 1 sign bit,
 * 5 exponent bits (bias 15), 10 fraction bits; exponent 0 = subnormal
 * (value = f * 2^-24), exponent 31 = infinity / NaN. */
double or_half_to_double(uint16_t h)
{
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = (f == 0) ? INFINITY : NAN;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return s ? -v : v;
}

/* The 6-bit scale and min of sub-block j (0..7) of a Q4_K super-block, read
 * from the 12 packed bytes sc12 (llama.cpp's get_scale_min_k4 packing):
 *   j < 4 : sc = low 6 bits of sc12[j],      m = low 6 bits of sc12[j+4]
 *   j >= 4: sc = low 4 bits of sc12[j+4] | (top 2 bits of sc12[j-4]) << 4
 *           m  = high 4 bits of sc12[j+4] | (top 2 bits of sc12[j])   << 4 */
int or_q4k_scale_min(const uint8_t *sc12, int j, int *sc, int *m)
{
    if (!sc12 || !sc || !m || j < 0 || j > 7)
        return -1;
    if (j < 4) {
        *sc = sc12[j] & 63;
        *m = sc12[j + 4] & 63;
    } else {
        *sc = (sc12[j + 4] & 15) | ((sc12[j - 4] >> 6) << 4);
        *m = (sc12[j + 4] >> 4) | ((sc12[j] >> 6) << 4);
    }
    return 0;
}

/* The 4-bit quant and sub-block index of weight i (0..255) of a Q4_K
 * super-block whose 128 quant bytes are qs. */
static int q4k_quant(const uint8_t *qs, int i, int *sub)
{
    int c = i / 64, l = i % 64;
    if (l < 32) {
        *sub = 2 * c;
        return qs[32 * c + l] & 15;
    }
    *sub = 2 * c + 1;
    return qs[32 * c + l - 32] >> 4;
}

/* Decode one 144-byte Q4_K super-block into 256 exact values. */
int or_dequant_block_q4k(const uint8_t *blk, double *w)
{
    if (!blk || !w)
        return -1;
    double d = or_half_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
    double dmin = or_half_to_double((uint16_t)(blk[2] | (blk[3] << 8)));
    const uint8_t *sc12 = blk + 4;
    const uint8_t *qs = blk + 16;
    for (int i = 0; i < 256; ++i) {
        int j, sc, m;
        int q = q4k_quant(qs, i, &j);
        or_q4k_scale_min(sc12, j, &sc, &m);
        /* d*sc*q has at most 11+6+4 significant bits and dmin*m at most
         * 11+6, so both products and their difference are exact in fp64. */
        w[i] = d * sc * q - dmin * m;
    }
    return 0;
}

/* Decode one 34-byte Q8_0 block into 32 exact values. */
int or_dequant_block_q8_0(const uint8_t *blk, double *w)
{
    if (!blk || !w)
        return -1;
    double d = or_half_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
    for (int i = 0; i < 32; ++i) {
        int q = (int)blk[2 + i];
        if (q > 127)
            q -= 256; /* two's complement int8 */
        w[i] = d * q;
    }
    return 0;
}

/* Decode one 176-byte Q5_K super-block into 256 exact values. */
int or_dequant_block_q5k(const uint8_t *blk, double *w)
{
    if (!blk || !w)
        return -1;
    double d = or_half_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
    double dmin = or_half_to_double((uint16_t)(blk[2] | (blk[3] << 8)));
    const uint8_t *sc12 = blk + 4;
    const uint8_t *qh = blk + 16;
    const uint8_t *qs = blk + 48;
    for (int i = 0; i < 256; ++i) {
        int j, sc, m;
        int lo = q4k_quant(qs, i, &j); /* same nibble order as Q4_K */
        int c = i / 64, l = i % 64;
        int hi = (qh[l % 32] >> (2 * c + (l >= 32))) & 1;
        int q5 = lo | (hi << 4);
        or_q4k_scale_min(sc12, j, &sc, &m);
        /* d*sc*q5: at most 11+6+5 significant bits; exact in fp64. */
        w[i] = d * sc * q5 - dmin * m;
    }
    return 0;
}

/* Decode one 210-byte Q6_K super-block into 256 exact values. */
int or_dequant_block_q6k(const uint8_t *blk, double *w)
{
    if (!blk || !w)
        return -1;
    const uint8_t *ql = blk;
    const uint8_t *qh = blk + 128;
    const uint8_t *scales = blk + 192;
    double d = or_half_to_double((uint16_t)(blk[208] | (blk[209] << 8)));
    for (int i = 0; i < 256; ++i) {
        int n = i / 128, r = i % 128, t = r / 32, l = r % 32;
        int byte = ql[64 * n + 32 * (t & 1) + l];
        int lo = (t >= 2) ? (byte >> 4) : (byte & 15);
        int hi = (qh[32 * n + l] >> (2 * t)) & 3;
        int q = (lo | (hi << 4)) - 32;
        int sc = (int)scales[i / 16];
        if (sc > 127)
            sc -= 256; /* int8 scale */
        w[i] = d * sc * q;
    }
    return 0;
}

/* Decode one 18-byte IQ4_NL block into 32 exact values. */
int or_dequant_block_iq4nl(const uint8_t *blk, double *w)
{
    if (!blk || !w)
        return -1;
    double d = or_half_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
    const uint8_t *qs = blk + 2;
    for (int j = 0; j < 16; ++j) {
        w[j] = d * iq4nl_table[qs[j] & 15];
        w[16 + j] = d * iq4nl_table[qs[j] >> 4];
    }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Matrix geometry                                                         */
/* ---------------------------------------------------------------------- */

/* Bytes of one row of K weights, or -1 when K does not fill whole blocks. */
int64_t or_row_bytes(int fmt, int64_t K)
{
    if (K <= 0)
        return -1;
    if (fmt == OR_Q4_K)
        return (K % 256) ? -1 : (K / 256) * 144;
    if (fmt == OR_Q8_0)
        return (K % 32) ? -1 : (K / 32) * 34;
    if (fmt == OR_Q5_K)
        return (K % 256) ? -1 : (K / 256) * 176;
    if (fmt == OR_Q6_K)
        return (K % 256) ? -1 : (K / 256) * 210;
    if (fmt == OR_IQ4_NL)
        return (K % 32) ? -1 : (K / 32) * 18;
    return -1;
}

/* Decode row r (all K weights) of a row-major GGUF matrix. */
static void dequant_row(int fmt, const uint8_t *w, int64_t K, int64_t rb,
                        int64_t r, double *out)
{
    const uint8_t *row = w + r * rb;
    if (fmt == OR_Q4_K) {
        for (int64_t b = 0; b < K / 256; ++b)
            or_dequant_block_q4k(row + b * 144, out + b * 256);
    } else if (fmt == OR_Q5_K) {
        for (int64_t b = 0; b < K / 256; ++b)
            or_dequant_block_q5k(row + b * 176, out + b * 256);
    } else if (fmt == OR_Q6_K) {
        for (int64_t b = 0; b < K / 256; ++b)
            or_dequant_block_q6k(row + b * 210, out + b * 256);
    } else if (fmt == OR_IQ4_NL) {
        for (int64_t b = 0; b < K / 32; ++b)
            or_dequant_block_iq4nl(row + b * 18, out + b * 32);
    } else {
        for (int64_t b = 0; b < K / 32; ++b)
            or_dequant_block_q8_0(row + b * 34, out + b * 32);
    }
}

/* out[nrows][K] = exact weights of rows row0 .. row0+nrows-1. */
int or_dequant_rows(int fmt, const uint8_t *w, int64_t N, int64_t K,
                    int64_t row0, int64_t nrows, double *out)
{
    int64_t rb = or_row_bytes(fmt, K);
    if (!w || !out || rb < 0 || N <= 0 || row0 < 0 || nrows < 0 ||
        row0 + nrows > N)
        return -1;
    for (int64_t i = 0; i < nrows; ++i)
        dequant_row(fmt, w, K, rb, row0 + i, out + i * K);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Products                                                                */
/* ---------------------------------------------------------------------- */

/* Decode-then-dot for selected rows and M activation vectors:
 *   Y[m*nrows + i] = sum_k w[rows[i]][k] * X[m*ldx + k]
 *   C[m*nrows + i] = sum_k |w[rows[i]][k] * X[m*ldx + k]|   (C may be NULL)
 * X is fp32 (the activations are kept in f32, never quantized); every
 * product and sum is taken in fp64.  rows == NULL means rows 0..nrows-1.
 * nthreads > 1 spreads rows over OpenMP threads (each row is summed by one
 * thread in index order, so the result does not depend on nthreads). */
int or_gemv(int fmt, const uint8_t *w, int64_t N, int64_t K,
            const float *X, int64_t M, int64_t ldx,
            const int64_t *rows, int64_t nrows,
            double *Y, double *C, int nthreads)
{
    int64_t rb = or_row_bytes(fmt, K);
    if (!w || !X || !Y || rb < 0 || N <= 0 || M <= 0 || ldx < K || nrows < 0)
        return -1;
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows ? rows[i] : i;
        if (r < 0 || r >= N)
            return -2;
    }
    int bad = 0;
#ifdef _OPENMP
    if (nthreads < 1)
        nthreads = 1;
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double *wr = (double *)malloc((size_t)K * sizeof(double));
        if (!wr) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            bad = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
            for (int64_t i = 0; i < nrows; ++i) {
                int64_t r = rows ? rows[i] : i;
                dequant_row(fmt, w, K, rb, r, wr);
                for (int64_t m = 0; m < M; ++m) {
                    const float *x = X + m * ldx;
                    double s = 0.0, a = 0.0;
                    for (int64_t k = 0; k < K; ++k) {
                        double p = wr[k] * (double)x[k];
                        s += p;
                        a += fabs(p);
                    }
                    Y[m * nrows + i] = s;
                    if (C)
                        C[m * nrows + i] = a;
                }
            }
            free(wr);
        }
    }
    return bad ? -3 : 0;
}

/* Round a float to bfloat16 (round to nearest, ties to even), from the
 * definition: the two bf16 neighbours of f are its bit pattern truncated to
 * the top 16 bits and the next pattern up in magnitude; pick the nearer, and
 * on a tie the one whose last kept bit is 0.  NaN stays a quiet NaN. */
uint16_t or_bf16_from_float(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu))
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lower = u >> 16;
    uint32_t rest = u & 0xffffu;
    if (rest > 0x8000u || (rest == 0x8000u && (lower & 1u)))
        return (uint16_t)(lower + 1u);
    return (uint16_t)lower;
}

/* bfloat16 bit pattern -> double (bf16 is the top half of a binary32). */
double or_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* The prefill product with bf16 operands, for any weight format.  Each
 * weight is taken as bf16(RN_fp32(w)): the exact value rounded to fp32, then
 * to bf16.  X is M
 * rows of K bfloat16 patterns (leading dimension ldx).  Then
 *   Y[m*nrows + i] = sum_k w_bf16[rows[i]][k] * x_bf16[m][k]   (fp64)
 *   C[m*nrows + i] = sum_k |w[rows[i]][k] * x_bf16[m][k]|  (exact w)  */
int or_gemm_bf16_fmt(int fmt, const uint8_t *w, int64_t N, int64_t K,
                     const uint16_t *X, int64_t M, int64_t ldx,
                     const int64_t *rows, int64_t nrows,
                     double *Y, double *C, int nthreads)
{
    int64_t rb = or_row_bytes(fmt, K);
    if (!w || !X || !Y || rb < 0 || N <= 0 || M <= 0 || ldx < K || nrows < 0)
        return -1;
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows ? rows[i] : i;
        if (r < 0 || r >= N)
            return -2;
    }
    int bad = 0;
#ifdef _OPENMP
    if (nthreads < 1)
        nthreads = 1;
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double *wr = (double *)malloc((size_t)K * 2 * sizeof(double));
        if (!wr) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            bad = 1;
        } else {
            double *wb = wr + K;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
            for (int64_t i = 0; i < nrows; ++i) {
                int64_t r = rows ? rows[i] : i;
                dequant_row(fmt, w, K, rb, r, wr);
                for (int64_t k = 0; k < K; ++k)
                    wb[k] = or_bf16_to_double(or_bf16_from_float((float)wr[k]));
                for (int64_t m = 0; m < M; ++m) {
                    const uint16_t *x = X + m * ldx;
                    double s = 0.0, a = 0.0;
                    for (int64_t k = 0; k < K; ++k) {
                        double xv = or_bf16_to_double(x[k]);
                        s += wb[k] * xv;
                        a += fabs(wr[k] * xv);
                    }
                    Y[m * nrows + i] = s;
                    if (C)
                        C[m * nrows + i] = a;
                }
            }
            free(wr);
        }
    }
    return bad ? -3 : 0;
}

/* The Q4_K prefill product (or_gemm_bf16_fmt for Q4_K). */
int or_gemm_bf16(const uint8_t *w, int64_t N, int64_t K,
                 const uint16_t *X, int64_t M, int64_t ldx,
                 const int64_t *rows, int64_t nrows,
                 double *Y, double *C, int nthreads)
{
    return or_gemm_bf16_fmt(OR_Q4_K, w, N, K, X, M, ldx, rows, nrows, Y, C, nthreads);
}

/* SwiGLU between the gate and up projections of an expert FFN:
 *   h = silu(g) * u,  silu(z) = z / (1 + exp(-z))       (fp64, libm exp) */
int or_swiglu(const double *g, const double *u, int64_t n, double *h)
{
    if (!g || !u || !h || n < 0)
        return -1;
    for (int64_t i = 0; i < n; ++i)
        h[i] = g[i] / (1.0 + exp(-g[i])) * u[i];
    return 0;
}

/* Number of OpenMP threads available (1 when built without OpenMP). */
int or_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------------- */
/* Q8_K activations (the integer-dot variant)                              */
/* ---------------------------------------------------------------------- */

/* "Frink Inference: the Rust alternative to llama.cpp", section "Where
 * llama.cpp is still ahead": llama.cpp quantizes the activations to Q8_K
 * before a K-quant dot product, which is why its K-quant logits drift from
 * an f32 engine's.  The pages name the format only; the layout and the
 * quantizer here are GGUF's Q8_K (reading: llama.cpp's reference row
 * quantizer):
 *   block of 256 activations, 292 bytes:
 *     [0..3]     d, binary32
 *     [4..259]   q[256], int8
 *     [260..291] bsums[16], int16: bsums[g] = sum of q[16g .. 16g+15]
 *   max = the signed value of the first element with the largest |x| (an
 *   element replaces the running choice only when strictly larger);
 *   max == 0: d = 0 and every q = 0.  Otherwise, in binary32 arithmetic,
 *   iscale = -127 / max, q_j = min(127, round-half-even(iscale * x_j)),
 *   d = 1 / iscale.  The value a code stands for is d * q_j.
 * The divisions and the product decide integer codes, so they are taken in
 * binary32 exactly as written (one rounding each), not in fp64. */
int or_quantize_q8_k(const float *x, int64_t K, uint8_t *out)
{
    if (!x || !out || K <= 0 || K % 256)
        return -1;
    for (int64_t b = 0; b < K / 256; ++b) {
        const float *xb = x + b * 256;
        uint8_t *ob = out + b * 292;
        float amax = 0.f, max = 0.f;
        for (int j = 0; j < 256; ++j) {
            float ax = fabsf(xb[j]);
            if (ax > amax) {
                amax = ax;
                max = xb[j];
            }
        }
        int8_t q[256];
        float d;
        if (amax == 0.f) {
            d = 0.f;
            memset(q, 0, sizeof(q));
        } else {
            volatile float iscale = -127.f / max;
            for (int j = 0; j < 256; ++j) {
                volatile float t = iscale * xb[j];
                long v = lrintf(t); /* the default rounding mode: half to even */
                q[j] = (int8_t)(v > 127 ? 127 : v);
            }
            d = 1.f / iscale;
        }
        memcpy(ob, &d, 4);
        memcpy(ob + 4, q, 256);
        for (int g = 0; g < 16; ++g) {
            int s = 0;
            for (int j = 0; j < 16; ++j)
                s += q[16 * g + j];
            int16_t s16 = (int16_t)s;
            memcpy(ob + 260 + 2 * g, &s16, 2);
        }
    }
    return 0;
}

/* The activations Q8_K blocks stand for: x[k] = d_b * q_k (exact in fp64). */
int or_dequant_q8_k(const uint8_t *xq, int64_t K, double *x)
{
    if (!xq || !x || K <= 0 || K % 256)
        return -1;
    for (int64_t b = 0; b < K / 256; ++b) {
        float d;
        memcpy(&d, xq + b * 292, 4);
        const int8_t *q = (const int8_t *)(xq + b * 292 + 4);
        for (int j = 0; j < 256; ++j)
            x[b * 256 + j] = (double)d * (double)q[j];
    }
    return 0;
}

/* The integer-dot GEMV against Q8_K activations:
 *   Y[i] = sum_k w[i][k] * xhat[k],  xhat = the values the Q8_K blocks stand for,
 *   C[i] = sum_k |w[i][k] * xhat[k]|                           (C may be NULL).
 * llama.cpp's integer kernel adds q_w * q_x in int32 per sub-block and
 * applies the block scales afterwards; that only regroups this sum (every
 * integer partial is exact), so the definition is the decode-then-dot of the
 * exact weights with the exact dequantized activations, in fp64. */
int or_gemv_q8k(int fmt, const uint8_t *w, int64_t N, int64_t K, const uint8_t *xq,
                double *Y, double *C, int nthreads)
{
    int64_t rb = or_row_bytes(fmt, K);
    if (!w || !xq || !Y || rb < 0 || N <= 0 || K % 256)
        return -1;
    double *xh = (double *)malloc((size_t)K * sizeof(double));
    if (!xh)
        return -3;
    or_dequant_q8_k(xq, K, xh);
    int bad = 0;
#ifdef _OPENMP
    if (nthreads < 1)
        nthreads = 1;
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double *wr = (double *)malloc((size_t)K * sizeof(double));
        if (!wr) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            bad = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
            for (int64_t i = 0; i < N; ++i) {
                dequant_row(fmt, w, K, rb, i, wr);
                double s = 0.0, a = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    double p = wr[k] * xh[k];
                    s += p;
                    a += fabs(p);
                }
                Y[i] = s;
                if (C)
                    C[i] = a;
            }
            free(wr);
        }
    }
    free(xh);
    return bad ? -3 : 0;
}
