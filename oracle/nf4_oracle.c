/*
 * nf4_oracle.c -- plain, slow CPU oracle for the QLoRA NF4 frozen-base linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's CPU-baseline
 * leg may load this library.  It shares no code, header, table or constant generator with
 * the CUDA library; neither side includes or links the other.
 *
 * Every routine restates a definition from the source pages, cited by page title and
 * section:
 *   [QLoRA-paperclase]  "QLoRA -- La base en 4 bits, LoRA encima: absmax, NormalFloat y
 *                        cuanto se ahorra" (paperclase.com, LoRA course, lesson 8)
 *   [QLoRA-ultralytics] "QLoRA" glossary entry (ultralytics.com), section "Como funciona a
 *                        QLoRA", its NF4 snippet and the printed MSE
 *   [QLoRA-skillverse]  "Capitulo 1: Que es QLoRA?" (docs.skillversehub.com), section
 *                        "Componentes clave"
 * Readings where the pages are silent are marked READING and are listed in the design notes.
 *
 * Arithmetic: fp32 where the pages' torch code computes in fp32 (the quantizer's division and
 * distances), fp64 for everything that is "exact up to rounding order" (the layer products).
 * The file must be compiled with -ffp-contract=off so that no multiply-add is fused except
 * where fmaf() is written explicitly.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------------------ */
/* Standard normal distribution.                                                         */
/* ------------------------------------------------------------------------------------ */

/* Upper tail Q(x) = P(Z > x) = erfc(x / sqrt 2) / 2, from the definition of Phi. */
static double upper_tail(double x) { return 0.5 * erfc(x / sqrt(2.0)); }

/* Phi^{-1}(p) by bisection on the monotone tail function: the plainest correct inverse.
 * The root x >= 0 of Q(x) = t is searched on [0, 40], with t = 1 - p for p > 1/2 (exact in
 * fp64 by Sterbenz's lemma) and t = p for p < 1/2 (then Phi^{-1}(p) = -x by symmetry); Q
 * keeps full relative precision in the tail.  Stops when the bracket is two adjacent
 * doubles. */
double orc_norm_ppf(double p)
{
    if (p == 0.5) return 0.0;
    if (p <= 0.0) return -INFINITY;
    if (p >= 1.0) return INFINITY;
    double sign = (p < 0.5) ? -1.0 : 1.0;
    double target = (p < 0.5) ? p : 1.0 - p;
    double lo = 0.0, hi = 40.0; /* Q(lo) >= target > Q(hi) */
    for (int it = 0; it < 4000; ++it) {
        double mid = 0.5 * (lo + hi);
        if (mid <= lo || mid >= hi) break;
        if (upper_tail(mid) >= target) lo = mid; else hi = mid;
    }
    /* pick the endpoint whose tail is closer to the target */
    double elo = fabs(upper_tail(lo) - target), ehi = fabs(upper_tail(hi) - target);
    return sign * ((ehi < elo) ? hi : lo);
}

/* ------------------------------------------------------------------------------------ */
/* Level tables.                                                                         */
/* ------------------------------------------------------------------------------------ */

/* linspace(a, b, n)[i] in fp64. */
static double lin(double a, double b, int n, int i) { return a + (b - a) * (double)i / (double)(n - 1); }

/* NF4 levels "as built in bitsandbytes" [QLoRA-ultralytics, NF4 snippet]:
 * 8 positive levels Phi^{-1}(linspace(0.9677083, 0.5, 9)[:-1]), 7 negative levels
 * -Phi^{-1}(linspace(0.9677083, 0.5, 8)[:-1]), one exact zero; sorted ascending and
 * divided by the largest (Phi^{-1}(0.9677083)).
 * READING: the page builds the table in fp32 torch ops; here each level is computed in fp64
 * and rounded to fp32 once, which fixes one format constant for every implementation.
 * Output: 16 floats, ascending. */
void orc_nf4_levels(float out[16])
{
    const double top = 0.9677083;
    double v[16];
    int n = 0;
    for (int j = 0; j < 7; ++j) v[n++] = -orc_norm_ppf(lin(top, 0.5, 8, j));
    v[n++] = 0.0;
    for (int i = 0; i < 8; ++i) v[n++] = orc_norm_ppf(lin(top, 0.5, 9, i));
    /* insertion sort (ascending) */
    for (int i = 1; i < 16; ++i) {
        double x = v[i];
        int j = i - 1;
        while (j >= 0 && v[j] > x) { v[j + 1] = v[j]; --j; }
        v[j + 1] = x;
    }
    double mx = v[15];
    for (int i = 0; i < 16; ++i) out[i] = (float)(v[i] / mx);
}

/* The toy NF4 table of [QLoRA-paperclase, "Parte 2 - NormalFloat", "Dieciseis niveles por
 * cuantiles"]: 8 quantiles on linspace(d, 0.5, 8) for the negatives (the last is 0),
 * 9 on linspace(0.5, 1 - d, 9) for the positives (the first is 0), joined without repeating
 * the zero and divided by the largest absolute value.  Only used to pin orc_norm_ppf
 * against the 2-decimal table the page prints. */
void orc_toy_levels(double d, double out[16])
{
    int n = 0;
    for (int i = 0; i < 8; ++i) out[n++] = orc_norm_ppf(lin(d, 0.5, 8, i));
    for (int i = 1; i < 9; ++i) out[n++] = orc_norm_ppf(lin(0.5, 1.0 - d, 9, i));
    double mx = 0.0;
    for (int i = 0; i < 16; ++i) if (fabs(out[i]) > mx) mx = fabs(out[i]);
    for (int i = 0; i < 16; ++i) out[i] /= mx;
}

/* ------------------------------------------------------------------------------------ */
/* absmax int4 (15 levels) -- [QLoRA-paperclase, "Parte 1", "absmax, en formulas"]:       */
/*   c_i = round(7 * w_i / max_j |w_j|),  w^_i = c_i * absmax / 7                           */
/* computed like the page's fp32 torch code: (w / absmax) * 7, round half to even, and    */
/* back as (c / 7) * absmax.                                                              */
/* ------------------------------------------------------------------------------------ */
void orc_int4_absmax(const float *w, int64_t n, float *absmax_out, int32_t *codes, float *w_hat)
{
    float am = 0.0f;
    for (int64_t i = 0; i < n; ++i) if (fabsf(w[i]) > am) am = fabsf(w[i]);
    for (int64_t i = 0; i < n; ++i) {
        float t = (w[i] / am) * 7.0f;
        float c = nearbyintf(t); /* default rounding mode: nearest, ties to even */
        codes[i] = (int32_t)c;
        w_hat[i] = (c / 7.0f) * am;
    }
    *absmax_out = am;
}

/* ------------------------------------------------------------------------------------ */
/* Nearest-level code: argmin_k |fl(x) - L_k| with fp32 distances, first index on ties    */
/* (torch argmin returns the first minimum) -- [QLoRA-paperclase, "Parte 4", "Una capa    */
/* QLoRA, a mano"; QLoRA-ultralytics, NF4 snippet].                                       */
/* ------------------------------------------------------------------------------------ */
static int nearest_level(float x, const float *levels, int nlev)
{
    int best = 0;
    float bd = fabsf(x - levels[0]);
    for (int k = 1; k < nlev; ++k) {
        float d = fabsf(x - levels[k]);
        if (d < bd) { bd = d; best = k; }
    }
    return best;
}

/* Blockwise absmax + nearest level over a flat array, blocks of `bs` consecutive values.
 * codes: one per value (unpacked).  absmax: one per block.
 * READING (all-zero block, unstated on the pages): absmax = 0 and every code is the index of
 * the exact-zero level, so the block dequantizes to exact zeros. */
void orc_blockwise_codes(const float *w, int64_t n, int64_t bs, const float *levels, int nlev,
                         uint8_t *codes, float *absmax)
{
    int zero_idx = 0;
    for (int k = 0; k < nlev; ++k) if (levels[k] == 0.0f) zero_idx = k;
    int64_t nb = n / bs;
    for (int64_t b = 0; b < nb; ++b) {
        const float *blk = w + b * bs;
        float am = 0.0f;
        for (int64_t i = 0; i < bs; ++i) if (fabsf(blk[i]) > am) am = fabsf(blk[i]);
        absmax[b] = am;
        for (int64_t i = 0; i < bs; ++i) {
            if (am == 0.0f) { codes[b * bs + i] = (uint8_t)zero_idx; continue; }
            float x = blk[i] / am;
            codes[b * bs + i] = (uint8_t)nearest_level(x, levels, nlev);
        }
    }
}

/* The reconstruction experiment of [QLoRA-ultralytics, NF4 snippet]: codes as above, then
 * restored = levels[code] * absmax in fp32 (no double quantization, no bf16), returns the
 * mean of the squared residuals (accumulated in fp64). */
double orc_blockwise_mse(const float *w, int64_t n, int64_t bs, const float *levels, int nlev)
{
    int64_t nb = n / bs;
    uint8_t *codes = (uint8_t *)malloc((size_t)n);
    float *am = (float *)malloc(sizeof(float) * (size_t)nb);
    orc_blockwise_codes(w, n, bs, levels, nlev, codes, am);
    double acc = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        float r = levels[codes[i]] * am[i / bs];
        double e = (double)(r - w[i]);
        acc += e * e;
    }
    free(codes);
    free(am);
    return acc / (double)n;
}

/* ------------------------------------------------------------------------------------ */
/* Packing: two 4-bit codes per byte ([QLoRA-paperclase, "Una capa QLoRA, a mano": the     */
/* real format packs two codes per byte).                                                */
/* READING (nibble order unstated): byte j = (c[2j] << 4) | c[2j+1], row-major order.     */
/* ------------------------------------------------------------------------------------ */
void orc_pack_nibbles(const uint8_t *codes, int64_t n, uint8_t *packed)
{
    for (int64_t j = 0; j < n / 2; ++j) packed[j] = (uint8_t)((codes[2 * j] << 4) | (codes[2 * j + 1] & 0xF));
}

void orc_unpack_nibbles(const uint8_t *packed, int64_t n, uint8_t *codes)
{
    for (int64_t j = 0; j < n / 2; ++j) {
        codes[2 * j] = (uint8_t)(packed[j] >> 4);
        codes[2 * j + 1] = (uint8_t)(packed[j] & 0xF);
    }
}

/* ------------------------------------------------------------------------------------ */
/* Double quantization of the block scales -- [QLoRA-paperclase, "Parte 3 - Cuanta       */
/* memoria", "Bits por parametro": 8 bits per absmax plus one 32-bit constant per 256     */
/* blocks; QLoRA-ultralytics, "Quantizacao dupla": scales quantized to 8 bits in blocks   */
/* of 256].  The pages fix only the block size and bit width.                             */
/* READING (the scheme): one fp32 offset mu per tensor (the mean of all block scales),   */
/* then per group of 256 blocks a symmetric absmax int8 code of (s_b - mu):               */
/*   c2_g = max_{b in g} |fl(s_b - mu)|                                                   */
/*   q_b  = clamp(rint(fl(fl(fl(s_b - mu) / c2_g) * 127)), -127, 127); q_b = 0 if c2_g = 0 */
/* READING (mu's rounding order, needed for bit-exactness): S_g = fp64 sum of the group's  */
/* scales in index order; the S_g are added by a pairwise tree (padded with zeros to a    */
/* power of two, level by level, elements 2i and 2i+1); mu = fl32(total / nb) with the    */
/* division in fp64.                                                                     */
/* ------------------------------------------------------------------------------------ */
float orc_dq_mean(const float *s, int64_t nb)
{
    int64_t ng = (nb + 255) / 256;
    int64_t p2 = 1;
    while (p2 < ng) p2 <<= 1;
    double *t = (double *)calloc((size_t)p2, sizeof(double));
    for (int64_t g = 0; g < ng; ++g) {
        double acc = 0.0;
        int64_t b1 = (g + 1) * 256 < nb ? (g + 1) * 256 : nb;
        for (int64_t b = g * 256; b < b1; ++b) acc += (double)s[b];
        t[g] = acc;
    }
    for (int64_t len = p2; len > 1; len >>= 1)
        for (int64_t i = 0; i < len / 2; ++i) t[i] = t[2 * i] + t[2 * i + 1];
    double total = t[0];
    free(t);
    return (float)(total / (double)nb);
}

void orc_double_quant(const float *s, int64_t nb, int8_t *q, float *c2, float *mu_out)
{
    float mu = orc_dq_mean(s, nb);
    int64_t ng = (nb + 255) / 256;
    for (int64_t g = 0; g < ng; ++g) {
        int64_t b0 = g * 256, b1 = (g + 1) * 256 < nb ? (g + 1) * 256 : nb;
        float m = 0.0f;
        for (int64_t b = b0; b < b1; ++b) {
            float d = fabsf(s[b] - mu);
            if (d > m) m = d;
        }
        c2[g] = m;
        for (int64_t b = b0; b < b1; ++b) {
            if (m == 0.0f) { q[b] = 0; continue; }
            float d = s[b] - mu;
            float t = (d / m) * 127.0f;
            float r = nearbyintf(t);
            if (r > 127.0f) r = 127.0f;
            if (r < -127.0f) r = -127.0f;
            q[b] = (int8_t)r;
        }
    }
    *mu_out = mu;
}

/* ------------------------------------------------------------------------------------ */
/* bf16 rounding, from the definition: round to the nearest value with an 8-bit          */
/* significand, ties to the candidate whose last significand bit is 0.                    */
/* (bf16 is the compute dtype of [QLoRA-skillverse, config snippet] and of the forward    */
/* pass in [QLoRA-ultralytics, "desquantiza ... para bfloat16"].)                          */
/* ------------------------------------------------------------------------------------ */
uint16_t orc_bf16_round(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    if (isnan(x)) return (uint16_t)((u >> 16) | 0x40); /* quiet NaN, sign kept */
    uint32_t lo_bits = u & 0xFFFF0000u;                 /* truncation toward zero    */
    uint32_t hi_bits = lo_bits + 0x10000u;              /* next magnitude up         */
    float lo, hi;
    memcpy(&lo, &lo_bits, 4);
    memcpy(&hi, &hi_bits, 4);
    if (u == lo_bits) return (uint16_t)(u >> 16);       /* already representable     */
    /* distances in fp64 are exact for these operands.  When the next magnitude up is the
     * infinity pattern, it stands for 2^128 (IEEE overflow rule for round-to-nearest). */
    double dlo = fabs((double)x - (double)lo);
    double dhi = isinf(hi) ? fabs(ldexp(1.0, 128) - fabs((double)x)) : fabs((double)hi - (double)x);
    uint32_t pick;
    if (dlo < dhi) pick = lo_bits;
    else if (dhi < dlo) pick = hi_bits;
    else pick = ((lo_bits >> 16) & 1u) ? hi_bits : lo_bits; /* tie: even significand */
    return (uint16_t)(pick >> 16);
}

/* The same rounding applied once to an fp64 value (no intermediate fp32 rounding): the two bf16
 * values around x are found from its binary exponent, and the nearer one is taken, ties to the
 * even significand.  Values below the smallest normal use the subnormal spacing 2^-133; past the
 * largest finite bf16 the result is infinity (IEEE round-to-nearest overflow rule). */
uint16_t orc_bf16_round_d(double x)
{
    if (isnan(x)) return 0x7FC0;
    const uint16_t sign = (x < 0) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                              /* a = m 2^e, m in [0.5, 1) */
    int q = e - 8;                             /* spacing of 8-bit significands at this binade */
    if (q < -133) q = -133;                    /* bf16 subnormal spacing */
    double step = ldexp(1.0, q);
    double lo = floor(a / step) * step;        /* exact: a / step only shifts the exponent */
    double hi = lo + step;
    double dlo = a - lo, dhi = hi - a;
    double pick;
    if (dlo < dhi) pick = lo;
    else if (dhi < dlo) pick = hi;
    else pick = (fmod(lo / step, 2.0) == 0.0) ? lo : hi;  /* tie: even significand */
    if (pick >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
    float f = (float)pick;                     /* exact: pick has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

double orc_bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* ------------------------------------------------------------------------------------ */
/* NF4 quantization of a weight matrix, as stored by the layer:                            */
/*   flatten W row-major, blocks of 64, absmax per block, nearest NF4 level per weight     */
/*   ([QLoRA-paperclase, "Una capa QLoRA, a mano"]; [QLoRA-ultralytics, NF4 bullet and     */
/*   snippet]), pack two codes per byte, then double-quantize the 64-blocks' scales.       */
/* Outputs: packed[rows*cols/2], qcode[nb], c2[ng], mu[1]; absmax[nb] (fp32 scales before */
/* double quantization) if non-NULL.                                                     */
/* ------------------------------------------------------------------------------------ */
void orc_nf4_quantize(const float *W, int64_t rows, int64_t cols, uint8_t *packed, int8_t *qcode,
                      float *c2, float *mu, float *absmax_out)
{
    float L[16];
    orc_nf4_levels(L);
    int64_t n = rows * cols, nb = n / 64;
    uint8_t *codes = (uint8_t *)malloc((size_t)n);
    float *am = (float *)malloc(sizeof(float) * (size_t)nb);
    orc_blockwise_codes(W, n, 64, L, 16, codes, am);
    orc_pack_nibbles(codes, n, packed);
    orc_double_quant(am, nb, qcode, c2, mu);
    if (absmax_out) memcpy(absmax_out, am, sizeof(float) * (size_t)nb);
    free(codes);
    free(am);
}

/* Dequantization to bf16 -- [QLoRA-paperclase, "Cuantiles", w^ = NF4[c] * absmax;       */
/* "Una capa QLoRA, a mano", forward]; [QLoRA-ultralytics: dequantized to bfloat16 just  */
/* before the matmul].  With double quantization the block scale is first rebuilt:      */
/*   k_g = fl32(c2_g / 127),  s'_b = fmaf(q_b, k_g, mu)   (one rounding)                   */
/*   W^  = bf16(fl32(NF4[c] * s'_b))                                                       */
/* ------------------------------------------------------------------------------------ */
float orc_dq_scale(int8_t q, float c2, float mu)
{
    float k = c2 / 127.0f;
    return fmaf((float)q, k, mu);
}

void orc_nf4_dequantize(const uint8_t *packed, const int8_t *qcode, const float *c2, float mu,
                        int64_t rows, int64_t cols, uint16_t *out_bf16)
{
    float L[16];
    orc_nf4_levels(L);
    int64_t n = rows * cols;
    for (int64_t i = 0; i < n; ++i) {
        uint8_t byte = packed[i / 2];
        int c = (i % 2 == 0) ? (byte >> 4) : (byte & 0xF);
        int64_t b = i / 64, g = b / 256;
        float s = orc_dq_scale(qcode[b], c2[g], mu);
        float v = L[c] * s;
        out_bf16[i] = orc_bf16_round(v);
    }
}

/* ------------------------------------------------------------------------------------ */
/* The QLoRA linear layer -- [QLoRA-paperclase, "Parte 4 - LoRA encima":                  */
/*   h = W^ x + (alpha/r) B A x   ("El gradiente atraviesa la base de 4 bits")             */
/*   dL/dx = (W^ + (alpha/r) B A)^T dL/dh;  dL/dW^ is not computed]                         */
/* [QLoRA-ultralytics, "Como funciona": backprop through the dequantized weights, only   */
/* the two LoRA matrices are updated].                                                   */
/* Shapes (torch linear convention): W^ [N,K], X [M,K], A [r,K], B [N,r], G = dL/dY [M,N].  */
/* Row-vector form: Y = X W^T + s U B^T with U = X A^T and s = alpha / r.                  */
/* Backward (chain rule on the same expression): V = G B,                                 */
/*   dX = G W^ + s V A,  dA = s V^T X,  dB = s G^T U.                                      */
/* All products in fp64 from the bf16 inputs; U and V are not rounded.                    */
/* ------------------------------------------------------------------------------------ */

/* Y rows and U rows for the listed token rows (nsel of them).  Y_out [nsel,N], U_out [nsel,r]. */
void orc_layer_fwd_rows(const uint16_t *What, const uint16_t *X, const uint16_t *A, const uint16_t *B,
                        int64_t M, int64_t N, int64_t K, int64_t r, double alpha,
                        const int64_t *sel, int64_t nsel, double *Y_out, double *U_out)
{
    (void)M;
    double s = alpha / (double)r;
    double *u = (double *)malloc(sizeof(double) * (size_t)(r > 0 ? r : 1));
    for (int64_t ii = 0; ii < nsel; ++ii) {
        int64_t m = sel[ii];
        for (int64_t j = 0; j < r; ++j) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += orc_bf16_to_double(X[m * K + k]) * orc_bf16_to_double(A[j * K + k]);
            u[j] = acc;
            if (U_out) U_out[ii * r + j] = acc;
        }
        for (int64_t n = 0; n < N; ++n) {
            double base = 0.0;
            for (int64_t k = 0; k < K; ++k) base += orc_bf16_to_double(X[m * K + k]) * orc_bf16_to_double(What[n * K + k]);
            double lora = 0.0;
            for (int64_t j = 0; j < r; ++j) lora += u[j] * orc_bf16_to_double(B[n * r + j]);
            Y_out[ii * N + n] = base + s * lora;
        }
    }
    free(u);
}

/* dX rows for the listed token rows.  dX_out [nsel,K]. */
void orc_layer_dx_rows(const uint16_t *What, const uint16_t *A, const uint16_t *B, const uint16_t *G,
                       int64_t M, int64_t N, int64_t K, int64_t r, double alpha,
                       const int64_t *sel, int64_t nsel, double *dX_out)
{
    (void)M;
    double s = alpha / (double)r;
    double *v = (double *)malloc(sizeof(double) * (size_t)(r > 0 ? r : 1));
    double *row = (double *)malloc(sizeof(double) * (size_t)K);
    for (int64_t ii = 0; ii < nsel; ++ii) {
        int64_t m = sel[ii];
        for (int64_t j = 0; j < r; ++j) {
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n) acc += orc_bf16_to_double(G[m * N + n]) * orc_bf16_to_double(B[n * r + j]);
            v[j] = acc;
        }
        for (int64_t k = 0; k < K; ++k) row[k] = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            double g = orc_bf16_to_double(G[m * N + n]);
            for (int64_t k = 0; k < K; ++k) row[k] += g * orc_bf16_to_double(What[n * K + k]);
        }
        for (int64_t k = 0; k < K; ++k) {
            double lora = 0.0;
            for (int64_t j = 0; j < r; ++j) lora += v[j] * orc_bf16_to_double(A[j * K + k]);
            dX_out[ii * K + k] = row[k] + s * lora;
        }
    }
    free(v);
    free(row);
}

/* Full adapter gradients: dA [r,K] = s V^T X and dB [N,r] = s G^T U over all M tokens. */
void orc_layer_adapter_grads(const uint16_t *X, const uint16_t *A, const uint16_t *B, const uint16_t *G,
                             int64_t M, int64_t N, int64_t K, int64_t r, double alpha,
                             double *dA_out, double *dB_out)
{
    double s = alpha / (double)r;
    double *U = (double *)calloc((size_t)(M * r), sizeof(double));
    double *V = (double *)calloc((size_t)(M * r), sizeof(double));
    for (int64_t m = 0; m < M; ++m)
        for (int64_t j = 0; j < r; ++j) {
            double au = 0.0, av = 0.0;
            for (int64_t k = 0; k < K; ++k) au += orc_bf16_to_double(X[m * K + k]) * orc_bf16_to_double(A[j * K + k]);
            for (int64_t n = 0; n < N; ++n) av += orc_bf16_to_double(G[m * N + n]) * orc_bf16_to_double(B[n * r + j]);
            U[m * r + j] = au;
            V[m * r + j] = av;
        }
    for (int64_t j = 0; j < r; ++j)
        for (int64_t k = 0; k < K; ++k) {
            double acc = 0.0;
            for (int64_t m = 0; m < M; ++m) acc += V[m * r + j] * orc_bf16_to_double(X[m * K + k]);
            dA_out[j * K + k] = s * acc;
        }
    for (int64_t n = 0; n < N; ++n)
        for (int64_t j = 0; j < r; ++j) {
            double acc = 0.0;
            for (int64_t m = 0; m < M; ++m) acc += orc_bf16_to_double(G[m * N + n]) * U[m * r + j];
            dB_out[n * r + j] = s * acc;
        }
    free(U);
    free(V);
}

/* Storage of one quantized matrix: 4-bit codes, one int8 scale code per 64-block, one fp32
 * constant per 256 blocks and the fp32 offset -- [QLoRA-paperclase, "Bits por parametro":
 * 4 + 8/64 + 32/(64*256) bits per parameter]. */
int64_t orc_nf4_storage_bytes(int64_t rows, int64_t cols)
{
    int64_t n = rows * cols, nb = n / 64, ng = (nb + 255) / 256;
    return n / 2 + nb + 4 * ng + 4;
}

/* Sampled adapter gradients for large shapes (same formulas as orc_layer_adapter_grads,
 * restricted to some rank indices j):
 *   dA[j, :] = s * sum_m V[m, j] X[m, :],  V[:, j] = G B[:, j]      (out [nj, K])
 *   dB[:, j] = s * sum_m G[m, :] U[m, j],  U[:, j] = X A[j, :]^T    (out [nj, N], i.e. transposed) */
void orc_layer_adapter_grads_cols(const uint16_t *X, const uint16_t *A, const uint16_t *B, const uint16_t *G,
                                  int64_t M, int64_t N, int64_t K, int64_t r, double alpha,
                                  const int64_t *jsel, int64_t nj, double *dA_rows, double *dB_cols)
{
    double s = alpha / (double)r;
    double *u = (double *)malloc(sizeof(double) * (size_t)M);
    double *v = (double *)malloc(sizeof(double) * (size_t)M);
    for (int64_t jj = 0; jj < nj; ++jj) {
        int64_t j = jsel[jj];
        for (int64_t m = 0; m < M; ++m) {
            double au = 0.0, av = 0.0;
            for (int64_t k = 0; k < K; ++k) au += orc_bf16_to_double(X[m * K + k]) * orc_bf16_to_double(A[j * K + k]);
            for (int64_t n = 0; n < N; ++n) av += orc_bf16_to_double(G[m * N + n]) * orc_bf16_to_double(B[n * r + j]);
            u[m] = au;
            v[m] = av;
        }
        for (int64_t k = 0; k < K; ++k) {
            double acc = 0.0;
            for (int64_t m = 0; m < M; ++m) acc += v[m] * orc_bf16_to_double(X[m * K + k]);
            dA_rows[jj * K + k] = s * acc;
        }
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t m = 0; m < M; ++m) acc += orc_bf16_to_double(G[m * N + n]) * u[m];
            dB_cols[jj * N + n] = s * acc;
        }
    }
    free(u);
    free(v);
}

/* ------------------------------------------------------------------------------------ */
/* Adapter merge ([QLoRA-ultralytics], "Compromissos" and "QLoRA e metodos relacionados":  */
/* to merge the adapters the base weight is first dequantized to 16 bits, and the merged   */
/* model keeps 16-bit weights):                                                            */
/*   W_m[n, k] = bf16(W^[n, k] + s sum_j B[n, j] A[j, k]),  s = alpha / r,                 */
/* with W^ the bf16 dequantized weight, the sum exact in fp64 from the bf16 adapters, and  */
/* one rounding to bf16 at the end (READING: the pages give no rounding order).            */
/* ------------------------------------------------------------------------------------ */
void orc_merge(const uint16_t *What, const uint16_t *A, const uint16_t *B, int64_t N, int64_t K, int64_t r,
               double alpha, uint16_t *out)
{
    double s = alpha / (double)r;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t k = 0; k < K; ++k) {
            double acc = 0.0;
            for (int64_t j = 0; j < r; ++j) acc += orc_bf16_to_double(B[n * r + j]) * orc_bf16_to_double(A[j * K + k]);
            out[n * K + k] = orc_bf16_round_d(orc_bf16_to_double(What[n * K + k]) + s * acc);
        }
    }
}

/* ------------------------------------------------------------------------------------ */
/* LoRA dropout on the adapter input ([coddykit], LoraConfig: lora_dropout=0.05): the       */
/* adapter branch sees x_d = x * mask / (1 - p) with mask ~ Bernoulli(1 - p) per element:    */
/*   h = W^ x + s B A x_d,   dX = G W^ + mask/(1-p) * (s (G B) A),                           */
/*   dA = s (G B)^T x_d,     dB = s G^T (x_d A^T).                                         */
/* READING (the pages give only p): the mask comes from the counter-based generator          */
/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",  */
/* SC'11): element e of the row-major [M, K] input uses word e % 4 of the block with counter */
/* (e / 4 as two 32-bit halves, offset as two 32-bit halves) and key (seed as two halves);  */
/* it is kept when word >= floor(p 2^32).                                                  */
/* ------------------------------------------------------------------------------------ */
static uint32_t mulhilo32(uint32_t a, uint32_t b, uint32_t *hi)
{
    uint64_t prod = (uint64_t)a * (uint64_t)b;
    *hi = (uint32_t)(prod >> 32);
    return (uint32_t)prod;
}

/* Philox4x32 with 10 rounds: each round multiplies counter words 0 and 2 by the round
 * multipliers, mixes the high halves with words 1, 3 and the key, and the key is bumped by
 * the Weyl constants between rounds. */
void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        uint32_t hi0, hi1;
        uint32_t lo0 = mulhilo32(0xD2511F53u, c0, &hi0);
        uint32_t lo1 = mulhilo32(0xCD9E8D57u, c2, &hi1);
        uint32_t n0 = hi1 ^ c1 ^ k0, n1 = lo1, n2 = hi0 ^ c3 ^ k1, n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* D[e] = 1 / (1 - p) where element e is kept, 0 where it is dropped (fp64), for e < n. */
void orc_dropout_scale(uint64_t seed, uint64_t offset, double p, int64_t n, double *D)
{
    uint32_t thr = (uint32_t)floor(p * 4294967296.0);
    double keep_scale = 1.0 / (1.0 - p);
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    for (int64_t e = 0; e < n; ++e) {
        uint64_t blk = (uint64_t)e / 4;
        uint32_t ctr[4] = {(uint32_t)blk, (uint32_t)(blk >> 32), (uint32_t)offset, (uint32_t)(offset >> 32)};
        uint32_t w[4];
        orc_philox4x32_10(ctr, key, w);
        D[e] = (w[e % 4] >= thr) ? keep_scale : 0.0;
    }
}

/* As orc_layer_fwd_rows, with the adapter input x * D (D [M, K] from orc_dropout_scale). */
void orc_layer_fwd_rows_drop(const uint16_t *What, const uint16_t *X, const uint16_t *A, const uint16_t *B,
                             int64_t M, int64_t N, int64_t K, int64_t r, double alpha, const double *D,
                             const int64_t *sel, int64_t nsel, double *Y_out, double *U_out)
{
    (void)M;
    double s = alpha / (double)r;
    double *u = (double *)malloc(sizeof(double) * (size_t)(r > 0 ? r : 1));
    for (int64_t ii = 0; ii < nsel; ++ii) {
        int64_t m = sel[ii];
        for (int64_t j = 0; j < r; ++j) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += orc_bf16_to_double(X[m * K + k]) * D[m * K + k] * orc_bf16_to_double(A[j * K + k]);
            u[j] = acc;
            if (U_out) U_out[ii * r + j] = acc;
        }
        for (int64_t n = 0; n < N; ++n) {
            double base = 0.0;
            for (int64_t k = 0; k < K; ++k) base += orc_bf16_to_double(X[m * K + k]) * orc_bf16_to_double(What[n * K + k]);
            double lora = 0.0;
            for (int64_t j = 0; j < r; ++j) lora += u[j] * orc_bf16_to_double(B[n * r + j]);
            Y_out[ii * N + n] = base + s * lora;
        }
    }
    free(u);
}

/* As orc_layer_dx_rows, with the adapter branch's input gradient multiplied by D. */
void orc_layer_dx_rows_drop(const uint16_t *What, const uint16_t *A, const uint16_t *B, const uint16_t *G,
                            int64_t M, int64_t N, int64_t K, int64_t r, double alpha, const double *D,
                            const int64_t *sel, int64_t nsel, double *dX_out)
{
    (void)M;
    double s = alpha / (double)r;
    double *v = (double *)malloc(sizeof(double) * (size_t)(r > 0 ? r : 1));
    double *row = (double *)malloc(sizeof(double) * (size_t)K);
    for (int64_t ii = 0; ii < nsel; ++ii) {
        int64_t m = sel[ii];
        for (int64_t j = 0; j < r; ++j) {
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n) acc += orc_bf16_to_double(G[m * N + n]) * orc_bf16_to_double(B[n * r + j]);
            v[j] = acc;
        }
        for (int64_t k = 0; k < K; ++k) row[k] = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            double g = orc_bf16_to_double(G[m * N + n]);
            for (int64_t k = 0; k < K; ++k) row[k] += g * orc_bf16_to_double(What[n * K + k]);
        }
        for (int64_t k = 0; k < K; ++k) {
            double lora = 0.0;
            for (int64_t j = 0; j < r; ++j) lora += v[j] * orc_bf16_to_double(A[j * K + k]);
            dX_out[ii * K + k] = row[k] + D[m * K + k] * s * lora;
        }
    }
    free(v);
    free(row);
}

/* As orc_layer_adapter_grads, with the adapter input x * D. */
void orc_layer_adapter_grads_drop(const uint16_t *X, const uint16_t *A, const uint16_t *B, const uint16_t *G,
                                  int64_t M, int64_t N, int64_t K, int64_t r, double alpha, const double *D,
                                  double *dA_out, double *dB_out)
{
    double s = alpha / (double)r;
    double *U = (double *)calloc((size_t)(M * r), sizeof(double));
    double *V = (double *)calloc((size_t)(M * r), sizeof(double));
    for (int64_t m = 0; m < M; ++m)
        for (int64_t j = 0; j < r; ++j) {
            double au = 0.0, av = 0.0;
            for (int64_t k = 0; k < K; ++k)
                au += orc_bf16_to_double(X[m * K + k]) * D[m * K + k] * orc_bf16_to_double(A[j * K + k]);
            for (int64_t n = 0; n < N; ++n) av += orc_bf16_to_double(G[m * N + n]) * orc_bf16_to_double(B[n * r + j]);
            U[m * r + j] = au;
            V[m * r + j] = av;
        }
    for (int64_t j = 0; j < r; ++j)
        for (int64_t k = 0; k < K; ++k) {
            double acc = 0.0;
            for (int64_t m = 0; m < M; ++m) acc += V[m * r + j] * orc_bf16_to_double(X[m * K + k]) * D[m * K + k];
            dA_out[j * K + k] = s * acc;
        }
    for (int64_t n = 0; n < N; ++n)
        for (int64_t j = 0; j < r; ++j) {
            double acc = 0.0;
            for (int64_t m = 0; m < M; ++m) acc += orc_bf16_to_double(G[m * N + n]) * U[m * r + j];
            dB_out[n * r + j] = s * acc;
        }
    free(U);
    free(V);
}

/* ------------------------------------------------------------------------------------ */
/* The adapters' optimizer step.  Only the two LoRA matrices are updated [QLoRA-ultralytics,   */
/* "Como funciona a QLoRA"]; their optimizer states are paged: kept in NVIDIA unified memory  */
/* and moved to CPU RAM under memory pressure [QLoRA-ultralytics, "Otimizadores paginados"    */
/* bullet; QLoRA-skillverse, "Componentes clave", "Optimizadores paginados"].  READING: the    */
/* pages name no update rule; the optimizer is AdamW (decoupled weight decay, Loshchilov and  */
/* Hutter, ICLR 2019), step t >= 1:                                                           */
/*   p <- p (1 - lr wd);  m <- b1 m + (1 - b1) g;  v <- b2 v + (1 - b2) g^2;                   */
/*   p <- p - lr (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps).                            */
/* In fp64 on fp32 inputs; the caller rounds.                                              */
/* ------------------------------------------------------------------------------------ */
void orc_adamw_step(double *p, const double *g, double *m, double *v, int64_t n, double lr, double b1, double b2,
                    double eps, double wd, int64_t t)
{
    double bc1 = 1.0 - pow(b1, (double)t), bc2 = 1.0 - pow(b2, (double)t);
    for (int64_t i = 0; i < n; ++i) {
        p[i] *= 1.0 - lr * wd;
        m[i] = b1 * m[i] + (1.0 - b1) * g[i];
        v[i] = b2 * v[i] + (1.0 - b2) * g[i] * g[i];
        p[i] -= lr * (m[i] / bc1) / (sqrt(v[i] / bc2) + eps);
    }
}
