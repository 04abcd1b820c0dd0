/*
 * oracle.c -- the CPU oracle for the ternary-g128 matrix product and the
 * normalized Sylvester-Walsh-Hadamard rotation.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is plain, slow, obviously correct C
 * that the tests, the smoke check and the benchmark's CPU-baseline leg use to
 * check the CUDA library.  The library never links, loads or calls it, and it
 * shares no code, header, table or helper with the library.
 *
 * Sources (the web pages this method is described on):
 *   [card]  "prism-ml/Ternary-Bonsai-27B-mlx-2bit - Hugging Face" model card,
 *           sections "Weight representation: ternary g128", "Memory
 *           requirement", "MLX packaging", "CUDA (NVIDIA GPUs)".
 *   [post]  "Ternary-Bonsai-2-9B-2bit" article, section 3 "Ternary weights and
 *           Hadamard rotation".
 *
 * What is computed, and the readings taken where the pages are silent:
 *   - A weight is t * s_g with t in {-1, 0, +1} and one FP16 scale s_g per 128
 *     consecutive weights along K ([card] "Weight representation").
 *   - Each t sits in a 2-bit slot ([card] "Memory requirement").  The code is
 *     q = t + 1 in {0, 1, 2}; q = 3 is invalid.  Sixteen codes fill one
 *     little-endian uint32, code k of a row in bits 2*(k%16) .. 2*(k%16)+1 of
 *     word k/16 of that row.  Rows are contiguous along K.  Scales are
 *     [N][K/128] row-major.
 *   - y[m][n] = sum_k x[m][k] * (q[n][k] - 1) * s[n][k/128], evaluated in
 *     double.  Every product of a bf16, a fp16 and +-1 is exact in double.
 *   - The rotation is x' = H_B (s (.) x) / sqrt(B) per block of B = 4096 along
 *     the last dimension, H_B the Sylvester (natural-order) Hadamard matrix
 *     H[i][j] = (-1)^popcount(i & j), and s an explicit +-1 sign vector
 *     ([post] section 3).  The inverse is x = s (.) (H_B x' / sqrt(B)).
 *
 *   - The 1-bit sibling ("binary g128"): the card names it at 1.125 bits per
 *     weight ([card] "Highlights" and "Benchmarks"), one bit per weight
 *     plus the same FP16 scale per 128.  The card's MLX packing (s_mlx = 2 s_g,
 *     bias = -s_g, [card] "MLX packaging") reproduces exactly +-s_g from a
 *     bit b in {0, 1}, so a weight is (2b - 1) * s_g.  Reading for the unstated
 *     order, as for the ternary codes: bit k%32 of little-endian uint32 word
 *     k/32 of the row.
 *   - The affine pack ([card] "MLX packaging": a scale and a bias per group):
 *     the same 2-bit slots with all four codes valid and w = s q + b, s and b
 *     FP16 per 128 weights.  Reading for the unstated order and precision: the
 *     slot order of the ternary codes, and FP16 biases like the scales.
 *
 *   - Native base-3 packing: the card gives the information content of a
 *     trit (log2 3, about 1.585 bits) and the 1.71 bits/weight it implies with
 *     the scale, and names packing at that density as future work ([card]
 *     "Weight representation" and "Memory requirement").  It gives no layout.
 *     Reading: five trits per byte, byte = q0 + 3 q1 + 9 q2 + 27 q3 + 81 q4
 *     (values 0..242) with q = t + 1 and trit i of the byte at K position
 *     5 j + i of its group; a 128-weight group is 25 such bytes and a 26th
 *     holding trits 125..127 as q0 + 3 q1 + 9 q2 (values 0..26); rows are
 *     [N][26 K/128] bytes.  That is 26 * 8 / 128 + 16 / 128 = 1.75 bits per
 *     weight with the FP16 scale.
 *
 * Parity pins live in the "not gpu" tests: brute-force dense matmul from an
 * explicitly expanded W, exhaustive pack/unpack patterns, the explicit
 * Hadamard matrix for n <= 64, H*H = n*I, Parseval, closed forms on e_0 and
 * constant vectors, power-of-two linearity in the scales, one-hot columns, the
 * bit-rate figures the card prints, and for the 1-bit and affine forms their
 * bit-exact agreement with the ternary product where the weights coincide
 * (w = +-s; b = -s) and with the 1-bit product for the card's MLX pair.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Number formats, decoded field by field (exact).                          */
/* ------------------------------------------------------------------------ */

/* bfloat16 bit pattern -> double.  bf16 is the top half of an IEEE binary32. */
double orc_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE binary16 bit pattern -> double: sign, 5-bit exponent (bias 15),
 * 10-bit fraction; exponent 0 is subnormal (fraction * 2^-24). */
double orc_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m + 1024), e - 25);
    return sign ? -v : v;
}

/* ------------------------------------------------------------------------ */
/* Packing: t in {-1,0,1} -> 2-bit code q = t + 1, 16 codes per uint32.      */
/* ------------------------------------------------------------------------ */

/* Packs t[N][K] into codes[N][K/16].  An entry outside {-1,0,1} is counted
 * and stored as the invalid code 3, so that a later validation rejects it.
 * Returns the number of invalid entries, or -1 if K is not a multiple of 16. */
long long orc_pack(const int8_t *t, int N, int K, uint32_t *codes)
{
    if (N < 0 || K < 0 || K % 16 != 0)
        return -1;
    long long bad = 0;
    int W = K / 16;
    for (int n = 0; n < N; ++n) {
        for (int w = 0; w < W; ++w) {
            uint32_t word = 0;
            for (int i = 0; i < 16; ++i) {
                int v = t[(size_t)n * K + (size_t)w * 16 + i];
                uint32_t q;
                if (v == -1)
                    q = 0;
                else if (v == 0)
                    q = 1;
                else if (v == 1)
                    q = 2;
                else {
                    q = 3;
                    ++bad;
                }
                word |= q << (2 * i);
            }
            codes[(size_t)n * W + w] = word;
        }
    }
    return bad;
}

/* One code, read straight from the definition of the layout. */
static int orc_code(const uint32_t *codes, int K, int n, int k)
{
    uint32_t word = codes[(size_t)n * (K / 16) + k / 16];
    return (int)((word >> (2 * (k % 16))) & 3u);
}

/* Unpacks codes[N][K/16] into t[N][K] = q - 1.  Code 3 is invalid: it is
 * counted and written as 0.  Returns the count, or -1 on a bad K. */
long long orc_unpack(const uint32_t *codes, int N, int K, int8_t *t)
{
    if (N < 0 || K < 0 || K % 16 != 0)
        return -1;
    long long bad = 0;
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k) {
            int q = orc_code(codes, K, n, k);
            if (q == 3) {
                ++bad;
                t[(size_t)n * K + k] = 0;
            } else {
                t[(size_t)n * K + k] = (int8_t)(q - 1);
            }
        }
    return bad;
}

/* ------------------------------------------------------------------------ */
/* The matrix product, straight from its definition.                        */
/* ------------------------------------------------------------------------ */

/* One output: y = sum_k x[m][k] * (q[n][k]-1) * s[n][k/128] and the error
 * scale a = sum_k |x[m][k] * w[n][k]|.  Returns 0, or -1 if a code is 3. */
static int orc_dot(const uint16_t *x, const uint32_t *codes,
                   const uint16_t *scales, int K, int m, int n,
                   double *y, double *a)
{
    int G = K / 128;
    double acc = 0.0, mag = 0.0;
    for (int k = 0; k < K; ++k) {
        int q = orc_code(codes, K, n, k);
        if (q == 3)
            return -1;
        double w = (double)(q - 1) * orc_f16_to_f64(scales[(size_t)n * G + k / 128]);
        double p = orc_bf16_to_f64(x[(size_t)m * K + k]) * w;
        acc += p;
        mag += fabs(p);
    }
    *y = acc;
    if (a)
        *a = mag;
    return 0;
}

static void orc_set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* y[M][N] (and a[M][N] if a != NULL) for x bf16 [M][K], codes [N][K/16],
 * scales fp16 [N][K/128].  nthreads > 0 sets the OpenMP thread count (the
 * loop over outputs is the only parallel part).  Returns 0, -1 for a code 3,
 * or -2 for a bad shape. */
int orc_matmul(const uint16_t *x, const uint32_t *codes, const uint16_t *scales,
               int M, int N, int K, double *y, double *a, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || K % 128 != 0)
        return -2;
    orc_set_threads(nthreads);
    int status = 0;
    long long total = (long long)M * N;
#pragma omp parallel for schedule(dynamic, 16)
    for (long long i = 0; i < total; ++i) {
        int m = (int)(i / N), n = (int)(i % N);
        double yy, aa;
        if (orc_dot(x, codes, scales, K, m, n, &yy, &aa) != 0) {
            status = -1;
            yy = NAN;
            aa = NAN;
        }
        y[i] = yy;
        if (a)
            a[i] = aa;
    }
    return status;
}

/* The same product at chosen outputs only: (ms[i], ns[i]) for i < count. */
int orc_matmul_sampled(const uint16_t *x, const uint32_t *codes,
                       const uint16_t *scales, int K, const int *ms,
                       const int *ns, int count, double *y, double *a,
                       int nthreads)
{
    if (K < 0 || K % 128 != 0)
        return -2;
    orc_set_threads(nthreads);
    int status = 0;
#pragma omp parallel for schedule(dynamic, 4)
    for (int i = 0; i < count; ++i) {
        double yy, aa;
        if (orc_dot(x, codes, scales, K, ms[i], ns[i], &yy, &aa) != 0) {
            status = -1;
            yy = NAN;
            aa = NAN;
        }
        y[i] = yy;
        if (a)
            a[i] = aa;
    }
    return status;
}

/* ------------------------------------------------------------------------ */
/* The 1-bit sibling: b in {0, 1}, w = (2b - 1) * s_g, 32 bits per uint32.   */
/* ------------------------------------------------------------------------ */

/* Packs t[N][K] in {-1, +1} into words[N][K/32]: bit k%32 of word k/32 is 1
 * for t = +1.  Any other entry is counted and stored as 0 (t = -1).  Returns
 * the count, or -1 if K is not a multiple of 32. */
long long orc_bin_pack(const int8_t *t, int N, int K, uint32_t *words)
{
    if (N < 0 || K < 0 || K % 32 != 0)
        return -1;
    long long bad = 0;
    int W = K / 32;
    for (int n = 0; n < N; ++n)
        for (int w = 0; w < W; ++w) {
            uint32_t word = 0;
            for (int i = 0; i < 32; ++i) {
                int v = t[(size_t)n * K + (size_t)w * 32 + i];
                if (v == 1)
                    word |= 1u << i;
                else if (v != -1)
                    ++bad;
            }
            words[(size_t)n * W + w] = word;
        }
    return bad;
}

/* One bit, read straight from the layout. */
static int orc_bit(const uint32_t *words, int K, int n, int k)
{
    return (int)((words[(size_t)n * (K / 32) + k / 32] >> (k % 32)) & 1u);
}

/* Unpacks words[N][K/32] into t[N][K] = 2b - 1.  Returns 0, or -1 on a bad K. */
int orc_bin_unpack(const uint32_t *words, int N, int K, int8_t *t)
{
    if (N < 0 || K < 0 || K % 32 != 0)
        return -1;
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            t[(size_t)n * K + k] = (int8_t)(2 * orc_bit(words, K, n, k) - 1);
    return 0;
}

/* One output of the binary product: y = sum_k x[m][k] (2b[n][k] - 1) s[n][k/128]
 * and a = sum_k |x[m][k] w[n][k]|. */
static void orc_bin_dot(const uint16_t *x, const uint32_t *words,
                        const uint16_t *scales, int K, int m, int n,
                        double *y, double *a)
{
    int G = K / 128;
    double acc = 0.0, mag = 0.0;
    for (int k = 0; k < K; ++k) {
        double w = (double)(2 * orc_bit(words, K, n, k) - 1) *
                   orc_f16_to_f64(scales[(size_t)n * G + k / 128]);
        double p = orc_bf16_to_f64(x[(size_t)m * K + k]) * w;
        acc += p;
        mag += fabs(p);
    }
    *y = acc;
    if (a)
        *a = mag;
}

/* y[M][N] (and a[M][N] if a != NULL) for x bf16 [M][K], words [N][K/32],
 * scales fp16 [N][K/128].  Returns 0, or -2 for a bad shape. */
int orc_bin_matmul(const uint16_t *x, const uint32_t *words, const uint16_t *scales,
                   int M, int N, int K, double *y, double *a, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || K % 128 != 0)
        return -2;
    orc_set_threads(nthreads);
    long long total = (long long)M * N;
#pragma omp parallel for schedule(dynamic, 16)
    for (long long i = 0; i < total; ++i) {
        double yy, aa;
        orc_bin_dot(x, words, scales, K, (int)(i / N), (int)(i % N), &yy, &aa);
        y[i] = yy;
        if (a)
            a[i] = aa;
    }
    return 0;
}

/* The binary product at chosen outputs only: (ms[i], ns[i]) for i < count. */
int orc_bin_matmul_sampled(const uint16_t *x, const uint32_t *words,
                           const uint16_t *scales, int K, const int *ms,
                           const int *ns, int count, double *y, double *a,
                           int nthreads)
{
    if (K < 0 || K % 128 != 0)
        return -2;
    orc_set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 4)
    for (int i = 0; i < count; ++i) {
        double yy, aa;
        orc_bin_dot(x, words, scales, K, ms[i], ns[i], &yy, &aa);
        y[i] = yy;
        if (a)
            a[i] = aa;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* The group-size-64 pack ([card] "Shipped components"): the same g128       */
/* weights, each scale repeated in both 64-value halves of its group.        */
/* ------------------------------------------------------------------------ */

/* s128[n][g] = s64[n][2g] for fp16 bit patterns s64 [N][K/64].  A group
 * whose two halves differ (bit for bit) is counted; its first half's scale is
 * kept.  Returns the count, or -1 if K is not a multiple of 128. */
long long orc_scales_from_g64(const uint16_t *s64, int N, int K, uint16_t *s128)
{
    if (N < 0 || K < 0 || K % 128 != 0)
        return -1;
    long long bad = 0;
    int G = K / 128;
    for (int n = 0; n < N; ++n)
        for (int g = 0; g < G; ++g) {
            uint16_t a = s64[(size_t)n * 2 * G + 2 * g], b = s64[(size_t)n * 2 * G + 2 * g + 1];
            if (a != b)
                ++bad;
            s128[(size_t)n * G + g] = a;
        }
    return bad;
}

/* ------------------------------------------------------------------------ */
/* MLX affine 2-bit dequantisation, w = s_mlx * q + bias, in float.          */
/* ([card] "MLX packaging": a group stores a scale and a bias.)              */
/* ------------------------------------------------------------------------ */

float orc_mlx_affine(int q, float s_mlx, float bias)
{
    return s_mlx * (float)q + bias;
}

/* The product on an affine pack: the same 2-bit slots, every code 0..3
 * valid, and per group a FP16 scale s and a FP16 bias b, so that
 * w[n][k] = s[n][k/128] * q[n][k] + b[n][k/128] ([card] "MLX packaging";
 * the ternary codes are the case b = -s, the card's literal pair
 * (2 s_g, -s_g) on codes {0, 1} the 1-bit case).  One output and its error
 * scale a = sum_k |x w|; every term is exact in double. */
static void orc_affine_dot(const uint16_t *x, const uint32_t *codes,
                           const uint16_t *scales, const uint16_t *biases,
                           int K, int m, int n, double *y, double *a)
{
    int G = K / 128;
    double acc = 0.0, mag = 0.0;
    for (int k = 0; k < K; ++k) {
        int q = orc_code(codes, K, n, k);
        size_t g = (size_t)n * G + k / 128;
        double w = orc_f16_to_f64(scales[g]) * (double)q + orc_f16_to_f64(biases[g]);
        double p = orc_bf16_to_f64(x[(size_t)m * K + k]) * w;
        acc += p;
        mag += fabs(p);
    }
    *y = acc;
    if (a)
        *a = mag;
}

/* y[M][N] (and a[M][N] if a != NULL) for x bf16 [M][K], codes [N][K/16],
 * scales and biases fp16 [N][K/128].  Returns 0, or -2 for a bad shape. */
int orc_affine_matmul(const uint16_t *x, const uint32_t *codes, const uint16_t *scales,
                      const uint16_t *biases, int M, int N, int K, double *y,
                      double *a, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || K % 128 != 0)
        return -2;
    orc_set_threads(nthreads);
    long long total = (long long)M * N;
#pragma omp parallel for schedule(dynamic, 16)
    for (long long i = 0; i < total; ++i) {
        double yy, aa;
        orc_affine_dot(x, codes, scales, biases, K, (int)(i / N), (int)(i % N), &yy, &aa);
        y[i] = yy;
        if (a)
            a[i] = aa;
    }
    return 0;
}

/* The affine product at chosen outputs only: (ms[i], ns[i]) for i < count. */
int orc_affine_matmul_sampled(const uint16_t *x, const uint32_t *codes,
                              const uint16_t *scales, const uint16_t *biases,
                              int K, const int *ms, const int *ns, int count,
                              double *y, double *a, int nthreads)
{
    if (K < 0 || K % 128 != 0)
        return -2;
    orc_set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 4)
    for (int i = 0; i < count; ++i) {
        double yy, aa;
        orc_affine_dot(x, codes, scales, biases, K, ms[i], ns[i], &yy, &aa);
        y[i] = yy;
        if (a)
            a[i] = aa;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Walsh-Hadamard transform in Sylvester (natural) order.                    */
/* ------------------------------------------------------------------------ */

/* H_n as a dense n*n matrix by the Sylvester recursion H_1 = [1],
 * H_2n = [[H_n, H_n], [H_n, -H_n]].  n must be a power of two. */
int orc_hadamard_explicit(int n, double *H)
{
    if (n < 1 || (n & (n - 1)) != 0)
        return -1;
    H[0] = 1.0;
    for (int h = 1; h < n; h *= 2) {
        for (int i = 0; i < h; ++i)
            for (int j = 0; j < h; ++j) {
                double v = H[(size_t)i * n + j];
                H[(size_t)i * n + j + h] = v;
                H[(size_t)(i + h) * n + j] = v;
                H[(size_t)(i + h) * n + j + h] = -v;
            }
    }
    return 0;
}

/* In place, unnormalized: v <- H_n v, by radix-2 butterflies
 * (a, b) -> (a + b, a - b) over strides 1, 2, 4, ..., n/2. */
int orc_fwht(double *v, int n)
{
    if (n < 1 || (n & (n - 1)) != 0)
        return -1;
    for (int h = 1; h < n; h *= 2)
        for (int i = 0; i < n; i += 2 * h)
            for (int j = i; j < i + h; ++j) {
                double a = v[j], b = v[j + h];
                v[j] = a + b;
                v[j + h] = a - b;
            }
    return 0;
}

/* The rotation of the activation's last dimension ([post] section 3):
 * for each row m and each block of B consecutive positions,
 * out = H_B (s (.) x) / sqrt(B).  x is bf16 [M][K], signs int8 [K] (+-1),
 * out double [M][K].  B a power of two dividing K. */
int orc_rotate(const uint16_t *x, const int8_t *signs, int M, int K, int B,
               double *out)
{
    if (B < 1 || (B & (B - 1)) != 0 || K % B != 0 || M < 0)
        return -1;
    double norm = 1.0 / sqrt((double)B);
    for (int m = 0; m < M; ++m)
        for (int b0 = 0; b0 < K; b0 += B) {
            double *v = out + (size_t)m * K + b0;
            for (int i = 0; i < B; ++i)
                v[i] = (double)signs[b0 + i] * orc_bf16_to_f64(x[(size_t)m * K + b0 + i]);
            orc_fwht(v, B);
            for (int i = 0; i < B; ++i)
                v[i] *= norm;
        }
    return 0;
}

/* The inverse rotation: x = s (.) (H_B x' / sqrt(B)), x' double [M][K]. */
int orc_unrotate(const double *xr, const int8_t *signs, int M, int K, int B,
                 double *out)
{
    if (B < 1 || (B & (B - 1)) != 0 || K % B != 0 || M < 0)
        return -1;
    double norm = 1.0 / sqrt((double)B);
    for (int m = 0; m < M; ++m)
        for (int b0 = 0; b0 < K; b0 += B) {
            double *v = out + (size_t)m * K + b0;
            memcpy(v, xr + (size_t)m * K + b0, sizeof(double) * (size_t)B);
            orc_fwht(v, B);
            for (int i = 0; i < B; ++i)
                v[i] *= norm * (double)signs[b0 + i];
        }
    return 0;
}

/* The rotated product: y = (rotate(x)) W^T with the rotated activation kept
 * in double, as the fused path keeps it on chip. */
int orc_rotate_matmul(const uint16_t *x, const int8_t *signs,
                      const uint32_t *codes, const uint16_t *scales, int M,
                      int N, int K, int B, double *y, double *a, int nthreads)
{
    if (M < 0 || N < 0 || K % 128 != 0)
        return -2;
    double *xr = (double *)malloc(sizeof(double) * (size_t)M * (size_t)K + 1);
    if (!xr)
        return -3;
    if (orc_rotate(x, signs, M, K, B, xr) != 0) {
        free(xr);
        return -2;
    }
    orc_set_threads(nthreads);
    int G = K / 128, status = 0;
    long long total = (long long)M * N;
#pragma omp parallel for schedule(dynamic, 16)
    for (long long i = 0; i < total; ++i) {
        int m = (int)(i / N), n = (int)(i % N);
        double acc = 0.0, mag = 0.0;
        for (int k = 0; k < K; ++k) {
            int q = orc_code(codes, K, n, k);
            if (q == 3) {
                status = -1;
                break;
            }
            double p = xr[(size_t)m * K + k] * (double)(q - 1) *
                       orc_f16_to_f64(scales[(size_t)n * G + k / 128]);
            acc += p;
            mag += fabs(p);
        }
        y[i] = acc;
        if (a)
            a[i] = mag;
    }
    free(xr);
    return status;
}

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Native base-3 packing (five trits per byte; see the header).              */
/* ------------------------------------------------------------------------ */

/* Trits per byte j of a group: 5, and 3 for the last one. */
static int orc_f3_count(int j) { return j < 25 ? 5 : 3; }

/* Packs t[N][K] in {-1,0,1} into out[N][26 K/128].  Returns the count of
 * entries outside {-1,0,1} (packed as 0), or -1 if K is not a multiple of
 * 128. */
long long orc_f3_pack(const int8_t *t, int N, int K, uint8_t *out)
{
    if (N < 0 || K < 0 || K % 128 != 0)
        return -1;
    long long bad = 0;
    int G = K / 128;
    for (int n = 0; n < N; ++n)
        for (int g = 0; g < G; ++g)
            for (int j = 0; j < 26; ++j) {
                int v = 0, p = 1;
                for (int i = 0; i < orc_f3_count(j); ++i) {
                    int tv = t[(size_t)n * K + (size_t)g * 128 + 5 * j + i];
                    int q = tv + 1;
                    if (q < 0 || q > 2) {
                        ++bad;
                        q = 0;
                    }
                    v += q * p;
                    p *= 3;
                }
                out[(size_t)n * G * 26 + (size_t)g * 26 + j] = (uint8_t)v;
            }
    return bad;
}

/* Digit i of a byte in base 3, by repeated division. */
static int orc_f3_digit(int v, int i)
{
    for (int r = 0; r < i; ++r)
        v /= 3;
    return v % 3;
}

/* Unpacks in[N][26 K/128] into t[N][K].  Returns the count of bytes out of
 * range (above 242, or above 26 for a group's last byte), or -1 on a bad K. */
long long orc_f3_unpack(const uint8_t *in, int N, int K, int8_t *t)
{
    if (N < 0 || K < 0 || K % 128 != 0)
        return -1;
    long long bad = 0;
    int G = K / 128;
    for (int n = 0; n < N; ++n)
        for (int g = 0; g < G; ++g)
            for (int j = 0; j < 26; ++j) {
                int v = in[(size_t)n * G * 26 + (size_t)g * 26 + j];
                if (v > (j < 25 ? 242 : 26))
                    ++bad;
                for (int i = 0; i < orc_f3_count(j); ++i)
                    t[(size_t)n * K + (size_t)g * 128 + 5 * j + i] = (int8_t)(orc_f3_digit(v, i) - 1);
            }
    return bad;
}

/* y[m][n] = sum_k x[m][k] (q[n][k] - 1) s[n][k/128] from the base-3 bytes, in
 * double, and a[m][n] = sum_k |x w| if a != NULL.  Returns 0, or -2 for a bad
 * shape. */
int orc_f3_matmul(const uint16_t *x, const uint8_t *packed, const uint16_t *scales, int M, int N, int K,
                  double *y, double *a, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || K % 128 != 0)
        return -2;
    orc_set_threads(nthreads);
    int G = K / 128;
    long long total = (long long)M * N;
#pragma omp parallel for schedule(dynamic, 16)
    for (long long i = 0; i < total; ++i) {
        int m = (int)(i / N), n = (int)(i % N);
        double acc = 0.0, mag = 0.0;
        for (int g = 0; g < G; ++g) {
            double sg = orc_f16_to_f64(scales[(size_t)n * G + g]);
            for (int j = 0; j < 26; ++j) {
                int v = packed[(size_t)n * G * 26 + (size_t)g * 26 + j];
                for (int q = 0; q < orc_f3_count(j); ++q) {
                    int k = g * 128 + 5 * j + q;
                    double p = orc_bf16_to_f64(x[(size_t)m * K + k]) * (double)(orc_f3_digit(v, q) - 1) * sg;
                    acc += p;
                    mag += fabs(p);
                }
            }
        }
        y[i] = acc;
        if (a)
            a[i] = mag;
    }
    return 0;
}

