/*
 * oracle.c -- plain, slow, obviously-correct CPU oracle for the W4A4 NVFP4
 * quantised projection.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * includes this file; only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark use it.  It shares no code, header, table or constant
 * generator with the CUDA path.
 *
 * What it follows (citations are page title + section):
 *   - FoldQuantVLA, Key Contribution 1 ("consistent folding", Proposition 1):
 *     one transformed activation basis, its inverse folded into the weight.
 *   - FoldQuantVLA, Key Contribution 2: channel scaling, block Hadamard rotation
 *     by the fast Walsh-Hadamard transform with block size beta = 64, dynamic
 *     per-token quantisation (no timestep-indexed scale tables).
 *   - QuantWAMs sec. 3.1, Eq. (1): the quantiser input is the transformed
 *     activation; the top-K channels of that basis stay in 16-bit (Fig. 1(d):
 *     FP16; sec. 4 "Quantization configuration": the exception path).
 *   - Q-WAM abstract: a tiny 16-bit low-rank branch plus 4-bit weights and
 *     activations for the complement, both dense matmuls.
 *   - LatentQuant abstract / QuantWAMs sec. 4 "Backend": NVFP4 W4A4.  NVFP4 is
 *     taken as: e2m1 element codes {0, 0.5, 1, 1.5, 2, 3, 4, 6} (+sign), one
 *     unsigned e4m3 scale per 16 consecutive K elements, one fp32 tensor scale.
 *
 * Readings fixed here (the pages leave them open):
 *   - smoothing is applied before the rotation (xs = x * inv_s, then FWHT) in the
 *     default order (FoldQuantVLA, Key Contribution 2: "channel scaling, block
 *     Hadamard"); the other order, rotation first (QuantWAMs sec. 3.1 Eq. (1):
 *     A R S^-1), is the `smooth_after` flag: xt = FWHT(x) * inv_s, with the fold
 *     R' = S H (W - P Q) and P = bf16(H S^-1 L1);
 *   - activations carry one fp32 scale per row, g = amax_row / (6 * 448);
 *     weights carry one per tensor;
 *   - block scale  sc = e4m3_rne_satfinite((bmax / 6) / g),
 *     dequant step d  = dec(sc) * g, code = e2m1_rne_satfinite(v / d)
 *     (code 0 when d == 0); every step is one IEEE fp32 operation, rounded
 *     to nearest even, no fused multiply-add;
 *   - e2m1 keeps the sign of its input (so -0.1 encodes as 0x8);
 *   - the low-rank factors are stored in bf16 with diag(s)^-1 folded into the
 *     down-projection: P = bf16(fp32(L1 * inv_s)), Q = bf16(L2); the weight
 *     complement is R = diag(s) (W - P Q) so the three branches recompose
 *     x W exactly in exact arithmetic;
 *   - the low-rank activation U = x P is rounded to bf16 (16-bit branch);
 *     outlier activations and weight rows are rounded to fp16.
 *
 * Parity pins (tests/test_oracle_pins.py): FWHT against the dense Sylvester
 * matrix, self-inverse and orthonormality; e2m1/e4m3 encoders exhaustively
 * against an independent IEEE ulp-grid rounding; round trips of representable
 * blocks; Proposition 1 folding invariance; reduction to a plain matmul;
 * bf16 rounding of fp64 values and U = bf16(x P) against exact rational
 * arithmetic rounded once (ties and their fp64 neighbours included); x_Omega
 * against the dense Sylvester product on exactly transformable rows; the int8
 * weight quantiser against numpy.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ formats */

/* e2m1 magnitudes indexed by the 3-bit magnitude code. */
static const double kE2M1[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_decode(uint8_t code)
{
    double m = kE2M1[code & 7];
    return (code & 8) ? -m : m;
}

/* Nearest e2m1 value to v; on an exact tie the even magnitude code wins;
 * |v| >= 6 saturates to 6; the sign of v is kept. */
uint8_t orc_e2m1_encode(float v)
{
    int neg = signbit(v) ? 1 : 0;
    double a = fabs((double)v);
    int best = 0;
    if (a >= 6.0) {
        best = 7;
    } else {
        double bd = a;                          /* distance to code 0 */
        for (int c = 1; c < 8; ++c) {
            double d = fabs(a - kE2M1[c]);
            if (d < bd || (d == bd && (c & 1) == 0)) {
                best = c;
                bd = d;
            }
        }
    }
    return (uint8_t)(best | (neg << 3));
}

/* Unsigned e4m3 (4 exponent bits, bias 7, 3 mantissa bits, no infinities,
 * code 0x7F is NaN and never produced; largest finite 0x7E = 448). */
double orc_e4m3_decode(uint8_t code)
{
    int e = (code >> 3) & 15, m = code & 7;
    if (e == 0) return ldexp((double)m, -9);            /* m/8 * 2^-6 */
    return ldexp(1.0 + m / 8.0, e - 7);
}

/* Nearest non-negative finite e4m3 value to v >= 0; tie -> even code;
 * v >= 448 saturates to 448. */
uint8_t orc_e4m3_encode(float v)
{
    double a = (double)v;
    if (!(a > 0.0)) return 0;
    if (a >= 448.0) return 0x7E;
    /* binary search for the first code whose value is >= a */
    int lo = 0, hi = 0x7E;
    while (lo < hi) {
        int mid = (lo + hi) / 2;
        if (orc_e4m3_decode((uint8_t)mid) >= a) hi = mid; else lo = mid + 1;
    }
    if (lo == 0) return 0;
    double up = orc_e4m3_decode((uint8_t)lo), dn = orc_e4m3_decode((uint8_t)(lo - 1));
    double du = up - a, dd = a - dn;
    if (du < dd) return (uint8_t)lo;
    if (dd < du) return (uint8_t)(lo - 1);
    return (uint8_t)((lo & 1) ? lo - 1 : lo);
}

/* fp32 -> bf16 bits, round to nearest even (IEEE). */
uint16_t orc_bf16_from_f32(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x7FFFFFu)) return 0x7FC0;
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

float orc_f32_from_bf16(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* fp64 -> bf16 bits with a single round-to-nearest-even. */
uint16_t orc_bf16_from_f64(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    int e;
    (void)frexp(a, &e);                     /* a = m 2^e, m in [0.5, 1) */
    int q = e - 8;                          /* quantum of an 8-bit significand */
    if (q < -133) q = -133;                 /* bf16 subnormal quantum */
    double r = nearbyint(ldexp(a, -q));     /* default rounding: nearest even */
    float f = (float)ldexp(r, q);           /* exact, or overflows to inf */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(sign | (u >> 16));
}

uint16_t orc_f16_from_f32(float f)
{
    _Float16 h = (_Float16)f;               /* IEEE conversion, nearest even */
    uint16_t b;
    memcpy(&b, &h, 2);
    return b;
}

float orc_f32_from_f16(uint16_t b)
{
    _Float16 h;
    memcpy(&h, &b, 2);
    return (float)h;
}

/* ------------------------------------------------------------------ FWHT */

/* In-place Walsh-Hadamard transform of a 64-block, Sylvester (natural) order,
 * strides 1, 2, 4, 8, 16, 32 in that order, then scaled by 1/sqrt(64) = 1/8.
 * Every add/sub is one fp32 operation. */
void orc_fwht64_f32(float *v)
{
    for (int h = 1; h < 64; h <<= 1)
        for (int i = 0; i < 64; ++i)
            if ((i & h) == 0) {
                float a = v[i], b = v[i + h];
                v[i] = a + b;
                v[i + h] = a - b;
            }
    for (int i = 0; i < 64; ++i) v[i] = v[i] * 0.125f;
}

/* Same transform in fp64, on a strided vector (used on weight columns). */
void orc_fwht64_f64(double *v, long stride)
{
    for (int h = 1; h < 64; h <<= 1)
        for (int i = 0; i < 64; ++i)
            if ((i & h) == 0) {
                double a = v[i * stride], b = v[(i + h) * stride];
                v[i * stride] = a + b;
                v[(i + h) * stride] = a - b;
            }
    for (int i = 0; i < 64; ++i) v[i * stride] = v[i * stride] * 0.125;
}

/* ------------------------------------------------------------------ NVFP4 */

#define NVFP4_G_DIV 2688.0f   /* 6 (largest e2m1) * 448 (largest e4m3) */

float orc_nvfp4_tensor_scale(float amax) { return amax / NVFP4_G_DIV; }

/* Quantise n values (n % 16 == 0) that share the fp32 tensor scale g.
 * codes: n/2 bytes, element 2i in the low nibble; scales: n/16 bytes. */
void orc_nvfp4_quantize(const float *v, long n, float g, uint8_t *codes, uint8_t *scales)
{
    for (long b = 0; b < n / 16; ++b) {
        const float *blk = v + 16 * b;
        float bmax = 0.0f;
        for (int i = 0; i < 16; ++i) {
            float a = fabsf(blk[i]);
            if (a > bmax) bmax = a;
        }
        uint8_t sc = 0;
        if (g != 0.0f) {
            float t = bmax / 6.0f;
            sc = orc_e4m3_encode(t / g);
        }
        float d = (float)orc_e4m3_decode(sc) * g;
        scales[b] = sc;
        for (int i = 0; i < 16; i += 2) {
            uint8_t c0 = 0, c1 = 0;
            if (d != 0.0f) {
                c0 = orc_e2m1_encode(blk[i] / d);
                c1 = orc_e2m1_encode(blk[i + 1] / d);
            }
            codes[8 * b + i / 2] = (uint8_t)(c0 | (c1 << 4));
        }
    }
}

/* Dequantised value of element k of a canonical NVFP4 vector (without g). */
static double nvfp4_elem(const uint8_t *codes, const uint8_t *scales, long k)
{
    uint8_t byte = codes[k / 2];
    uint8_t c = (k & 1) ? (byte >> 4) : (byte & 15);
    return orc_e2m1_decode(c) * orc_e4m3_decode(scales[k / 16]);
}

/* ------------------------------------------------------------------ activations */

/* Transform one activation row.  Default order: xs = fp32(x) * inv_s (fp32 multiply),
 * then the block-64 FWHT when rotate != 0.  smooth_after != 0 (QuantWAMs Eq. (1),
 * A R S^-1): the FWHT of fp32(x) first, then the multiply by inv_s.  Output fp32 [K]. */
static int g_smooth_after = 0;           /* set by the entry points below for one call */

void orc_act_transform_row(const uint16_t *x_bf16, long K, const float *inv_s, int rotate, float *xt)
{
    int after = g_smooth_after && rotate;
    for (long k = 0; k < K; ++k) {
        float xv = orc_f32_from_bf16(x_bf16[k]);
        xt[k] = (inv_s && !after) ? xv * inv_s[k] : xv;
    }
    if (rotate)
        for (long b = 0; b < K / 64; ++b) orc_fwht64_f32(xt + 64 * b);
    if (inv_s && after)
        for (long k = 0; k < K; ++k) xt[k] = xt[k] * inv_s[k];
}

/* Select the transform order for the following calls (0: smooth, then rotate; 1: rotate,
 * then smooth).  Not thread-safe across concurrent callers; the Python wrapper holds a lock. */
void orc_set_smooth_after(int v) { g_smooth_after = v ? 1 : 0; }

/* Quantise M activation rows.
 *   per_tensor == 0: one g per row (dynamic per-token); g[m] written for each row.
 *   per_tensor == 1: one g over all rows from their amax; g[0] written.
 *   per_tensor == 2: one fixed g for all rows, read from g[0] (a calibrated scale: the
 *                    NVFP4 block scales stay dynamic, only the fp32 tensor scale is fixed).
 * x_omega (nullable when n_omega == 0): fp16 bits [M, n_omega] of the transformed
 * values at the outlier channels, which are then zeroed before quantisation.
 * xt_out (nullable): the transformed rows after the outlier split, fp32 [M, K]. */
int orc_quantize_act(const uint16_t *x_bf16, long M, long K, const float *inv_s, int rotate,
                     const int32_t *omega, int n_omega, int per_tensor,
                     uint8_t *codes, uint8_t *scales, float *g, uint16_t *x_omega, float *xt_out,
                     int n_threads)
{
    if (K % 16 || (rotate && K % 64)) return -1;
    float *xt = (float *)malloc(sizeof(float) * (size_t)M * (size_t)K);
    if (!xt) return -4;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
#pragma omp parallel for schedule(static)
    for (long m = 0; m < M; ++m) {
        float *row = xt + m * K;
        orc_act_transform_row(x_bf16 + m * K, K, inv_s, rotate, row);
        for (int j = 0; j < n_omega; ++j) {
            x_omega[m * n_omega + j] = orc_f16_from_f32(row[omega[j]]);
            row[omega[j]] = 0.0f;
        }
    }
    float gt = 0.0f;
    if (per_tensor == 2) {
        gt = g[0];
    } else if (per_tensor) {
        float amax = 0.0f;
        for (long i = 0; i < M * K; ++i) {
            float a = fabsf(xt[i]);
            if (a > amax) amax = a;
        }
        gt = orc_nvfp4_tensor_scale(amax);
        g[0] = gt;
    }
#pragma omp parallel for schedule(static)
    for (long m = 0; m < M; ++m) {
        const float *row = xt + m * K;
        float gm = gt;
        if (!per_tensor) {
            float amax = 0.0f;
            for (long k = 0; k < K; ++k) {
                float a = fabsf(row[k]);
                if (a > amax) amax = a;
            }
            gm = orc_nvfp4_tensor_scale(amax);
            g[m] = gm;
        }
        orc_nvfp4_quantize(row, K, gm, codes + m * (K / 2), scales + m * (K / 16));
    }
    if (xt_out) memcpy(xt_out, xt, sizeof(float) * (size_t)M * (size_t)K);
    free(xt);
    return 0;
}

/* ------------------------------------------------------------------ weights */

/* Fold smoothing, low-rank complement and rotation into W [K, N] (fp32, row-major).
 *   inv_s = 1/s (fp32 division) per channel; P = bf16(fp32(L1 * inv_s)) [K, r];
 *   Q = bf16(L2) [r, N];
 *   R[k][n] = s_k * (W[k][n] - sum_j P[k][j] Q[j][n])   (fp64, j ascending),
 *   R' = block-64 FWHT of R along k (fp64) when rotate, rounded once to fp32;
 *   rows Omega of R' go to the fp16 slice W_omega [n_omega, N] and are zeroed.
 * Outputs: Rp fp32 [K, N] (after zeroing), W_omega fp16 bits, P, Q bf16 bits,
 * W_omega_f32 (nullable) the unrounded slice. */
int orc_fold_weights(const float *W, long K, long N, const float *s,
                     const float *L1, const float *L2, int r,
                     const int32_t *omega, int n_omega, int rotate,
                     float *Rp, uint16_t *W_omega, float *W_omega_f32,
                     uint16_t *P, uint16_t *Q, int n_threads)
{
    if (K % 16 || (rotate && K % 64)) return -1;
    int after = g_smooth_after && rotate;
    if (!after) {
        for (long k = 0; k < K; ++k)
            for (int j = 0; j < r; ++j) {
                float l = L1[k * r + j];
                if (s) l = l * (1.0f / s[k]);
                P[k * r + j] = orc_bf16_from_f32(l);
            }
    } else {
        /* P = H S^-1 L1: column j of L1 times inv_s = fp32(1/s), the block FWHT in fp64,
         * one rounding to bf16 */
        double *col = (double *)malloc(sizeof(double) * (size_t)K);
        if (!col) return -4;
        for (int j = 0; j < r; ++j) {
            for (long k = 0; k < K; ++k)
                col[k] = (double)L1[k * r + j] * (s ? (double)(1.0f / s[k]) : 1.0);
            for (long b = 0; b < K / 64; ++b) orc_fwht64_f64(col + 64 * b, 1);
            for (long k = 0; k < K; ++k) P[k * r + j] = orc_bf16_from_f64(col[k]);
        }
        free(col);
    }
    for (int j = 0; j < r; ++j)
        for (long n = 0; n < N; ++n) Q[(long)j * N + n] = orc_bf16_from_f32(L2[(long)j * N + n]);

    double *R = (double *)malloc(sizeof(double) * (size_t)K * (size_t)N);
    if (!R) return -4;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
#pragma omp parallel for schedule(static)
    for (long k = 0; k < K; ++k)
        for (long n = 0; n < N; ++n) {
            double lr = 0.0;
            for (int j = 0; j < r; ++j)
                lr += (double)orc_f32_from_bf16(P[k * r + j]) * (double)orc_f32_from_bf16(Q[(long)j * N + n]);
            double t = (double)W[k * N + n] - lr;
            R[k * N + n] = (s && !after) ? (double)s[k] * t : t;
        }
    if (rotate) {
#pragma omp parallel for schedule(static)
        for (long n = 0; n < N; ++n)
            for (long b = 0; b < K / 64; ++b) orc_fwht64_f64(R + (64 * b) * N + n, N);
    }
    if (s && after) {
        /* R' = S H (W - P Q): the rotated rows scaled by s after the transform */
#pragma omp parallel for schedule(static)
        for (long k = 0; k < K; ++k)
            for (long n = 0; n < N; ++n) R[k * N + n] = (double)s[k] * R[k * N + n];
    }
    for (long i = 0; i < K * N; ++i) Rp[i] = (float)R[i];
    free(R);
    for (int j = 0; j < n_omega; ++j)
        for (long n = 0; n < N; ++n) {
            float v = Rp[(long)omega[j] * N + n];
            W_omega[(long)j * N + n] = orc_f16_from_f32(v);
            if (W_omega_f32) W_omega_f32[(long)j * N + n] = v;
            Rp[(long)omega[j] * N + n] = 0.0f;
        }
    return 0;
}

/* NVFP4-quantise the folded weight: one fp32 g over the whole tensor, each output
 * column n quantised along k.  codes [N, K/2], scales [N, K/16]. */
int orc_quantize_weights(const float *Rp, long K, long N, uint8_t *codes, uint8_t *scales, float *gW)
{
    if (K % 16) return -1;
    float amax = 0.0f;
    for (long i = 0; i < K * N; ++i) {
        float a = fabsf(Rp[i]);
        if (a > amax) amax = a;
    }
    float g = orc_nvfp4_tensor_scale(amax);
    *gW = g;
    float *col = (float *)malloc(sizeof(float) * (size_t)K);
    if (!col) return -4;
    for (long n = 0; n < N; ++n) {
        for (long k = 0; k < K; ++k) col[k] = Rp[k * N + n];
        orc_nvfp4_quantize(col, K, g, codes + n * (K / 2), scales + n * (K / 16));
    }
    free(col);
    return 0;
}

/* ------------------------------------------------------------------ forward */

/* Low-rank activation U[m][j] = bf16( sum_k x[m][k] * P[k][j] ) with the sum in fp64. */
void orc_lowrank_act(const uint16_t *x_bf16, long M, long K, const uint16_t *P, int r, uint16_t *U)
{
#pragma omp parallel for schedule(static)
    for (long m = 0; m < M; ++m)
        for (int j = 0; j < r; ++j) {
            double acc = 0.0;
            for (long k = 0; k < K; ++k)
                acc += (double)orc_f32_from_bf16(x_bf16[m * K + k]) * (double)orc_f32_from_bf16(P[k * r + j]);
            U[m * r + j] = orc_bf16_from_f64(acc);
        }
}

/* Quantised forward, fp64:
 *   y[m][n] = gA[m] * gW * sum_k deqA[m][k] deqW[n][k]      (4-bit main product)
 *           + sum_j U[m][j] Q[j][n]                          (16-bit low-rank branch)
 *           + sum_c xo[m][c] Wo[c][n]                        (fp16 outlier slice)
 *           + b[n]
 * gA has M entries (per_tensor_act == 0) or one.  Outputs y fp64 [M, N]. */
int orc_linear_forward(const uint8_t *codesA, const uint8_t *scalesA, const float *gA, int per_tensor_act,
                       long M, const uint8_t *codesW, const uint8_t *scalesW, float gW, long N, long K,
                       const uint16_t *U, const uint16_t *Q, int r,
                       const uint16_t *x_omega, const uint16_t *W_omega, int n_omega,
                       const float *bias, double *y, int n_threads)
{
    double *deqW = (double *)malloc(sizeof(double) * (size_t)N * (size_t)K);
    if (!deqW) return -4;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
#pragma omp parallel for schedule(static)
    for (long n = 0; n < N; ++n)
        for (long k = 0; k < K; ++k)
            deqW[n * K + k] = nvfp4_elem(codesW + n * (K / 2), scalesW + n * (K / 16), k);
#pragma omp parallel
    {
        double *a = (double *)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(static)
        for (long m = 0; m < M; ++m) {
            for (long k = 0; k < K; ++k)
                a[k] = nvfp4_elem(codesA + m * (K / 2), scalesA + m * (K / 16), k);
            double ga = (double)(per_tensor_act ? gA[0] : gA[m]);
            for (long n = 0; n < N; ++n) {
                const double *w = deqW + n * K;
                double acc = 0.0;
                for (long k = 0; k < K; ++k) acc += a[k] * w[k];
                double v = acc * ga * (double)gW;
                double lr = 0.0;
                for (int j = 0; j < r; ++j)
                    lr += (double)orc_f32_from_bf16(U[m * r + j]) * (double)orc_f32_from_bf16(Q[(long)j * N + n]);
                double ot = 0.0;
                for (int c = 0; c < n_omega; ++c)
                    ot += (double)orc_f32_from_f16(x_omega[m * n_omega + c]) *
                          (double)orc_f32_from_f16(W_omega[(long)c * N + n]);
                v += lr + ot;
                if (bias) v += (double)bias[n];
                y[m * N + n] = v;
            }
        }
        free(a);
    }
    free(deqW);
    return 0;
}

/* Unquantised forward through the same transforms (Proposition 1 check):
 *   y = xt Rp + xo Wo + U Q + b, with xt the transformed rows (outliers zeroed),
 *   Rp the folded weight (outlier rows zeroed), xo / Wo the outlier slices and
 *   U = x P.  xo, Wo are fp32 here and U is kept in fp64 (no 16-bit rounding),
 *   so the result equals x W + b up to fp32 rounding of xt and Rp. */
int orc_forward_noquant(const float *xt, const float *xo, long M, long K, long N,
                        const float *Rp, const float *Wo, int n_omega,
                        const uint16_t *x_bf16, const uint16_t *P, const uint16_t *Q, int r,
                        const float *bias, double *y)
{
#pragma omp parallel for schedule(static)
    for (long m = 0; m < M; ++m) {
        double *u = (double *)malloc(sizeof(double) * (size_t)(r > 0 ? r : 1));
        for (int j = 0; j < r; ++j) {
            double acc = 0.0;
            for (long k = 0; k < K; ++k)
                acc += (double)orc_f32_from_bf16(x_bf16[m * K + k]) * (double)orc_f32_from_bf16(P[k * r + j]);
            u[j] = acc;
        }
        for (long n = 0; n < N; ++n) {
            double acc = 0.0;
            for (long k = 0; k < K; ++k) acc += (double)xt[m * K + k] * (double)Rp[k * N + n];
            for (int c = 0; c < n_omega; ++c) acc += (double)xo[m * n_omega + c] * (double)Wo[(long)c * N + n];
            for (int j = 0; j < r; ++j) acc += u[j] * (double)orc_f32_from_bf16(Q[(long)j * N + n]);
            if (bias) acc += (double)bias[n];
            y[m * N + n] = acc;
        }
        free(u);
    }
    return 0;
}

/* ------------------------------------------------------------------ W8A8 (INT8) */
/* Selective 8-bit projections (FoldQuantVLA, Key Contribution 3: o_proj and down_proj kept at
 * W8A8) in the same transformed basis as the 4-bit layers (Key Contribution 1: one basis for
 * every consumer).  Symmetric int8: per row of the activations, per output column of the
 * weights, scale = amax / 127, q = round-half-even(v / scale) clamped to [-127, 127]; both
 * steps one IEEE fp32 operation.  The product is accumulated exactly in int64. */

static int8_t int8_rne(float v, float scale)
{
    if (scale == 0.0f) return 0;
    float t = v / scale;
    double r = nearbyint((double)t);          /* default rounding mode: nearest even */
    if (r > 127.0) r = 127.0;
    if (r < -127.0) r = -127.0;
    return (int8_t)r;
}

float orc_int8_scale(float amax) { return amax / 127.0f; }

/* x bf16 [M, K] -> q int8 [M, K], a fp32 [M] (smoothing and rotation as for W4A4). */
int orc_quantize_act_int8(const uint16_t *x_bf16, long M, long K, const float *inv_s, int rotate,
                          int8_t *q, float *a, int n_threads)
{
    if (K % 16 || (rotate && K % 64)) return -1;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    int rc = 0;
#pragma omp parallel
    {
        float *xt = (float *)malloc(sizeof(float) * (size_t)K);
        if (!xt) {
#pragma omp atomic write
            rc = -4;
        } else {
#pragma omp for schedule(static)
            for (long m = 0; m < M; ++m) {
                orc_act_transform_row(x_bf16 + m * K, K, inv_s, rotate, xt);
                float amax = 0.0f;
                for (long k = 0; k < K; ++k) {
                    float v = fabsf(xt[k]);
                    if (v > amax) amax = v;
                }
                float s = orc_int8_scale(amax);
                a[m] = s;
                for (long k = 0; k < K; ++k) q[m * K + k] = int8_rne(xt[k], s);
            }
            free(xt);
        }
    }
    return rc;
}

/* Folded weight Rp fp32 [K, N] -> q int8 [N, K] (K-major), w fp32 [N]. */
int orc_quantize_weights_int8(const float *Rp, long K, long N, int8_t *q, float *w)
{
    for (long n = 0; n < N; ++n) {
        float amax = 0.0f;
        for (long k = 0; k < K; ++k) {
            float v = fabsf(Rp[k * N + n]);
            if (v > amax) amax = v;
        }
        float s = orc_int8_scale(amax);
        w[n] = s;
        for (long k = 0; k < K; ++k) q[n * K + k] = int8_rne(Rp[k * N + n], s);
    }
    return 0;
}

/* y[m][n] = (sum_k qa[m][k] qw[n][k]) * a[m] * w[n] + b[n]; exact int64 sum, fp64 epilogue. */
int orc_linear_forward_w8a8(const int8_t *qa, const float *a, long M, const int8_t *qw, const float *w, long N,
                            long K, const float *bias, double *y, int n_threads)
{
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
#pragma omp parallel for schedule(static)
    for (long m = 0; m < M; ++m)
        for (long n = 0; n < N; ++n) {
            int64_t acc = 0;
            for (long k = 0; k < K; ++k) acc += (int64_t)qa[m * K + k] * (int64_t)qw[n * K + k];
            double v = (double)acc * (double)a[m] * (double)w[n];
            if (bias) v += (double)bias[n];
            y[m * N + n] = v;
        }
    return 0;
}

/* ------------------------------------------------------------------ W8A8 (FP8) */
/* Upgraded layers in FP8 W8A8 (QuantWAMs sec. 4.2 "Backend": "upgraded layers use FP8 W8A8
 * kernels").  Reading: e4m3 values (4 exponent bits, bias 7, 3 mantissa bits, finite maximum
 * 448, sign bit 7) with one fp32 scale per token and per output column, scale = amax / 448,
 * q = e4m3_rne_satfinite(RN(v / scale)) -- the quotient one IEEE fp32 division, then one
 * rounding to e4m3; a zero scale gives zero codes.  Same transformed basis as the other
 * layers.  The product of two e4m3 values is exact in fp64, so the fp64 sum is exact up to
 * the fp64 accumulation. */

/* Signed e4m3 code of v (sign bit 7 | the unsigned code of |v|). */
uint8_t orc_e4m3s_encode(float v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0;
    return (uint8_t)(sign | orc_e4m3_encode(fabsf(v)));
}

double orc_e4m3s_decode(uint8_t c)
{
    double m = orc_e4m3_decode((uint8_t)(c & 0x7F));
    return (c & 0x80) ? -m : m;
}

float orc_fp8_scale(float amax) { return amax / 448.0f; }

static uint8_t fp8_code(float v, float scale)
{
    if (scale == 0.0f) return 0;
    return orc_e4m3s_encode(v / scale);
}

/* x bf16 [M, K] -> q e4m3 [M, K], a fp32 [M] (smoothing and rotation as for W4A4).  The
 * channels in omega (n_omega of them, nullable when 0) go to x_omega fp16 [M, n_omega] and are
 * zeroed before the row maximum, as in the 4-bit quantiser. */
int orc_quantize_act_fp8(const uint16_t *x_bf16, long M, long K, const float *inv_s, int rotate,
                         const int32_t *omega, int n_omega, uint16_t *x_omega,
                         uint8_t *q, float *a, int n_threads)
{
    if (K % 16 || (rotate && K % 64)) return -1;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    int rc = 0;
#pragma omp parallel
    {
        float *xt = (float *)malloc(sizeof(float) * (size_t)K);
        if (!xt) {
#pragma omp atomic write
            rc = -4;
        } else {
#pragma omp for schedule(static)
            for (long m = 0; m < M; ++m) {
                orc_act_transform_row(x_bf16 + m * K, K, inv_s, rotate, xt);
                for (int j = 0; j < n_omega; ++j) {
                    x_omega[m * n_omega + j] = orc_f16_from_f32(xt[omega[j]]);
                    xt[omega[j]] = 0.0f;
                }
                float amax = 0.0f;
                for (long k = 0; k < K; ++k) {
                    float v = fabsf(xt[k]);
                    if (v > amax) amax = v;
                }
                float s = orc_fp8_scale(amax);
                a[m] = s;
                for (long k = 0; k < K; ++k) q[m * K + k] = fp8_code(xt[k], s);
            }
            free(xt);
        }
    }
    return rc;
}

/* Folded weight Rp fp32 [K, N] -> q e4m3 [N, K] (K-major), w fp32 [N]. */
int orc_quantize_weights_fp8(const float *Rp, long K, long N, uint8_t *q, float *w)
{
    for (long n = 0; n < N; ++n) {
        float amax = 0.0f;
        for (long k = 0; k < K; ++k) {
            float v = fabsf(Rp[k * N + n]);
            if (v > amax) amax = v;
        }
        float s = orc_fp8_scale(amax);
        w[n] = s;
        for (long k = 0; k < K; ++k) q[n * K + k] = fp8_code(Rp[k * N + n], s);
    }
    return 0;
}

/* y[m][n] = (sum_k dec(qa[m][k]) dec(qw[n][k])) * a[m] * w[n] + b[n], fp64. */
int orc_linear_forward_fp8(const uint8_t *qa, const float *a, long M, const uint8_t *qw, const float *w, long N,
                           long K, const float *bias, double *y, int n_threads)
{
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
#pragma omp parallel for schedule(static)
    for (long m = 0; m < M; ++m)
        for (long n = 0; n < N; ++n) {
            double acc = 0.0;
            for (long k = 0; k < K; ++k) acc += orc_e4m3s_decode(qa[m * K + k]) * orc_e4m3s_decode(qw[n * K + k]);
            double v = acc * (double)a[m] * (double)w[n];
            if (bias) v += (double)bias[n];
            y[m * N + n] = v;
        }
    return 0;
}

/* ------------------------------------------------------------------ projected complement */
/* Q-WAM abstract (Action-Subspace Protection): a 16-bit low-rank branch protects the action
 * subspace and the complementary weights AND activations are quantised.  Reading: with the branch
 * factors L1 L2 = U_r S_r V_r^T (top-r SVD of the smoothed weight), the activation's complement is
 * x_c = xs - (xs U_r) U_r^T, in the rotated basis xt_c = xt - u Vt with u = the branch's bf16
 * down-projection x P (P = diag(1/s) L1, so xs U_r = u S_r^-1) and
 *   Vt[j][k] = bf16( (H L1[:, j])[k] / ||L1[:, j]||^2 )      (S_r^-2 L1^T H, fp64, one rounding).
 * Each element: acc = xt[k]; acc = fma(-u[j], Vt[j][k], acc) for j = 0 .. r-1 in that order (fp32).
 * The weight complement R = (I - U_r U_r^T) W_s already gives xc R = xs R, so the folding identity
 * holds unchanged; only the quantiser's input changes (then the kept-channel split and NVFP4). */

/* Vt [r, K] bf16 bits from L1 [K, r] (fp32), rotate as in the fold. */
int orc_projection_basis(const float *L1, long K, int r, int rotate, uint16_t *Vt)
{
    double *col = (double *)malloc(sizeof(double) * (size_t)K);
    if (!col) return -4;
    for (int j = 0; j < r; ++j) {
        double nrm = 0.0;
        for (long k = 0; k < K; ++k) {
            col[k] = (double)L1[k * r + j];
            nrm += col[k] * col[k];
        }
        if (rotate)
            for (long b = 0; b < K / 64; ++b) orc_fwht64_f64(col + 64 * b, 1);
        for (long k = 0; k < K; ++k) Vt[(long)j * K + k] = orc_bf16_from_f64(nrm > 0.0 ? col[k] / nrm : 0.0);
    }
    free(col);
    return 0;
}

/* xt_c = xt - u Vt for M rows: xt fp32 [M, K] in place, u bf16 [M, r], Vt bf16 [r, K]. */
void orc_project_complement(float *xt, long M, long K, const uint16_t *u, const uint16_t *Vt, int r)
{
#pragma omp parallel for schedule(static)
    for (long m = 0; m < M; ++m)
        for (long k = 0; k < K; ++k) {
            float acc = xt[m * K + k];
            for (int j = 0; j < r; ++j)
                acc = fmaf(-orc_f32_from_bf16(u[m * r + j]), orc_f32_from_bf16(Vt[(long)j * K + k]), acc);
            xt[m * K + k] = acc;
        }
}

/* The activation quantiser on the projected complement: transform, subtract u Vt, kept-channel
 * split, per-row NVFP4 (as orc_quantize_act with per_tensor = 0). */
int orc_quantize_act_projected(const uint16_t *x_bf16, long M, long K, const float *inv_s, int rotate,
                               const int32_t *omega, int n_omega, const uint16_t *u, const uint16_t *Vt, int r,
                               uint8_t *codes, uint8_t *scales, float *g, uint16_t *x_omega, float *xt_out)
{
    if (K % 16 || (rotate && K % 64)) return -1;
    float *xt = (float *)malloc(sizeof(float) * (size_t)M * (size_t)K);
    if (!xt) return -4;
    for (long m = 0; m < M; ++m) orc_act_transform_row(x_bf16 + m * K, K, inv_s, rotate, xt + m * K);
    orc_project_complement(xt, M, K, u, Vt, r);
#pragma omp parallel for schedule(static)
    for (long m = 0; m < M; ++m) {
        float *row = xt + m * K;
        for (int j = 0; j < n_omega; ++j) {
            x_omega[m * n_omega + j] = orc_f16_from_f32(row[omega[j]]);
            row[omega[j]] = 0.0f;
        }
        float amax = 0.0f;
        for (long k = 0; k < K; ++k) {
            float a = fabsf(row[k]);
            if (a > amax) amax = a;
        }
        float gm = orc_nvfp4_tensor_scale(amax);
        g[m] = gm;
        orc_nvfp4_quantize(row, K, gm, codes + m * (K / 2), scales + m * (K / 16));
    }
    if (xt_out) memcpy(xt_out, xt, sizeof(float) * (size_t)M * (size_t)K);
    free(xt);
    return 0;
}

/* ------------------------------------------------------------------ W4A8 */
/* A8-protected steps (QuantWAMs sec. 4.2 and sec. 5: one of ten Fast-WAM action steps, two of twenty
 * and six of fifty LingBot-VA steps run their activations at 8 bits).  Reading: the 4-bit layer keeps
 * its NVFP4 weights, low-rank branch and fp16 kept channels; its activations are quantised to e4m3
 * per token (orc_quantize_act_fp8, with the kept-channel split).  fp64:
 *   y[m][n] = a[m] gW sum_k dec8(qa[m][k]) deqW[n][k] + sum_j U Q + sum_c x_O W_O + b. */
int orc_linear_forward_w4a8(const uint8_t *qa, const float *a, long M, const uint8_t *codesW,
                            const uint8_t *scalesW, float gW, long N, long K, const uint16_t *U, const uint16_t *Q,
                            int r, const uint16_t *x_omega, const uint16_t *W_omega, int n_omega,
                            const float *bias, double *y, int n_threads)
{
    double *deqW = (double *)malloc(sizeof(double) * (size_t)N * (size_t)K);
    if (!deqW) return -4;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
#pragma omp parallel for schedule(static)
    for (long n = 0; n < N; ++n)
        for (long k = 0; k < K; ++k)
            deqW[n * K + k] = nvfp4_elem(codesW + n * (K / 2), scalesW + n * (K / 16), k);
#pragma omp parallel for schedule(static)
    for (long m = 0; m < M; ++m)
        for (long n = 0; n < N; ++n) {
            double acc = 0.0;
            for (long k = 0; k < K; ++k) acc += orc_e4m3s_decode(qa[m * K + k]) * deqW[n * K + k];
            double v = acc * (double)a[m] * (double)gW;
            for (int j = 0; j < r; ++j)
                v += (double)orc_f32_from_bf16(U[m * r + j]) * (double)orc_f32_from_bf16(Q[(long)j * N + n]);
            for (int c = 0; c < n_omega; ++c)
                v += (double)orc_f32_from_f16(x_omega[m * n_omega + c]) * (double)orc_f32_from_f16(W_omega[(long)c * N + n]);
            if (bias) v += (double)bias[n];
            y[m * N + n] = v;
        }
    free(deqW);
    return 0;
}

/* ------------------------------------------------------------------ outlier calibration */
/* QuantWAMs sec. 3.1 Eq. (1)-(3): the pooled squared energy of each channel of the transformed
 * activation, z(c) = mean_t xt[t, c]^2 (one context, pi = 1), and the Top-K channels by z, which
 * stay in 16-bit.  xt is the quantiser's own transform of each row (fp32, the same steps and
 * order as orc_act_transform_row); each square and the sum over rows are taken in fp64, rows in
 * ascending order.  Ties in z go to the lower channel index; the selected set is returned in
 * ascending channel order. */
int orc_pooled_energy(const uint16_t *x_bf16, long M, long K, const float *inv_s, int rotate, double *z)
{
    float *xt = (float *)malloc(sizeof(float) * (size_t)K);
    if (!xt) return -4;
    for (long k = 0; k < K; ++k) z[k] = 0.0;
    for (long m = 0; m < M; ++m) {
        orc_act_transform_row(x_bf16 + m * K, K, inv_s, rotate, xt);
        for (long k = 0; k < K; ++k) z[k] += (double)xt[k] * (double)xt[k];
    }
    for (long k = 0; k < K; ++k) z[k] = M > 0 ? z[k] / (double)M : 0.0;
    free(xt);
    return 0;
}

/* The n channels with the largest z (ties: lower index first), ascending. */
int orc_topk_channels(const double *z, long K, int n, int32_t *omega)
{
    if (n < 0 || n > K) return -1;
    char *taken = (char *)calloc((size_t)K, 1);
    if (!taken) return -4;
    for (int j = 0; j < n; ++j) {
        long best = -1;
        for (long k = 0; k < K; ++k)
            if (!taken[k] && (best < 0 || z[k] > z[best])) best = k;   /* strict: the lower index wins ties */
        taken[best] = 1;
    }
    int j = 0;
    for (long k = 0; k < K; ++k)
        if (taken[k]) omega[j++] = (int32_t)k;
    free(taken);
    return 0;
}

/* ------------------------------------------------------------------ Conv3d */
/* NVFP4 execution of the video VAE's 3x3x3 convolutions (LatentQuant, Abstract).  Plainest
 * reading: the input tensor is quantised once, per voxel along channels (16-channel blocks)
 * with one fp32 scale for the whole tensor (an implicit-GEMM row mixes 27 voxels, so a
 * per-voxel scale would not factor out); no smoothing, rotation, low-rank or kept channels.
 * The weight [C_out, C_in, 3, 3, 3] is laid out as K = (kd, kh, kw, c_in) and quantised per
 * output channel along K with one fp32 scale per tensor.  The convolution itself is the
 * direct definition with zero padding 1, on the dequantised values, accumulated in fp64. */

/* xq: codes [V, C/2] and scales [V, C/16] of the voxels (V = D H W, voxel v = (d H + h) W + w),
 * gx the tensor scale; wq: codes [N, 27 C / 2], scales [N, 27 C / 16], gw.
 * Computes y[n][v] for the listed voxels (y is [n_vox, N]). */
int orc_conv3d_forward(const uint8_t *xcodes, const uint8_t *xscales, float gx, long C, long D, long H, long W,
                       const uint8_t *wcodes, const uint8_t *wscales, float gw, long N,
                       const int64_t *vox, long n_vox, double *y, int n_threads)
{
    const long K = 27 * C;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
#pragma omp parallel for schedule(static)
    for (long i = 0; i < n_vox; ++i) {
        const long v = vox[i];
        const long d = v / (H * W), h = (v / W) % H, w = v % W;
        for (long n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int kd = 0; kd < 3; ++kd)
                for (int kh = 0; kh < 3; ++kh)
                    for (int kw = 0; kw < 3; ++kw) {
                        const long di = d + kd - 1, hi = h + kh - 1, wi = w + kw - 1;
                        if (di < 0 || di >= D || hi < 0 || hi >= H || wi < 0 || wi >= W) continue;
                        const long vin = (di * H + hi) * W + wi;
                        const long k0 = ((kd * 3 + kh) * 3 + kw) * C;
                        for (long c = 0; c < C; ++c)
                            acc += nvfp4_elem(xcodes + vin * (C / 2), xscales + vin * (C / 16), c) *
                                   nvfp4_elem(wcodes + n * (K / 2), wscales + n * (K / 16), k0 + c);
                    }
            y[i * N + n] = acc * (double)gx * (double)gw;
        }
    }
    return 0;
}
