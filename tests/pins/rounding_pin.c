/*
 * rounding_pin.c -- independent check of the oracle's e2m1 / e4m3 encoders.
 *
 * The oracle encodes by a nearest-point search over the decoded grid.  This file
 * restates the same roundings the IEEE-754 way instead: a value is divided by the
 * quantum (ulp) of its binade, rounded half-to-even with nearbyint(), multiplied
 * back and saturated to the largest finite value; the result is then mapped to
 * its bit pattern from the format's field layout.  Both formats:
 *   e2m1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; largest 6.
 *   e4m3: 4 exponent (bias 7), 3 mantissa bits, no infinities; largest 448.
 * Every fp32 bit pattern (NaNs excluded) is compared, spread over OpenMP threads.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

typedef uint8_t (*enc_fn)(float);

static uint8_t e2m1_ieee(float v)
{
    int neg = signbit(v) ? 1 : 0;
    double a = fabs((double)v);
    double q = a < 2.0 ? 0.5 : (a < 4.0 ? 1.0 : 2.0);
    double r = (a >= 8.0) ? 6.0 : nearbyint(a / q) * q;
    if (r > 6.0) r = 6.0;
    int code;
    if (r < 1.0) code = (int)(r * 2.0);                 /* subnormal: 0 or 0.5 */
    else {
        int e;
        double m = frexp(r, &e);                        /* r = m 2^e, m in [0.5,1) */
        int exp_field = e;                              /* unbiased exponent e-1, bias 1 */
        int man = (int)(m * 4.0) - 2;                   /* 1 mantissa bit */
        code = (exp_field << 1) | man;
    }
    return (uint8_t)(code | (neg << 3));
}

static uint8_t e4m3_ieee(float v)
{
    double a = (double)v;
    if (!(a > 0.0)) return 0;
    if (a >= 448.0) return 0x7E;
    int e;
    (void)frexp(a, &e);
    int ub = e - 1;                                     /* a in [2^ub, 2^(ub+1)) */
    double q = ub < -6 ? ldexp(1.0, -9) : ldexp(1.0, ub - 3);
    double r = nearbyint(a / q) * q;
    if (r > 448.0) r = 448.0;
    if (r == 0.0) return 0;
    if (r < ldexp(1.0, -6)) return (uint8_t)(r / ldexp(1.0, -9));
    (void)frexp(r, &e);
    ub = e - 1;
    int man = (int)(r / ldexp(1.0, ub - 3)) - 8;
    return (uint8_t)(((ub + 7) << 3) | man);
}

/* Returns the number of mismatching fp32 patterns; first mismatch in *first. */
long pin_e2m1_all(enc_fn f, uint32_t *first)
{
    long bad = 0;
    uint32_t fb = 0;
#pragma omp parallel for reduction(+:bad) schedule(static)
    for (long i = 0; i <= 0xFFFFFFFFL; ++i) {
        uint32_t u = (uint32_t)i;
        if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x7FFFFFu)) continue;
        float v;
        memcpy(&v, &u, 4);
        if (f(v) != e2m1_ieee(v)) {
            bad++;
#pragma omp critical
            { if (!fb) fb = u; }
        }
    }
    *first = fb;
    return bad;
}

long pin_e4m3_all(enc_fn f, uint32_t *first)
{
    long bad = 0;
    uint32_t fb = 0;
#pragma omp parallel for reduction(+:bad) schedule(static)
    for (long i = 0; i <= 0x7F800000L; ++i) {           /* +0 .. +inf */
        uint32_t u = (uint32_t)i;
        float v;
        memcpy(&v, &u, 4);
        if (f(v) != e4m3_ieee(v)) {
            bad++;
#pragma omp critical
            { if (!fb) fb = u; }
        }
    }
    *first = fb;
    return bad;
}

uint8_t pin_e2m1_one(float v) { return e2m1_ieee(v); }
uint8_t pin_e4m3_one(float v) { return e4m3_ieee(v); }
