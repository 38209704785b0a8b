// quant_math.cuh -- NVFP4 element coding shared by the activation quantisers.
#pragma once
#include "ptx.cuh"

namespace wq {

// Codes of v[i] / d for 8 values, bit-identical to e2m1_rn_satfinite(RN(v / d)).  One IEEE
// reciprocal r = RN(1/d) per block; q = RN(v r) is within 2^-22 (relative) of RN(v / d), so
// when q (1 - 2^-21) and q (1 + 2^-21) convert to the same codes, RN(v / d) -- which lies
// between them, and the e2m1 rounding is monotone in |x| -- converts to those codes too.
// A pair whose bracket straddles a rounding boundary is recomputed with the exact division.
// r = RN(1 / d), computed once per 16-element block by the caller.
__device__ __forceinline__ uint32_t e2m1_codes8_r(const float* v, float d, float r) {
    const bool r_ok = r < 3.0e38f;                       // d is not subnormal-small
    uint32_t word = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t code;
        if (r_ok) {
            const float a = __fmul_rn(v[2 * q], r), b = __fmul_rn(v[2 * q + 1], r);
            const uint32_t lo = cvt_e2m1x2(__fmul_rn(a, 0.99999952316284180f), __fmul_rn(b, 0.99999952316284180f));
            const uint32_t hi = cvt_e2m1x2(__fmul_rn(a, 1.00000047683715820f), __fmul_rn(b, 1.00000047683715820f));
            code = lo;
            if (lo != hi) code = cvt_e2m1x2(__fdiv_rn(v[2 * q], d), __fdiv_rn(v[2 * q + 1], d));
        } else {
            code = cvt_e2m1x2(__fdiv_rn(v[2 * q], d), __fdiv_rn(v[2 * q + 1], d));
        }
        word |= code << (8 * q);
    }
    return word;
}

__device__ __forceinline__ uint32_t e2m1_codes8(const float* v, float d) { return e2m1_codes8_r(v, d, __frcp_rn(d)); }

// Symmetric 8-bit values of v[i] / a for 8 values, identical to clamp(rint(RN(v / a)), +-127)
// (round half to even).  Same bracket argument as above with the integer rounding points;
// |v| <= 127 a keeps every quotient finite.
// r = RN(1 / a), computed once per row by the caller.
__device__ __forceinline__ void int8_values8_r(const float* v, float a, float r, float (&q)[8]) {
    const bool r_ok = r < 3.0e38f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        float t;
        if (r_ok) {
            const float x = __fmul_rn(v[e], r);
            const float lo = rintf(__fmul_rn(x, 0.99999952316284180f));
            const float hi = rintf(__fmul_rn(x, 1.00000047683715820f));
            t = lo == hi ? lo : rintf(__fdiv_rn(v[e], a));
        } else {
            t = rintf(__fdiv_rn(v[e], a));
        }
        q[e] = fminf(fmaxf(t, -127.0f), 127.0f);
    }
}

}  // namespace wq
