// quant_math.cuh -- NVFP4 element coding shared by the activation quantisers.
#pragma once
#include "ptx.cuh"

namespace wq {

// The exact quotients, out of line: they are reached only when a bracket below straddles a
// rounding point (or the reciprocal is unusable), so the common path carries no division code
// and fetches fewer instructions.
static __device__ __noinline__ uint32_t e2m1_pair_div(float a, float b, float d) {
    return cvt_e2m1x2(__fdiv_rn(a, d), __fdiv_rn(b, d));
}
static __device__ __noinline__ float int8_div(float v, float a) { return rintf(__fdiv_rn(v, a)); }
static __device__ __noinline__ uint32_t e4m3_div(float bm, float g) { return cvt_e4m3(__fdiv_rn(__fdiv_rn(bm, 6.0f), g)); }

// kOut selects the out-of-line forms (code that runs once per CTA, where instruction fetch
// dominates) or the inline ones (persistent loops, where a call would cost register spills).
template <bool kOut>
__device__ __forceinline__ uint32_t e2m1_div2(float a, float b, float d) {
    if constexpr (kOut) return e2m1_pair_div(a, b, d);
    else return cvt_e2m1x2(__fdiv_rn(a, d), __fdiv_rn(b, d));
}
template <bool kOut>
__device__ __forceinline__ float int8_div1(float v, float a) {
    if constexpr (kOut) return int8_div(v, a);
    else return rintf(__fdiv_rn(v, a));
}
template <bool kOut>
__device__ __forceinline__ uint32_t e4m3_div1(float bm, float g) {
    if constexpr (kOut) return e4m3_div(bm, g);
    else return cvt_e4m3(__fdiv_rn(__fdiv_rn(bm, 6.0f), g));
}

// Codes of v[i] / d for 8 values, bit-identical to e2m1_rn_satfinite(RN(v / d)).  One IEEE
// reciprocal r = RN(1/d) per block; q = RN(v r) is within 2^-22 (relative) of RN(v / d), so
// when q (1 - 2^-21) and q (1 + 2^-21) convert to the same codes, RN(v / d) -- which lies
// between them, and the e2m1 rounding is monotone in |x| -- converts to those codes too.
// A pair whose bracket straddles a rounding boundary is recomputed with the exact division.
// r = RN(1 / d), computed once per 16-element block by the caller.
template <bool kOut = false>
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
            if (lo != hi) code = e2m1_div2<kOut>(v[2 * q], v[2 * q + 1], d);
        } else {
            code = e2m1_div2<kOut>(v[2 * q], v[2 * q + 1], d);
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
template <bool kOut = false>
__device__ __forceinline__ void int8_values8_r(const float* v, float a, float r, float (&q)[8]) {
    const bool r_ok = r < 3.0e38f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        float t;
        if (r_ok) {
            const float x = __fmul_rn(v[e], r);
            const float lo = rintf(__fmul_rn(x, 0.99999952316284180f));
            const float hi = rintf(__fmul_rn(x, 1.00000047683715820f));
            t = lo;
            if (lo != hi) t = int8_div1<kOut>(v[e], a);
        } else {
            t = int8_div1<kOut>(v[e], a);
        }
        q[e] = fminf(fmaxf(t, -127.0f), 127.0f);
    }
}

}  // namespace wq
