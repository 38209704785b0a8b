// quant_block.cuh -- the per-block steps of the activation quantiser, shared by the
// stand-alone quantiser (wq_quant.cu) and the fused small-batch forward (wq_fused.cu).
//
// A warp handles one 64-channel block of 16 rows: lane l owns row l % 16 and half l / 16 (32
// channels held as 16 packed pairs (channel k, channel k + 16)).  See wq_quant.cu for the
// operation and the pages it follows.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "quant_math.cuh"

namespace wq {
namespace {

constexpr unsigned kQFullMask = 0xFFFFFFFFu;

// ------------------------------------------------------------------ shared-memory helpers
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ float4 ld_shared_v4f(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ float2 ld_shared_v2f(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void st_shared_v2f(uint32_t addr, float a, float b) {
    asm volatile("st.shared.v2.f32 [%0], {%1, %2};" :: "r"(addr), "f"(a), "f"(b) : "memory");
}
__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
    asm volatile("st.shared.f32 [%0], %1;" :: "r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// ------------------------------------------------------------------ packed fp32 pairs
// A lane's 32 channels of a block are held as 16 pairs P[k] = (channel k, channel k + 16) of
// its half, so the FWHT butterflies at strides 1..8 and the elementwise multiplies run as
// packed two-lane fp32 instructions; each lane is rounded to nearest on its own, exactly as
// the scalar operation would be.
typedef unsigned long long f2;
__device__ __forceinline__ f2 pk2(float lo, float hi) {
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float lo2(f2 x) {
    float a;
    asm("{\n\t.reg .f32 t;\n\tmov.b64 {%0, t}, %1;\n\t}" : "=f"(a) : "l"(x));
    return a;
}
__device__ __forceinline__ float hi2(f2 x) {
    float b;
    asm("{\n\t.reg .f32 t;\n\tmov.b64 {t, %0}, %1;\n\t}" : "=f"(b) : "l"(x));
    return b;
}
__device__ __forceinline__ f2 add2(f2 a, f2 b) {
    f2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2 sub2(f2 a, f2 b) {
    f2 r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
    f2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {   // RN(a b + c) per lane
    f2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// ------------------------------------------------------------------ per-block steps
// Row r, half `half` of a raw 16 x 64 bf16 box (128-byte swizzle: 16-byte chunk c of row r at
// c ^ (r % 8)) -> 16 pairs of smoothed and rotated values.  invs: shared address of the
// block's 64 inv_s values stored pair-wise (per half: s_k, s_k+16 for k = 0..15), or 0.
// FWHT in the pages' order: strides 1, 2, 4, 8 between pairs, 16 inside a pair, 32 with the
// partner lane (lane ^ 16 holds the other half of the row: a + b there, a - b here, as one
// fused multiply-add with an exact +-1 product), then the exact 1/8 normalisation.
// rotate: bit 0 = the block FWHT; bit 1 = smooth after the rotation (QuantWAMs sec. 3.1
// Eq. (1), A R S^-1) instead of before it (FoldQuantVLA, Key Contribution 2).
__device__ __forceinline__ void load_transform(uint32_t box, int r, int half, uint32_t invs, int rotate,
                                               f2 (&P)[16]) {
    const bool smooth_after = (rotate & 3) == 3;
    uint32_t w[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t c = static_cast<uint32_t>(4 * half + j);
        const uint4 q = ld_shared_v4(box + static_cast<uint32_t>(r) * 128u + ((c ^ (static_cast<uint32_t>(r) & 7u)) << 4));
        w[j][0] = q.x; w[j][1] = q.y; w[j][2] = q.z; w[j][3] = q.w;
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const uint32_t a = w[k / 8][(k % 8) / 2], b = w[2 + k / 8][(k % 8) / 2];
        P[k] = (k & 1) ? pk2(__uint_as_float(a & 0xFFFF0000u), __uint_as_float(b & 0xFFFF0000u))
                       : pk2(__uint_as_float(a << 16), __uint_as_float(b << 16));
    }
    if (invs != 0u && !smooth_after) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 sv = ld_shared_v4f(invs + 128u * half + 16u * j);
            P[2 * j] = mul2(P[2 * j], pk2(sv.x, sv.y));
            P[2 * j + 1] = mul2(P[2 * j + 1], pk2(sv.z, sv.w));
        }
    }
    if (rotate & 1) {
#pragma unroll
        for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
            for (int k = 0; k < 16; ++k)
                if ((k & h) == 0) {
                    const f2 a = P[k], b = P[k + h];
                    P[k] = add2(a, b);
                    P[k + h] = sub2(a, b);
                }
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const float a = lo2(P[k]), b = hi2(P[k]);
            P[k] = pk2(__fadd_rn(a, b), __fsub_rn(a, b));
        }
        const float sgn = half ? -1.0f : 1.0f;
        const f2 sg = pk2(sgn, sgn);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const f2 o = pk2(__shfl_xor_sync(kQFullMask, lo2(P[k]), 16), __shfl_xor_sync(kQFullMask, hi2(P[k]), 16));
            P[k] = fma2(P[k], sg, o);
        }
        const f2 c8 = pk2(0.125f, 0.125f);
#pragma unroll
        for (int k = 0; k < 16; ++k) P[k] = mul2(P[k], c8);
        if (invs != 0u && smooth_after) {
            // the same pair-ordered inv_s: rotation keeps channel positions
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float4 sv = ld_shared_v4f(invs + 128u * half + 16u * j);
                P[2 * j] = mul2(P[2 * j], pk2(sv.x, sv.y));
                P[2 * j + 1] = mul2(P[2 * j + 1], pk2(sv.z, sv.w));
            }
        }
    }
}

// Zero the kept channels of this half (bit e of `mine`: channel e): a kept channel becomes +0
// and every other value keeps all its bits, the sign of a zero included.
__device__ __forceinline__ void apply_keep(f2 (&P)[16], uint32_t mine) {
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const uint32_t a = ((mine >> k) & 1u) - 1u;          // channel k: 0 if kept, else all ones
        const uint32_t b = ((mine >> (k + 16)) & 1u) - 1u;   // channel k + 16
        P[k] &= (static_cast<f2>(b) << 32) | a;
    }
}

// e4m3(RN(RN(bm / 6) / g)), the block scale.  t = RN(RN(bm c6) rg) with c6 = RN(1/6) and
// rg = RN(1/g) is within 6 ulp-units of 2^-24 (relative) of the two-division value, so when
// t (1 - 2^-20) and t (1 + 2^-20) convert to the same code, that value (which lies between
// them; the conversion is monotone) converts to it too.  Otherwise, and when a product could
// leave the normal range, the two divisions are done.
template <bool kOut = false>
__device__ __forceinline__ uint32_t scale_code(float bm, float g, float rg) {
    if (g == 0.0f || bm == 0.0f) return 0u;
    const float u = __fmul_rn(bm, 0.16666667163372040f);
    if (rg < 3.0e38f && u >= 1.0e-36f) {
        const float t = __fmul_rn(u, rg);
        const uint32_t lo = cvt_e4m3(__fmul_rn(t, 0.99999904632568359f));
        const uint32_t hi = cvt_e4m3(__fmul_rn(t, 1.00000095367431641f));
        if (lo == hi) return lo;
    }
    return e4m3_div1<kOut>(bm, g);
}

// Maxima of |x| over the half's two 16-element blocks (channels 0..15: the pairs' first lanes).
__device__ __forceinline__ void absmax_pairs(const f2 (&P)[16], float& ma, float& mb) {
    ma = 0.0f;
    mb = 0.0f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        ma = fmaxf(ma, fabsf(lo2(P[k])));
        mb = fmaxf(mb, fabsf(hi2(P[k])));
    }
}

// Codes of channels (k, k+1) of both 16-blocks of the half (pairs P0 = P[k], P1 = P[k+1]), by
// the reciprocal-and-bracket argument of e2m1_codes8_r, two blocks per packed multiply.
template <bool kOut = false>
__device__ __forceinline__ void codes_2x2(f2 P0, f2 P1, f2 rr, float da, float db, uint32_t& ca, uint32_t& cb) {
    const f2 mlo = pk2(0.99999952316284180f, 0.99999952316284180f);
    const f2 mhi = pk2(1.00000047683715820f, 1.00000047683715820f);
    const f2 q0 = mul2(P0, rr), q1 = mul2(P1, rr);
    const f2 l0 = mul2(q0, mlo), l1 = mul2(q1, mlo), h0 = mul2(q0, mhi), h1 = mul2(q1, mhi);
    const uint32_t alo = cvt_e2m1x2(lo2(l0), lo2(l1)), ahi = cvt_e2m1x2(lo2(h0), lo2(h1));
    const uint32_t blo = cvt_e2m1x2(hi2(l0), hi2(l1)), bhi = cvt_e2m1x2(hi2(h0), hi2(h1));
    ca = alo;
    cb = blo;
    if (alo != ahi) ca = e2m1_div2<kOut>(lo2(P0), lo2(P1), da);
    if (blo != bhi) cb = e2m1_div2<kOut>(hi2(P0), hi2(P1), db);
}

// The block's share of U = x P: A = the raw 16 x 64 box, every n-tile of P.  Each
// (block, n-tile) is accumulated on the tensor cores from zero and added to the warp's
// partial (shared memory, mma fragment order, 512 B per n-tile) with an fp32 add, so the
// tensor-core accumulation depth stays at 64 whatever K is.
__device__ __forceinline__ void u_frags(uint32_t box, int lane, uint32_t (&a)[4][4]) {
    const uint32_t arow = static_cast<uint32_t>((lane & 7) + 8 * ((lane >> 3) & 1));
#pragma unroll
    for (int f = 0; f < 4; ++f) {
        const uint32_t chunk = static_cast<uint32_t>(2 * f + (lane >> 4));
        ldmatrix_x4(box + arow * 128u + ((chunk ^ (arow & 7u)) << 4), a[f][0], a[f][1], a[f][2], a[f][3]);
    }
    __syncwarp();                          // the box is read before a partial may land on it
}
// Up to four n-tiles of one block at once: the tensor-core chains of different n-tiles are
// independent, so they are issued interleaved (k-step outer, n-tile inner) in one basic block;
// each chain still runs its four k-steps in order from zero.  Then the warp's partial of each
// n-tile is written (first block) or read, added to and written back.
template <int NG>
__device__ __forceinline__ void u_group(const uint32_t (&a)[4][4], const uint4 (&q)[NG][2], uint32_t ua0, bool first) {
    float t[NG][4];
#pragma unroll
    for (int g = 0; g < NG; ++g) t[g][0] = t[g][1] = t[g][2] = t[g][3] = 0.0f;
#pragma unroll
    for (int f = 0; f < 4; ++f)
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            const uint4& qq = q[g][f >> 1];
            mma_bf16_16816(t[g], a[f][0], a[f][1], a[f][2], a[f][3], (f & 1) ? qq.z : qq.x, (f & 1) ? qq.w : qq.y);
        }
    if (first) {
#pragma unroll
        for (int g = 0; g < NG; ++g) st_shared_v4f(ua0 + static_cast<uint32_t>(g) * 512u, t[g][0], t[g][1], t[g][2], t[g][3]);
    } else {
        float4 o[NG];
#pragma unroll
        for (int g = 0; g < NG; ++g) o[g] = ld_shared_v4f(ua0 + static_cast<uint32_t>(g) * 512u);
#pragma unroll
        for (int g = 0; g < NG; ++g)
            st_shared_v4f(ua0 + static_cast<uint32_t>(g) * 512u, __fadd_rn(o[g].x, t[g][0]), __fadd_rn(o[g].y, t[g][1]),
                          __fadd_rn(o[g].z, t[g][2]), __fadd_rn(o[g].w, t[g][3]));
    }
}
// P fragments from global memory (block kb of the whole table).
template <int NT>
__device__ __forceinline__ void u_step(uint32_t box, int lane, int kb, const uint32_t* pfrag, uint32_t upart, bool first) {
    constexpr int NG = NT < 4 ? NT : 4;
    uint32_t a[4][4];
    u_frags(box, lane, a);
#pragma unroll
    for (int n0 = 0; n0 < NT; n0 += NG) {
        uint4 q[NG][2];
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            const uint4* pb = reinterpret_cast<const uint4*>(pfrag + (static_cast<size_t>(kb * NT + n0 + g) * 32 + lane) * 8);
            q[g][0] = __ldg(pb);
            q[g][1] = __ldg(pb + 1);
        }
        u_group<NG>(a, q, upart + (static_cast<uint32_t>(n0) * 32u + lane) * 16u, first);
    }
}
// P fragments of one block staged in shared memory at `pf` (NT x 32 lanes x 32 bytes).
template <int NT>
__device__ __forceinline__ void u_step_smem(uint32_t box, int lane, uint32_t pf, uint32_t upart, bool first) {
    constexpr int NG = NT < 4 ? NT : 4;
    uint32_t a[4][4];
    u_frags(box, lane, a);
#pragma unroll
    for (int n0 = 0; n0 < NT; n0 += NG) {
        uint4 q[NG][2];
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            const uint32_t pb = pf + (static_cast<uint32_t>(n0 + g) * 32u + lane) * 32u;
            q[g][0] = ld_shared_v4(pb);
            q[g][1] = ld_shared_v4(pb + 16u);
        }
        u_group<NG>(a, q, upart + (static_cast<uint32_t>(n0) * 32u + lane) * 16u, first);
    }
}

// Codes of this lane's half row (32 channels in pair order: channels 0..15 the pairs' first
// lanes, 16..31 their second lanes) and the e4m3 scales of its two 16-blocks with maxima bma,
// bmb: w[0], w[1] hold channels 0..7, 8..15 and w[2], w[3] channels 16..23, 24..31 (element 2i
// in the low nibble of byte i); gsc is the row's tensor scale and rg = RN(1 / gsc).
template <bool kOut = false>
__device__ __forceinline__ void nvfp4_half_codes(const f2 (&P)[16], float bma, float bmb, float gsc, float rg,
                                                 uint32_t (&w)[4], uint32_t& sa, uint32_t& sb) {
    sa = scale_code<kOut>(bma, gsc, rg);
    sb = scale_code<kOut>(bmb, gsc, rg);
    const float da = __fmul_rn(dec_e4m3(sa), gsc), db = __fmul_rn(dec_e4m3(sb), gsc);
    const float ra = __frcp_rn(da), rb = __frcp_rn(db);
    w[0] = w[1] = w[2] = w[3] = 0u;
    uint32_t bad = (ra < 3.0e38f && rb < 3.0e38f) ? 0u : 1u;
    if (!bad) {
        // both blocks have a non-zero, non-tiny scale: every code from the bracket of e2m1_codes8_r,
        // two blocks per packed multiply; a straddled bracket anywhere sends the half to the exact
        // quotients below (one branch per half instead of one per pair)
        const f2 rr = pk2(ra, rb);
        const f2 mlo = pk2(0.99999952316284180f, 0.99999952316284180f);
        const f2 mhi = pk2(1.00000047683715820f, 1.00000047683715820f);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            uint32_t lb[4], hb[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int k = 8 * j + 2 * e;
                const f2 q0 = mul2(P[k], rr), q1 = mul2(P[k + 1], rr);
                const f2 l0 = mul2(q0, mlo), l1 = mul2(q1, mlo), h0 = mul2(q0, mhi), h1 = mul2(q1, mhi);
                const uint32_t alo = cvt_e2m1x2(lo2(l0), lo2(l1)), ahi = cvt_e2m1x2(lo2(h0), lo2(h1));
                const uint32_t blo = cvt_e2m1x2(hi2(l0), hi2(l1)), bhi = cvt_e2m1x2(hi2(h0), hi2(h1));
                bad |= (alo ^ ahi) | (blo ^ bhi);
                lb[e] = alo;
                hb[e] = blo;
            }
            w[j] = __byte_perm(__byte_perm(lb[0], lb[1], 0x0040), __byte_perm(lb[2], lb[3], 0x0040), 0x5410);
            w[2 + j] = __byte_perm(__byte_perm(hb[0], hb[1], 0x0040), __byte_perm(hb[2], hb[3], 0x0040), 0x5410);
        }
    }
    if (bad) {
        float va[16], vb[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            va[k] = lo2(P[k]);
            vb[k] = hi2(P[k]);
        }
        if (da != 0.0f) {
            w[0] = e2m1_codes8_r<kOut>(va, da, ra);
            w[1] = e2m1_codes8_r<kOut>(va + 8, da, ra);
        }
        if (db != 0.0f) {
            w[2] = e2m1_codes8_r<kOut>(vb, db, rb);
            w[3] = e2m1_codes8_r<kOut>(vb + 8, db, rb);
        }
    }
}

// U entry of fragment index idx = (nt 32 + lane) 4 + e: row gq + 8 (e / 2), column
// 8 nt + 2 cq + e % 2, with gq = lane / 4, cq = lane % 4.
__device__ __forceinline__ void frag_pos(int idx, int& rr, int& cc) {
    const int nt = idx / 128, ln = (idx / 4) % 32, e = idx % 4;
    rr = (ln >> 2) + 8 * (e >> 1);
    cc = 8 * nt + 2 * (ln & 3) + (e & 1);
}

}  // namespace
}  // namespace wq
