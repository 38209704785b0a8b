// wq_quant.cu -- fused activation transform + NVFP4 quantiser (one pass over x).
//
// Per activation row (FoldQuantVLA, Key Contribution 2: channel scaling, block Hadamard
// via the FWHT with beta = 64, dynamic per-token quantisation; QuantWAMs sec. 3.1 Eq. (1):
// the quantiser sees x R S^-1 and the Top-K channels of that basis stay in FP16):
//   xs   = fp32(x) * inv_s                       (one fp32 multiply)
//   xt   = FWHT64(xs) per 64-block               (strides 1,2,4 in registers; 8,16,32 across
//                                                 lanes by shuffles; then * 1/8)
//   x_O  = fp16(xt[O]); xt[O] = 0                (outlier split)
//   g    = amax(|xt|) / 2688                     (fp32 tensor scale of the row)
//   sc_b = e4m3((bmax_b / 6) / g), d_b = dec(sc_b) * g, code = e2m1(xt / d_b)
//   U    = bf16(x P)                             (16-bit low-rank down-projection, Q-WAM ASP)
// Every rounding step is an explicit _rn intrinsic so no multiply-add contraction can
// change a bit.  Thread layout: TPR threads per row, each owning CPT chunks of 8
// consecutive channels (one 128-bit load each); chunk c of a row is owned by thread
// c % TPR, so the 8 chunks of a 64-block sit in 8 consecutive lanes.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int kThreads = 256;
constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ void bf16x8_to_f32(const uint4& raw, float (&f)[8]) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

template <int TPR, int CPT, int R>
__global__ void __launch_bounds__(kThreads) quantize_act_kernel(const QuantArgs a) {
    constexpr int RPC = kThreads / TPR;   // rows per CTA
    constexpr int WPR = TPR / 32;         // warps per row
    __shared__ float s_red[RPC][WPR];
    __shared__ float s_u[R > 0 ? RPC : 1][WPR][R > 0 ? R : 1];

    const int tid = threadIdx.x, lane = tid & 31;
    const int rloc = tid / TPR, t = tid % TPR, wrow = t / 32;
    const int row = blockIdx.x * RPC + rloc;
    const bool row_ok = row < a.M;
    const int K = a.K, nch = K / 8;
    const uint4* xrow = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) +
                                                       static_cast<size_t>(row_ok ? row : 0) * K);

    // ---- one 128-bit load per chunk, all issued up front
    uint4 raw[CPT];
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int c = t + i * TPR;
        raw[i] = (row_ok && c < nch) ? __ldg(xrow + c) : make_uint4(0, 0, 0, 0);
    }

    // ---- smoothing
    float v[CPT][8];
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        bf16x8_to_f32(raw[i], v[i]);
        const int c = t + i * TPR;
        if (a.inv_s != nullptr && c < nch) {
            const float4* sp = reinterpret_cast<const float4*>(a.inv_s + 8 * c);
            const float4 s0 = __ldg(sp), s1 = __ldg(sp + 1);
            const float s[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) v[i][e] = __fmul_rn(v[i][e], s[e]);
        }
    }

    // ---- block-64 FWHT, stride order 1, 2, 4 (in registers) then 8, 16, 32 (lanes)
    if (a.rotate) {
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
#pragma unroll
            for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if ((e & h) == 0) {
                        const float p = v[i][e], q = v[i][e + h];
                        v[i][e] = __fadd_rn(p, q);
                        v[i][e + h] = __fsub_rn(p, q);
                    }
            }
#pragma unroll
            for (int m = 1; m < 8; m <<= 1) {
                const bool upper = (lane & m) != 0;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float o = __shfl_xor_sync(kFull, v[i][e], m);
                    v[i][e] = upper ? __fsub_rn(o, v[i][e]) : __fadd_rn(v[i][e], o);
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) v[i][e] = __fmul_rn(v[i][e], 0.125f);
        }
    }

    // ---- outlier split (rotated basis)
    if (a.n_out > 0 && row_ok) {
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const int c = t + i * TPR;
            if (c < nch) {
                const uint4 pw = __ldg(reinterpret_cast<const uint4*>(a.omega_pos + 8 * c));
                const uint32_t w[4] = {pw.x, pw.y, pw.z, pw.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int pos = static_cast<int16_t>((w[e / 2] >> (16 * (e & 1))) & 0xFFFFu);
                    if (pos >= 0) {
                        a.xo[static_cast<size_t>(row) * a.n_out + pos] =
                            __half_as_ushort(__float2half_rn(v[i][e]));
                        v[i][e] = 0.0f;
                    }
                }
            }
        }
    }

    // ---- row amax -> fp32 tensor scale
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < CPT; ++i)
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(v[i][e]));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, off));
    if constexpr (WPR > 1) {
        if (lane == 0) s_red[rloc][wrow] = amax;
        __syncthreads();
        amax = s_red[rloc][0];
#pragma unroll
        for (int w = 1; w < WPR; ++w) amax = fmaxf(amax, s_red[rloc][w]);
    }
    const float g = __fdiv_rn(amax, 2688.0f);
    if (t == 0 && row_ok) a.g[row] = g;

    // ---- block scales and e2m1 codes
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int c = t + i * TPR;
        float cm = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) cm = fmaxf(cm, fabsf(v[i][e]));
        const float bm = fmaxf(cm, __shfl_xor_sync(kFull, cm, 1));
        uint32_t sc = 0;
        if (g != 0.0f) sc = cvt_e4m3(__fdiv_rn(__fdiv_rn(bm, 6.0f), g));
        const float d = __fmul_rn(dec_e4m3(sc), g);
        uint32_t word = 0;
        if (d != 0.0f) {
#pragma unroll
            for (int p = 0; p < 4; ++p)
                word |= cvt_e2m1x2(__fdiv_rn(v[i][2 * p], d), __fdiv_rn(v[i][2 * p + 1], d)) << (8 * p);
        }
        const bool ok = row_ok && c < nch;
        if (ok)
            *reinterpret_cast<uint32_t*>(a.codes + static_cast<size_t>(row) * (K / 2) + 4 * c) = word;
        const uint32_t s1 = __shfl_down_sync(kFull, sc, 2);
        const uint32_t s2 = __shfl_down_sync(kFull, sc, 4);
        const uint32_t s3 = __shfl_down_sync(kFull, sc, 6);
        if (ok && (lane & 7) == 0) {
            const uint32_t w4 = sc | (s1 << 8) | (s2 << 16) | (s3 << 24);
            size_t off;
            if (a.sf_layout == WQ_SCALE_LAYOUT_MMA)
                off = (static_cast<size_t>(row / kBlockM) * (K / 64) + c / 8) * kSfAtom +
                      (row % 32) * 16 + ((row % kBlockM) / 32) * 4;
            else
                off = static_cast<size_t>(row) * (K / 16) + (c / 8) * 4;
            *reinterpret_cast<uint32_t*>(a.sf + off) = w4;
        }
    }

    // ---- 16-bit low-rank down-projection U = bf16(x P)
    if constexpr (R > 0) {
        float acc[R];
#pragma unroll
        for (int j = 0; j < R; ++j) acc[j] = 0.0f;
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const int c = t + i * TPR;
            if (c < nch) {
                float xf[8];
                bf16x8_to_f32(raw[i], xf);
                const uint4* prow = reinterpret_cast<const uint4*>(a.P + static_cast<size_t>(8 * c) * R);
#pragma unroll
                for (int e = 0; e < 8; ++e)
#pragma unroll
                    for (int jj = 0; jj < R / 8; ++jj) {
                        const uint4 pv = __ldg(prow + e * (R / 8) + jj);
                        float pf[8];
                        bf16x8_to_f32(pv, pf);
#pragma unroll
                        for (int q = 0; q < 8; ++q) acc[8 * jj + q] = fmaf(xf[e], pf[q], acc[8 * jj + q]);
                    }
            }
        }
#pragma unroll
        for (int j = 0; j < R; ++j)
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc[j] += __shfl_xor_sync(kFull, acc[j], off);
        if (lane == 0)
#pragma unroll
            for (int j = 0; j < R; ++j) s_u[rloc][wrow][j] = acc[j];
        __syncthreads();
        if (row_ok)
            for (int j = t; j < R; j += TPR) {
                float s = 0.0f;
#pragma unroll
                for (int w = 0; w < WPR; ++w) s += s_u[rloc][w][j];
                a.u[static_cast<size_t>(row) * R + j] = __bfloat16_as_ushort(__float2bfloat16_rn(s));
            }
    }
}

template <int TPR, int CPT>
cudaError_t launch_r(const QuantArgs& a, cudaStream_t st) {
    const int rows_per_cta = kThreads / TPR;
    const dim3 grid((a.M + rows_per_cta - 1) / rows_per_cta);
    switch (a.r) {
        case 0: quantize_act_kernel<TPR, CPT, 0><<<grid, kThreads, 0, st>>>(a); break;
        case 16: quantize_act_kernel<TPR, CPT, 16><<<grid, kThreads, 0, st>>>(a); break;
        case 32: quantize_act_kernel<TPR, CPT, 32><<<grid, kThreads, 0, st>>>(a); break;
        case 64: quantize_act_kernel<TPR, CPT, 64><<<grid, kThreads, 0, st>>>(a); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <int TPR>
cudaError_t launch_cpt(const QuantArgs& a, int cpt, cudaStream_t st) {
    switch (cpt) {
        case 1: return launch_r<TPR, 1>(a, st);
        case 2: return launch_r<TPR, 2>(a, st);
        case 4: return launch_r<TPR, 4>(a, st);
        case 6: return launch_r<TPR, 6>(a, st);
        case 8: return launch_r<TPR, 8>(a, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_quantize_act(const QuantArgs& a, cudaStream_t st) {
    if (a.M <= 0) return cudaSuccess;
    const int nch = a.K / 8;
    static const int kTpr[4] = {32, 64, 128, 256};
    static const int kCpt[5] = {1, 2, 4, 6, 8};
    for (int ti = 0; ti < 4; ++ti) {
        const int need = (nch + kTpr[ti] - 1) / kTpr[ti];
        if (need > 8) continue;
        int cpt = 8;
        for (int ci = 0; ci < 5; ++ci)
            if (kCpt[ci] >= need) { cpt = kCpt[ci]; break; }
        switch (kTpr[ti]) {
            case 32: return launch_cpt<32>(a, cpt, st);
            case 64: return launch_cpt<64>(a, cpt, st);
            case 128: return launch_cpt<128>(a, cpt, st);
            default: return launch_cpt<256>(a, cpt, st);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace wq
