// wq_conv.cu -- the video VAE's 3x3x3 convolution (padding 1, batch B) as an NVFP4 implicit GEMM
// (LatentQuant, Abstract: NVFP4 execution of the Wan VAE).
//
// Reading taken: the input is quantised once, per voxel along channels (16-channel blocks, e4m3
// scales) with one fp32 scale for the whole [B, C, D, H, W] tensor -- a GEMM row gathers 27 voxels, so a
// per-voxel scale would not factor out of the accumulator; no smoothing or rotation.  The
// weight [C_out, C_in, 3, 3, 3] is the GEMM operand [N = C_out, K = (kd, kh, kw, c_in)].
//
//   conv_amax_kernel   per-CTA maxima of |x| (the tensor scale's pre-pass)
//   conv_quant_kernel  64-voxel x C tiles of the NCDHW input, transposed through shared
//                      memory, quantised per voxel -> voxel-major codes [V, C/2], scales [V, C/16]
//   conv_gemm_kernel   persistent tcgen05 GEMM: M = voxels, N = C_out, K = 27 C_in.  A work item
//                      is 128 voxels by up to three 128-column tiles (three TMEM accumulators),
//                      so every gathered A stage feeds the MMAs of all of them.  A stage is 128
//                      channels of one tap.  Warps 2-5 gather the A rows (one output voxel
//                      each) with cp.async -- zero-filled where the tap falls in the padding --
//                      into the 64-byte-swizzled K-major layout and the scale atoms; warp 0
//                      brings the weight tiles by TMA; warp 1 issues tcgen05.cp + mxf4nvf4 MMAs;
//                      warps 6-9 scale the TMEM accumulators and store bf16 NCDHW.
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "quant_math.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int kAmaxThreads = 256;
constexpr int kVox = 64;                      // voxels per quantiser tile
constexpr int kConvThreads = 320;
constexpr uint32_t kATile = 128 * 64;         // 128 rows x 64 bytes (128 fp4 channels)
constexpr int kGroup = 3;                     // column tiles per work item (TMEM accumulators)
// stage: A tile, kGroup weight tiles, 2 A scale atoms, 2 scale atoms per weight tile
constexpr uint32_t kCStage = (1 + kGroup) * kATile + 2 * (1 + kGroup) * kSfAtom;
constexpr uint32_t kSfbOff = (1 + kGroup) * kATile + 2 * kSfAtom;
constexpr uint32_t kSfCols = 8 * (1 + kGroup);   // TMEM scale columns per stage
constexpr int kMaxStagesTmem = static_cast<int>((512 - 128 * kGroup) / kSfCols);
constexpr int kGatherDepth = 2;               // stages of cp.async in flight per gather thread
constexpr uint32_t kConvMaxSmem = 232448;

__global__ void __launch_bounds__(kAmaxThreads) conv_amax_kernel(const uint4* __restrict__ x, size_t n8,
                                                                 float* __restrict__ partial) {
    __shared__ float red[kAmaxThreads / 32];
    float m = 0.0f;
    for (size_t i = static_cast<size_t>(blockIdx.x) * kAmaxThreads + threadIdx.x; i < n8;
         i += static_cast<size_t>(gridDim.x) * kAmaxThreads) {
        const uint4 v = __ldg(x + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            m = fmaxf(m, fabsf(__uint_as_float(w[j] << 16)));
            m = fmaxf(m, fabsf(__uint_as_float(w[j] & 0xFFFF0000u)));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float r = red[0];
        for (int i = 1; i < kAmaxThreads / 32; ++i) r = fmaxf(r, red[i]);
        partial[blockIdx.x] = r;
    }
}

// Voxels are numbered over the batch: v = b V1 + (d H + h) W + w, V1 = D H W (a multiple of 8, so
// an 8-voxel group never straddles two samples).
__global__ void __launch_bounds__(256) conv_quant_kernel(const uint16_t* __restrict__ x, int C, int V, int V1,
                                                         const float* __restrict__ partial, int n_partial,
                                                         uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                                                         float* __restrict__ g_out) {
    extern __shared__ uint8_t sm[];
    uint16_t* tile = reinterpret_cast<uint16_t*>(sm);                         // [C][kVox]
    uint8_t* oc = sm + static_cast<size_t>(C) * kVox * 2;                     // [kVox][C/2]
    uint8_t* os = oc + static_cast<size_t>(kVox) * (C / 2);                   // [kVox][C/16]
    __shared__ float red[8];

    float amax = 0.0f;
    for (int i = threadIdx.x; i < n_partial; i += 256) amax = fmaxf(amax, partial[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = amax;
    __syncthreads();
    amax = red[0];
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
    const float g = __fdiv_rn(amax, 2688.0f);
    if (blockIdx.x == 0 && threadIdx.x == 0) *g_out = g;

    const int v0 = blockIdx.x * kVox;
    const int nv = min(kVox, V - v0);
    for (int i = threadIdx.x; i < C * (kVox / 8); i += 256) {
        const int c = i / (kVox / 8), q = i % (kVox / 8);
        uint4 val = make_uint4(0, 0, 0, 0);
        if (8 * q < nv) {
            const int gv = v0 + 8 * q, b = gv / V1, lv = gv % V1;
            val = __ldg(reinterpret_cast<const uint4*>(x + (static_cast<size_t>(b) * C + c) * V1 + lv));
        }
        *reinterpret_cast<uint4*>(tile + c * kVox + 8 * q) = val;
    }
    __syncthreads();
    for (int t = threadIdx.x; t < kVox * (C / 16); t += 256) {
        const int v = t % kVox, blk = t / kVox;
        float e[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) e[j] = __uint_as_float(static_cast<uint32_t>(tile[(blk * 16 + j) * kVox + v]) << 16);
        float bm = 0.0f;
#pragma unroll
        for (int j = 0; j < 16; ++j) bm = fmaxf(bm, fabsf(e[j]));
        uint32_t sc = 0;
        if (g != 0.0f) sc = cvt_e4m3(__fdiv_rn(__fdiv_rn(bm, 6.0f), g));
        const float d = __fmul_rn(dec_e4m3(sc), g);
        const float (&lo)[8] = *reinterpret_cast<const float(*)[8]>(e);
        const float (&hi)[8] = *reinterpret_cast<const float(*)[8]>(e + 8);
        const uint32_t w0 = d != 0.0f ? e2m1_codes8(lo, d) : 0u;
        const uint32_t w1 = d != 0.0f ? e2m1_codes8(hi, d) : 0u;
        *reinterpret_cast<uint2*>(oc + v * (C / 2) + blk * 8) = make_uint2(w0, w1);
        os[v * (C / 16) + blk] = static_cast<uint8_t>(sc);
    }
    __syncthreads();
    const size_t cbytes = static_cast<size_t>(nv) * (C / 2), sbytes = static_cast<size_t>(nv) * (C / 16);
    for (size_t i = threadIdx.x; i < cbytes / 16; i += 256)
        reinterpret_cast<uint4*>(codes + static_cast<size_t>(v0) * (C / 2))[i] = reinterpret_cast<const uint4*>(oc)[i];
    for (size_t i = threadIdx.x; i < sbytes / 4; i += 256)
        reinterpret_cast<uint32_t*>(scales + static_cast<size_t>(v0) * (C / 16))[i] = reinterpret_cast<const uint32_t*>(os)[i];
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                 :: "r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;"
                 :: "r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

struct ConvParams {
    int C, D, H, W, V, V1, N, K, stages;     // V = B V1 voxels over the batch, V1 = D H W
    const uint8_t* xcodes;
    const uint8_t* xscales;
    const float* gx;
    float gw;
    const uint8_t* sfb;
    __nv_bfloat16* y;
    int* err;
};

__global__ void __launch_bounds__(kConvThreads, 1)
conv_gemm_kernel(const __grid_constant__ CUtensorMap tmB, const ConvParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw_addr);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int S = p.stages;
    const uint32_t off_bar = static_cast<uint32_t>(S) * kCStage;
    const uint32_t bar_full = base + off_bar;
    const uint32_t bar_empty = bar_full + 8u * S;
    const uint32_t bar_tfull = bar_empty + 8u * S;
    const uint32_t bar_tempty = bar_tfull + 8u;
    const uint32_t bar_final = bar_tempty + 8u;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base_ptr + off_bar + 8u * (2 * S + 3));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int n_tiles = (p.N + 127) / 128;
    const int n_groups = (n_tiles + kGroup - 1) / kGroup;
    const int items = ((p.V + 127) / 128) * n_groups;
    const int cpt = p.C / 128;                      // stages per tap
    const int nst = 27 * cpt;                       // stages per item
    const int num_kb = p.K / 64;
    // work item -> row block and its column tiles [nb0, nb0 + ng)
    auto item_rc = [&](int item, int& mb, int& nb0, int& ng) {
        mb = item / n_groups;
        nb0 = (item % n_groups) * kGroup;
        ng = min(kGroup, n_tiles - nb0);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_full + 8u * s, 1 + 128);  // TMA arrival + one per gather thread
            mbar_init(bar_empty + 8u * s, 1);
        }
        mbar_init(bar_tfull, 1);
        mbar_init(bar_tempty, 4);
        mbar_init(bar_final, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------------ weights by TMA
        if (lane == 0) {
            tma_prefetch_desc(&tmB);
            int stage = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < items && ok; item += gridDim.x) {
                int mb, nb0, ng;
                item_rc(item, mb, nb0, ng);
                for (int s = 0; s < nst; ++s) {
                    if (!mbar_wait(bar_empty + 8u * stage, ph ^ 1u, abort_flag, p.err, 21)) { ok = false; break; }
                    const uint32_t fb = bar_full + 8u * stage;
                    const uint32_t st = base + static_cast<uint32_t>(stage) * kCStage;
                    mbar_arrive_expect_tx(fb, static_cast<uint32_t>(ng) * (kATile + 2 * kSfAtom));
                    for (int g = 0; g < ng; ++g) {
                        tma_load_2d(st + static_cast<uint32_t>(1 + g) * kATile, &tmB, s * 64, (nb0 + g) * 128, fb);
                        bulk_load(st + kSfbOff + static_cast<uint32_t>(2 * g) * kSfAtom,
                                  p.sfb + (static_cast<size_t>(nb0 + g) * num_kb + 2 * s) * kSfAtom, 2 * kSfAtom, fb);
                    }
                    if (++stage == S) { stage = 0; ph ^= 1u; }
                }
            }
        }
    } else if (warp >= 2 && warp <= 5) {
        // ------------------------------------------------------------ A gather (one voxel per thread)
        const int r = threadIdx.x - 64;
        int stage = 0;
        uint32_t ph = 0;
        int pend[kGatherDepth + 1];
        int npend = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < items && ok; item += gridDim.x) {
            int mb, nb0, ng;
            item_rc(item, mb, nb0, ng);
            const int m = mb * 128 + r;
            const bool m_ok = m < p.V;
            const int bsm = m / p.V1, lm = m % p.V1;                 // sample, voxel in the sample
            const int d = lm / (p.H * p.W), h = (lm / p.W) % p.H, w = lm % p.W;
            for (int s = 0; s < nst; ++s) {
                const int tap = s / cpt, cc = s % cpt;
                const int kd = tap / 9, kh = (tap / 3) % 3, kw = tap % 3;
                const int di = d + kd - 1, hi = h + kh - 1, wi = w + kw - 1;
                const bool valid = m_ok && di >= 0 && di < p.D && hi >= 0 && hi < p.H && wi >= 0 && wi < p.W;
                const size_t vin = valid ? static_cast<size_t>(bsm) * p.V1 + (static_cast<size_t>(di) * p.H + hi) * p.W + wi : 0;
                if (!mbar_wait(bar_empty + 8u * stage, ph ^ 1u, abort_flag, p.err, 22)) { ok = false; break; }
                const uint32_t st = base + static_cast<uint32_t>(stage) * kCStage;
                const uint8_t* src = p.xcodes + vin * (p.C / 2) + cc * 64;
                const uint32_t sw = (static_cast<uint32_t>(r) >> 1) & 3u;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    cp_async16(st + static_cast<uint32_t>(r) * 64u + ((static_cast<uint32_t>(j) ^ sw) << 4), src + 16 * j,
                               valid ? 16u : 0u);
                const uint8_t* ssrc = p.xscales + vin * (p.C / 16) + cc * 8;
                const uint32_t sfa = st + (1 + kGroup) * kATile + static_cast<uint32_t>(r % 32) * 16u +
                                     static_cast<uint32_t>(r / 32) * 4u;
                cp_async4(sfa, ssrc, valid ? 4u : 0u);
                cp_async4(sfa + kSfAtom, ssrc + 4, valid ? 4u : 0u);
                cp_async_commit();
                pend[npend++] = stage;
                if (npend > kGatherDepth) {
                    cp_async_wait<kGatherDepth>();
                    fence_proxy_async_smem();
                    mbar_arrive(bar_full + 8u * pend[0]);
                    for (int q = 0; q < kGatherDepth; ++q) pend[q] = pend[q + 1];
                    --npend;
                }
                if (++stage == S) { stage = 0; ph ^= 1u; }
            }
        }
        cp_async_wait<0>();
        fence_proxy_async_smem();
        for (int q = 0; q < npend; ++q) mbar_arrive(bar_full + 8u * pend[q]);
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
            int stage = 0, tl = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < items && ok; item += gridDim.x, ++tl) {
                int mb, nb0, ng;
                item_rc(item, mb, nb0, ng);
                // one set of accumulators: the epilogue has drained the previous item
                if (!mbar_wait(bar_tempty, (static_cast<uint32_t>(tl) & 1u) ^ 1u, abort_flag, p.err, 23)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int s = 0; s < nst; ++s) {
                    if (!mbar_wait(bar_full + 8u * stage, ph, abort_flag, p.err, 24)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t st = base + static_cast<uint32_t>(stage) * kCStage;
                    // scale slot of the stage: A at +4 kb, weight tile g at +8 + 8 g + 4 kb
                    const uint32_t sf_t = tmem + 128u * kGroup + kSfCols * static_cast<uint32_t>(stage);
                    for (int kb = 0; kb < 2; ++kb) {
                        tmem_cp_32x128b_x4(sf_t + 4u * kb, smem_desc(st + (1 + kGroup) * kATile + kSfAtom * kb, 0, 128, 0));
                        for (int g = 0; g < ng; ++g)
                            tmem_cp_32x128b_x4(sf_t + 8u + 8u * g + 4u * kb,
                                               smem_desc(st + kSfbOff + kSfAtom * (2 * g + kb), 0, 128, 0));
                    }
                    const uint64_t ad = smem_desc(st, 16, 512, 4);            // 64-byte swizzle, 8-row groups
                    for (int kb = 0; kb < 2; ++kb)
                        for (int g = 0; g < ng; ++g) {
                            const uint64_t bd = smem_desc(st + static_cast<uint32_t>(1 + g) * kATile, 16, 512, 4);
                            mma_nvf4(tmem + 128u * g, ad + 2u * kb, bd + 2u * kb, idesc, sf_t + 4u * kb,
                                     sf_t + 8u + 8u * g + 4u * kb, (s | kb) != 0 ? 1u : 0u);
                        }
                    tc_commit(bar_empty + 8u * stage);
                    if (++stage == S) { stage = 0; ph ^= 1u; }
                }
                if (!ok) break;
                tc_commit(bar_tfull);
            }
            tc_commit(bar_final);
            mbar_wait(bar_final, 0, abort_flag, p.err, 25);
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 6-9)
        const int q = warp & 3;
        const uint32_t t_lane = static_cast<uint32_t>(q * 32) << 16;
        const float alpha = __fmul_rn(__ldg(p.gx), p.gw);
        int tl = 0;
        for (int item = blockIdx.x; item < items; item += gridDim.x, ++tl) {
            int mb, nb0, ng;
            item_rc(item, mb, nb0, ng);
            if (!mbar_wait(bar_tfull, static_cast<uint32_t>(tl) & 1u, abort_flag, p.err, 26)) break;
            tc_fence_after();
            const int m = mb * 128 + q * 32 + lane;
            for (int g = 0; g < ng; ++g)
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t acc[32];
                    tmem_ld_32x32b_x32(tmem + 128u * g + 32u * ch + t_lane, acc);
                    tmem_wait_ld();
                    if (m < p.V) {
                        const size_t ybase = static_cast<size_t>(m / p.V1) * p.N * p.V1 + m % p.V1;
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int n = (nb0 + g) * 128 + ch * 32 + i;
                            if (n < p.N)
                                p.y[ybase + static_cast<size_t>(n) * p.V1] = __float2bfloat16_rn(alpha * __uint_as_float(acc[i]));
                        }
                    }
                }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_tempty);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

size_t conv_workspace_bytes(int C, int V, int num_sms) {
    auto al = [](size_t v) { return (v + 1023) / 1024 * 1024; };
    return al(static_cast<size_t>(2 * num_sms + 1) * 4) + al(static_cast<size_t>(V) * C / 2) +
           al(static_cast<size_t>(V) * C / 16);
}

cudaError_t launch_conv_quant(const ConvArgs& a, cudaStream_t st) {
    const size_t n8 = static_cast<size_t>(a.C) * a.V / 8;
    const int grid_a = 2 * a.num_sms;
    conv_amax_kernel<<<grid_a, kAmaxThreads, 0, st>>>(reinterpret_cast<const uint4*>(a.x), n8, a.partial);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t smem = static_cast<size_t>(a.C) * kVox * 2 + static_cast<size_t>(kVox) * (a.C / 2) +
                        static_cast<size_t>(kVox) * (a.C / 16);
    static bool attr = false;
    if (!attr) {
        e = cudaFuncSetAttribute(conv_quant_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    conv_quant_kernel<<<(a.V + kVox - 1) / kVox, 256, smem, st>>>(static_cast<const uint16_t*>(a.x), a.C, a.V,
                                                                 a.D * a.H * a.W, a.partial, grid_a, a.codes,
                                                                 a.scales, a.g);
    return cudaGetLastError();
}

cudaError_t launch_conv_gemm(const ConvArgs& a, cudaStream_t st) {
    int stages = static_cast<int>((kConvMaxSmem - 1024 - 256) / kCStage);
    if (stages > kMaxStagesTmem) stages = kMaxStagesTmem;   // scale slots beside the accumulators
    // a gather thread holds kGatherDepth stages unsignalled while it waits for a free one
    if (stages <= kGatherDepth + 1) return cudaErrorInvalidConfiguration;
    const size_t smem = static_cast<size_t>(stages) * kCStage + 256 + 1024;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(conv_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kConvMaxSmem));
        if (e != cudaSuccess) return e;
        attr = true;
    }
    ConvParams p{};
    p.C = a.C; p.D = a.D; p.H = a.H; p.W = a.W; p.V = a.V; p.V1 = a.D * a.H * a.W; p.N = a.N; p.K = 27 * a.C;
    p.stages = stages;
    p.xcodes = a.codes; p.xscales = a.scales; p.gx = a.g; p.gw = a.gw; p.sfb = a.sfb;
    p.y = static_cast<__nv_bfloat16*>(a.y); p.err = a.err;
    const int n_tiles = (a.N + 127) / 128;
    const int items = ((a.V + 127) / 128) * ((n_tiles + kGroup - 1) / kGroup);
    const int grid = items < a.num_sms ? items : a.num_sms;
    conv_gemm_kernel<<<grid, kConvThreads, smem, st>>>(*a.tmB, p);
    return cudaGetLastError();
}

}  // namespace wq
