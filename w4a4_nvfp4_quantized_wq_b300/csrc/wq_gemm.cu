// wq_gemm.cu -- NVFP4 x NVFP4 block-scaled GEMM on the 5th-generation tensor cores
// (tcgen05, kind::mxf4nvf4, ue4m3 scale per 16 K elements) with the fused epilogue
//     y = gA[m] gW acc4 + (U Q + x_O W_O) + b        -> bf16
// (QuantWAMs sec. 4.2 "Backend": NVFP4 W4A4 kernels plus the 16-bit exception path for the
// kept channels; Q-WAM abstract: the 16-bit low-rank branch runs as a dense matmul too.)
//
// One persistent CTA per SM, 6 warps:
//   warp 0    TMA producer: A/B code tiles (128 x 256 fp4, 128B swizzle) and the block-scale
//             atoms into an S-stage shared-memory ring; the side operands (U, Q^T, x_O, W_O^T)
//             once per tile.
//   warp 1    TMEM allocator + MMA issuer (one thread): tcgen05.cp of the scale factors into
//             TMEM, 4 x tcgen05.mma (K = 64 each) per stage, then the 16-bit side MMAs
//             (kind::f16) into a separate TMEM accumulator; tcgen05.commit frees smem stages
//             and publishes finished accumulators.
//   warps 2-5 epilogue: tcgen05.ld of the fp32 accumulators (lane quadrant = warp % 4),
//             scale, add side + bias, bf16, swizzled smem staging, TMA store.
// TMEM (512 columns): accumulator buffers at 0 and 128 (double buffered so the epilogue of
// tile t overlaps the main loop of tile t+1), side accumulator at 256, scale-factor slots
// (32 columns per ring stage) after that.
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int kThreads = 192;
constexpr uint32_t kTileBytes = 128 * 128;               // 128 rows x 128 bytes (256 fp4)
constexpr uint32_t kStageBytes = 2 * kTileBytes + 2 * 4 * kSfAtom;
constexpr uint32_t kYHalfBytes = 32 * 128;               // 32 rows x 64 bf16
constexpr uint32_t kYBytes = 4 * 2 * kYHalfBytes;
constexpr uint32_t kBarBytes = 256;
constexpr uint32_t kMaxSmem = 232448;

struct Plan {
    int stages;
    uint32_t u_bytes, xo_bytes;      // one side tile (U and Q^T share u_bytes; x_O, W_O^T xo_bytes)
    uint32_t off_side, off_y, off_bar, total;
    uint32_t sf_col;                 // first TMEM column of the scale-factor slots
};

struct KParams {
    int M, N, K, r, n_out, stages;
    uint32_t u_bytes, xo_bytes, off_side, off_y, off_bar, sf_col;
    const uint8_t* sfa;
    const uint8_t* sfb;
    const float* gA;
    float gW;
    const float* bias;
    int* err;
};

Plan make_plan(int r, int n_out) {
    Plan p{};
    p.u_bytes = 128u * 2u * static_cast<uint32_t>(r);
    p.xo_bytes = 128u * 2u * static_cast<uint32_t>(n_out);
    const uint32_t side = 2 * p.u_bytes + 2 * p.xo_bytes;
    const bool has_side = side > 0;
    p.sf_col = has_side ? 384 : 256;
    const int tmem_slots = static_cast<int>((512 - p.sf_col) / 32);
    int s = static_cast<int>((kMaxSmem - 1024 - side - kYBytes - kBarBytes) / kStageBytes);
    if (s > tmem_slots) s = tmem_slots;
    if (s > 8) s = 8;
    p.stages = s;
    p.off_side = static_cast<uint32_t>(s) * kStageBytes;
    p.off_y = p.off_side + side;
    p.off_bar = p.off_y + kYBytes;
    p.total = p.off_bar + kBarBytes + 1024;
    return p;
}

__device__ __forceinline__ uint32_t swizzle_mode_for_row_bytes(uint32_t row_bytes) {
    return row_bytes == 128 ? 2u : (row_bytes == 64 ? 4u : 6u);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

__global__ void __launch_bounds__(kThreads, 1)
nvfp4_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmU, const __grid_constant__ CUtensorMap tmQ,
                  const __grid_constant__ CUtensorMap tmXO, const __grid_constant__ CUtensorMap tmWO,
                  const __grid_constant__ CUtensorMap tmY, const KParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw_addr);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int S = p.stages;
    const uint32_t bar_full = base + p.off_bar;
    const uint32_t bar_empty = bar_full + 8u * S;
    const uint32_t bar_tfull = bar_empty + 8u * S;
    const uint32_t bar_tempty = bar_tfull + 16u;
    const uint32_t bar_sfull = bar_tempty + 16u;
    const uint32_t bar_sempty = bar_sfull + 8u;
    const uint32_t bar_stempty = bar_sempty + 8u;
    const uint32_t bar_final = bar_stempty + 8u;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base_ptr + p.off_bar + 8u * (2 * S + 8));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int M = p.M, N = p.N;
    const bool has_side = (p.r + p.n_out) > 0;
    const int n_tiles = (N + 127) / 128;
    const int tiles = ((M + 127) / 128) * n_tiles;
    const int num_kb = p.K / 64;
    const int num_kt = (num_kb + 3) / 4;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_full + 8u * s, 1);
            mbar_init(bar_empty + 8u * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_tfull + 8u * b, 1);
            mbar_init(bar_tempty + 8u * b, 4);
        }
        mbar_init(bar_sfull, 1);
        mbar_init(bar_sempty, 1);
        mbar_init(bar_stempty, 4);
        mbar_init(bar_final, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmY);
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
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t ph = 0, sph = 0;
            uint32_t issued = 0, issued_ph = 0;       // per-stage "ever armed" bit and its parity
            bool ok = true;
            for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
                const int mb = tile / n_tiles, nb = tile % n_tiles;
                for (int kt = 0; kt < num_kt; ++kt) {
                    if (!mbar_wait(bar_empty + 8u * stage, ph ^ 1u, abort_flag, p.err, 1)) { ok = false; break; }
                    const int kb0 = kt * 4;
                    const int nkb = min(4, num_kb - kb0);
                    const uint32_t fb = bar_full + 8u * stage;
                    const uint32_t sA = base + static_cast<uint32_t>(stage) * kStageBytes;
                    mbar_arrive_expect_tx(fb, 2 * kTileBytes + 2u * nkb * kSfAtom);
                    tma_load_2d(sA, &tmA, kt * 128, mb * 128, fb);
                    tma_load_2d(sA + kTileBytes, &tmB, kt * 128, nb * 128, fb);
                    bulk_load(sA + 2 * kTileBytes, p.sfa + (static_cast<size_t>(mb) * num_kb + kb0) * kSfAtom,
                              nkb * kSfAtom, fb);
                    bulk_load(sA + 2 * kTileBytes + 4 * kSfAtom,
                              p.sfb + (static_cast<size_t>(nb) * num_kb + kb0) * kSfAtom, nkb * kSfAtom, fb);
                    issued |= 1u << stage;
                    issued_ph = (issued_ph & ~(1u << stage)) | (ph << stage);
                    if (++stage == S) { stage = 0; ph ^= 1u; }
                }
                if (ok && has_side) {
                    if (!mbar_wait(bar_sempty, sph ^ 1u, abort_flag, p.err, 2)) { ok = false; break; }
                    const uint32_t sU = base + p.off_side;
                    mbar_arrive_expect_tx(bar_sfull, 2 * p.u_bytes + 2 * p.xo_bytes);
                    if (p.r) {
                        tma_load_2d(sU, &tmU, 0, mb * 128, bar_sfull);
                        tma_load_2d(sU + p.u_bytes, &tmQ, 0, nb * 128, bar_sfull);
                    }
                    if (p.n_out) {
                        tma_load_2d(sU + 2 * p.u_bytes, &tmXO, 0, mb * 128, bar_sfull);
                        tma_load_2d(sU + 2 * p.u_bytes + p.xo_bytes, &tmWO, 0, nb * 128, bar_sfull);
                    }
                    sph ^= 1u;
                }
            }
            // never leave with copies still landing in shared memory
            for (int s = 0; s < S; ++s)
                if (issued & (1u << s))
                    mbar_wait(bar_full + 8u * s, (issued_ph >> s) & 1u, abort_flag, p.err, 3);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            // instruction descriptors: M = 128, N = 128, K-major A and B
            const uint32_t mn = ((128u >> 3) << 17) | ((128u >> 4) << 24);
            const uint32_t idesc_fp4 = (1u << 7) | (1u << 10) | mn;          // e2m1 x e2m1, ue4m3 scales
            const uint32_t idesc_bf16 = (1u << 4) | (1u << 7) | (1u << 10) | mn;  // bf16 x bf16 -> f32
            const uint32_t idesc_f16 = (1u << 4) | mn;                         // f16 x f16 -> f32
            int stage = 0;
            uint32_t ph = 0, sph = 0;
            int tl = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x, ++tl) {
                const int buf = tl & 1;
                const uint32_t aph = (static_cast<uint32_t>(tl) >> 1) & 1u;
                if (!mbar_wait(bar_tempty + 8u * buf, aph ^ 1u, abort_flag, p.err, 4)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_acc = tmem + 128u * buf;
                for (int kt = 0; kt < num_kt; ++kt) {
                    if (!mbar_wait(bar_full + 8u * stage, ph, abort_flag, p.err, 5)) { ok = false; break; }
                    tc_fence_after();
                    const int nkb = min(4, num_kb - kt * 4);
                    const uint32_t sA = base + static_cast<uint32_t>(stage) * kStageBytes;
                    const uint32_t sf_t = tmem + p.sf_col + 32u * stage;
                    for (int kb = 0; kb < nkb; ++kb) {
                        tmem_cp_32x128b_x4(sf_t + 4u * kb, smem_desc(sA + 2 * kTileBytes + kSfAtom * kb, 0, 128, 0));
                        tmem_cp_32x128b_x4(sf_t + 16u + 4u * kb,
                                           smem_desc(sA + 2 * kTileBytes + 4 * kSfAtom + kSfAtom * kb, 0, 128, 0));
                    }
                    const uint64_t ad = smem_desc(sA, 16, 1024, 2);
                    const uint64_t bd = smem_desc(sA + kTileBytes, 16, 1024, 2);
                    for (int kb = 0; kb < nkb; ++kb)
                        mma_nvf4(d_acc, ad + 2u * kb, bd + 2u * kb, idesc_fp4, sf_t + 4u * kb, sf_t + 16u + 4u * kb,
                                 (kt | kb) != 0 ? 1u : 0u);
                    tc_commit(bar_empty + 8u * stage);
                    if (++stage == S) { stage = 0; ph ^= 1u; }
                }
                if (!ok) break;
                if (has_side) {
                    if (!mbar_wait(bar_sfull, sph, abort_flag, p.err, 6)) { ok = false; break; }
                    if (!mbar_wait(bar_stempty, sph ^ 1u, abort_flag, p.err, 7)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_side = tmem + 256u;
                    const uint32_t sU = base + p.off_side;
                    uint32_t acc = 0;
                    if (p.r) {
                        const uint32_t rb = 2u * p.r, sw = swizzle_mode_for_row_bytes(rb);
                        const uint64_t ud = smem_desc(sU, 16, 8 * rb, sw);
                        const uint64_t qd = smem_desc(sU + p.u_bytes, 16, 8 * rb, sw);
                        for (int j = 0; j < p.r / 16; ++j, acc = 1)
                            mma_f16(d_side, ud + 2u * j, qd + 2u * j, idesc_bf16, acc);
                    }
                    if (p.n_out) {
                        const uint32_t ob = 2u * p.n_out, sw = swizzle_mode_for_row_bytes(ob);
                        const uint64_t xd = smem_desc(sU + 2 * p.u_bytes, 16, 8 * ob, sw);
                        const uint64_t wd = smem_desc(sU + 2 * p.u_bytes + p.xo_bytes, 16, 8 * ob, sw);
                        for (int c = 0; c < p.n_out / 16; ++c, acc = 1)
                            mma_f16(d_side, xd + 2u * c, wd + 2u * c, idesc_f16, acc);
                    }
                    tc_commit(bar_sempty);
                    sph ^= 1u;
                }
                tc_commit(bar_tfull + 8u * buf);
            }
            // every MMA this thread issued has completed before TMEM is released
            tc_commit(bar_final);
            mbar_wait(bar_final, 0, abort_flag, p.err, 8);
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 2..5)
        const int q = warp & 3;                        // TMEM lane quadrant of this warp
        const uint32_t ystage = base + p.off_y + static_cast<uint32_t>(q) * 2u * kYHalfBytes;
        const uint32_t t_lane = static_cast<uint32_t>(q * 32) << 16;
        int tl = 0;
        for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++tl) {
            const int mb = tile / n_tiles, nb = tile % n_tiles;
            const int buf = tl & 1;
            const uint32_t aph = (static_cast<uint32_t>(tl) >> 1) & 1u;
            if (!mbar_wait(bar_tfull + 8u * buf, aph, abort_flag, p.err, 9)) break;
            tc_fence_after();
            if (lane == 0) bulk_wait_group_read0();     // staging free again
            __syncwarp();
            const int row = mb * 128 + q * 32 + lane;
            const float alpha = row < M ? __fmul_rn(__ldg(p.gA + row), p.gW) : 0.0f;
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t acc[32], sd[32];
                tmem_ld_32x32b_x32(tmem + 128u * buf + 32u * ch + t_lane, acc);
                if (has_side) tmem_ld_32x32b_x32(tmem + 256u + 32u * ch + t_lane, sd);
                tmem_wait_ld();
                uint32_t packed[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int n0 = nb * 128 + ch * 32 + 2 * i;
                    float y0 = alpha * __uint_as_float(acc[2 * i]);
                    float y1 = alpha * __uint_as_float(acc[2 * i + 1]);
                    if (has_side) {
                        y0 += __uint_as_float(sd[2 * i]);
                        y1 += __uint_as_float(sd[2 * i + 1]);
                    }
                    if (p.bias != nullptr) {
                        if (n0 < N) y0 += __ldg(p.bias + n0);
                        if (n0 + 1 < N) y1 += __ldg(p.bias + n0 + 1);
                    }
                    packed[i] = pack_bf16x2(y0, y1);
                }
                const uint32_t hb = ystage + static_cast<uint32_t>(ch >> 1) * kYHalfBytes + lane * 128u;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const uint32_t j = static_cast<uint32_t>((ch & 1) * 4 + jj);
                    st_shared_v4(hb + ((j ^ (lane & 7u)) << 4), packed[4 * jj], packed[4 * jj + 1],
                                 packed[4 * jj + 2], packed[4 * jj + 3]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar_tempty + 8u * buf);
                if (has_side) mbar_arrive(bar_stempty);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                const int y0 = mb * 128 + q * 32;
                if (y0 < M) {
                    tma_store_2d(&tmY, ystage, nb * 128, y0);
                    if (nb * 128 + 64 < N) tma_store_2d(&tmY, ystage + kYHalfBytes, nb * 128 + 64, y0);
                }
                bulk_commit_group();
            }
        }
        if (lane == 0) bulk_wait_group0();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t st) {
    if (a.M <= 0) return cudaSuccess;
    const Plan pl = make_plan(a.r, a.n_out);
    if (pl.stages < 2) return cudaErrorInvalidConfiguration;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(nvfp4_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kMaxSmem));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    KParams kp{};
    kp.M = a.M; kp.N = a.N; kp.K = a.K; kp.r = a.r; kp.n_out = a.n_out; kp.stages = pl.stages;
    kp.u_bytes = pl.u_bytes; kp.xo_bytes = pl.xo_bytes; kp.off_side = pl.off_side; kp.off_y = pl.off_y;
    kp.off_bar = pl.off_bar; kp.sf_col = pl.sf_col;
    kp.sfa = a.sfa; kp.sfb = a.sfb; kp.gA = a.gA; kp.gW = a.gW; kp.bias = a.bias; kp.err = a.err;
    const int tiles = ((a.M + 127) / 128) * ((a.N + 127) / 128);
    const int grid = tiles < a.num_sms ? tiles : a.num_sms;
    nvfp4_gemm_kernel<<<grid, kThreads, pl.total, st>>>(*a.tmA, *a.tmB, *a.tmU, *a.tmQ, *a.tmXO, *a.tmWO,
                                                         *a.tmY, kp);
    return cudaGetLastError();
}

}  // namespace wq
