// wq_gemm.cu -- NVFP4 x NVFP4 block-scaled GEMM on the 5th-generation tensor cores
// (tcgen05, kind::mxf4nvf4, ue4m3 scale per 16 K elements) with the fused epilogue
//     y = gA[m] gW acc4 + (U Q + x_O W_O) + b        -> bf16
// (QuantWAMs sec. 4.2 "Backend": NVFP4 W4A4 kernels plus the 16-bit exception path for the
// kept channels; Q-WAM abstract: the 16-bit low-rank branch runs as a dense matmul too.)
//
// One persistent CTA per SM, 10 warps:
//   warp 0    TMA producer: A/B code tiles (128 x 256 fp4, 128B swizzle) and the block-scale
//             atoms into an S-stage shared-memory ring; the side operands (U, Q^T, x_O, W_O^T)
//             once per tile.
//   warp 1    TMEM allocator + MMA issuer (one thread): tcgen05.cp of the scale factors into
//             TMEM, 4 x tcgen05.mma (K = 64 each) per stage, then the 16-bit side MMAs
//             (kind::f16) into a separate TMEM accumulator; tcgen05.commit frees smem stages
//             and publishes finished accumulators.
//   warps 2-9 epilogue: two warps per TMEM lane quadrant (quadrant = warp % 4), each owning
//             64 of the tile's 128 columns: tcgen05.ld of the fp32 accumulators, scale, add
//             side + bias, bf16, swizzled smem staging, one TMA store per warp.
// TMEM (512 columns): accumulator buffers at 0 and 128 (double buffered so the epilogue of
// tile t overlaps the main loop of tile t+1), side accumulator at 256, scale-factor slots
// (32 columns per ring stage) after that.
//
// Few output tiles (batch-1 shapes): the K range of one tile is split over a thread-block
// cluster of `split` CTAs (2..16).  Each CTA accumulates its K slice in TMEM and every CTA
// reduces a slice of the tile's rows over all peers, in rank order (deterministic), and
// stores bf16.  Push form (the default when the ring stages a CTA never fills can hold the
// rows): each CTA stores each row of alpha * acc (rank 0 adds the side branch) straight into
// the shared memory of the rank that reduces it, one slot per sender, and after one cluster
// barrier the sums read local shared memory.  Pull form: each CTA keeps its partial and the
// reducing ranks read every peer's through distributed shared memory between two barriers.
//
// kW8 = true runs the same pipeline on the selective 8-bit layers (FoldQuantVLA, Key
// Contribution 3): int8 codes stored as bf16 (|q| <= 127 is exact in bf16, products are
// exact in fp32) through tcgen05.mma kind::f16, 64 K per stage, no block scales, epilogue
// y = a[m] w[n] acc + b.
//
// The kernel is launched as a programmatic dependent of the activation quantiser: weight
// tiles are requested before griddepcontrol.wait, activation tiles after it.  It lets the
// next grid in the stream start its prologue early.
#include <cuda_bf16.h>

#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>

#include "ptx.cuh"
#include "wq_internal.h"

#ifdef WQ_TRACE
// Timeline probes for kernel development builds only (never defined in the product build).
__device__ unsigned long long g_wq_trace[4096 * 16];
#define WQ_TRACE_AT(slot) (g_wq_trace[blockIdx.x * 16 + (slot)] = wq::global_timer_ns())
__device__ unsigned long long g_wq_tile_trace[64 * 8];
#define WQ_TILE_AT(tl, slot) do { if (blockIdx.x == 0 && (tl) < 64) g_wq_tile_trace[(tl) * 8 + (slot)] = wq::global_timer_ns(); } while (0)
extern "C" WQ_API int wq_tile_trace_read(void* host, size_t bytes) {
    return static_cast<int>(cudaMemcpyFromSymbol(host, g_wq_tile_trace, bytes));
}
extern "C" WQ_API int wq_trace_read(void* host, size_t bytes) {
    return static_cast<int>(cudaMemcpyFromSymbol(host, g_wq_trace, bytes));
}
#else
#define WQ_TRACE_AT(slot) ((void)0)
#define WQ_TILE_AT(tl, slot) ((void)0)
#endif

namespace wq {
namespace {

constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr uint32_t kTileBytes = 128 * 128;               // 128 rows x 128 bytes (256 fp4)
constexpr uint32_t kStageBytes = 2 * kTileBytes + 2 * 4 * kSfAtom;
constexpr uint32_t kYHalfBytes = 32 * 128;               // one warp's 32 rows x 64 bf16
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
    int split;                       // CTAs per output tile (cluster x size); 1 = persistent
    __nv_bfloat16* y;                // output, written directly by the split-K reduction
    uint32_t u_bytes, xo_bytes, off_side, off_y, off_bar, sf_col;
    uint32_t off_recv;               // split-K push form: receive slots (in unused ring stages); 0 = pull
    const uint8_t* sfa;
    const uint8_t* sfb;
    const float* gA;
    float gW;
    const float* bias;
    const float* colscale;           // per-output-column scale (8-bit layers) or null
    int* err;
    int fp8;                         // 8-bit layer with e4m3 values (kind::f8f6f4, 128 K per stage)
};

__host__ __device__ constexpr uint32_t stage_bytes(bool w8) { return w8 ? 2 * kTileBytes : kStageBytes; }

Plan make_plan(int r, int n_out, int max_stages, bool w8) {
    Plan p{};
    p.u_bytes = 128u * 2u * static_cast<uint32_t>(r);
    p.xo_bytes = 128u * 2u * static_cast<uint32_t>(n_out);
    const uint32_t side = 2 * p.u_bytes + 2 * p.xo_bytes;
    const bool has_side = side > 0;
    p.sf_col = has_side ? 384 : 256;
    const int tmem_slots = static_cast<int>((512 - p.sf_col) / 32);
    int s = static_cast<int>((kMaxSmem - 1024 - side - kYBytes - kBarBytes) / stage_bytes(w8));
    if (s > tmem_slots) s = tmem_slots;
    if (s > max_stages) s = max_stages;
    p.stages = s;
    p.off_side = static_cast<uint32_t>(s) * stage_bytes(w8);
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

__device__ __forceinline__ float4 lds_v4f(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

template <bool kW8>
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
    const int n_tiles = (N + 127) / 128;
    const int tiles = ((M + 127) / 128) * n_tiles;
    constexpr uint32_t kSB = stage_bytes(kW8);
    const int kStageX = (kW8 && !p.fp8) ? 64 : 128;   // TMA x extent of a stage (elements)
    const int num_kb = p.K / 64;
    const int num_kt = kW8 ? (p.fp8 ? (num_kb + 1) / 2 : num_kb) : (num_kb + 3) / 4;
    const bool split = p.split > 1;
    const uint32_t rank = split ? cluster_ctarank() : 0u;
    const int tile_first = split ? static_cast<int>(blockIdx.x) / p.split : static_cast<int>(blockIdx.x);
    const int tile_step = split ? tiles : static_cast<int>(gridDim.x);
    const int kt_lo = split ? static_cast<int>(rank) * num_kt / p.split : 0;
    const int kt_hi = split ? (static_cast<int>(rank) + 1) * num_kt / p.split : num_kt;
    const bool has_side = (p.r + p.n_out) > 0 && rank == 0;

    if (threadIdx.x == 0) {
        WQ_TRACE_AT(0);
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_full + 8u * s, 1);
            mbar_init(bar_empty + 8u * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_tfull + 8u * b, 1);
            mbar_init(bar_tempty + 8u * b, kEpiWarps);
        }
        mbar_init(bar_sfull, 1);
        mbar_init(bar_sempty, 1);
        mbar_init(bar_stempty, kEpiWarps);
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
    // push form: peers store into this CTA's shared memory only once every CTA of the cluster
    // has started (this barrier is waited right before the first remote store)
    const bool push = split && p.off_recv != 0u;
    if (push) cluster_arrive();
    bool start_waited = false;        // each thread waits on that barrier exactly once
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    if (threadIdx.x == 0) WQ_TRACE_AT(1);
    // the next kernel in the stream may begin its prologue; it waits for this grid to
    // complete before it touches memory
    griddep_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t ph = 0, sph = 0;
            uint32_t issued = 0, issued_ph = 0;       // per-stage "ever armed" bit and its parity
            bool ok = true, first = true;
            for (int tile = tile_first; tile < tiles && ok; tile += tile_step) {
                const int mb = tile / n_tiles, nb = tile % n_tiles;
                int kt = kt_lo;
                if (first) {
                    // weights of the first stages go out before the previous grid finishes
                    first = false;
                    const int pre = min(S, kt_hi - kt_lo);
                    for (int i = 0; i < pre; ++i) {
                        const int kb0 = (kt_lo + i) * 4, nkb = min(4, num_kb - kb0);
                        const uint32_t fb = bar_full + 8u * i;
                        const uint32_t sA = base + static_cast<uint32_t>(i) * kSB;
                        mbar_arrive_expect_tx(fb, 2 * kTileBytes + (kW8 ? 0u : 2u * nkb * kSfAtom));
                        tma_load_2d(sA + kTileBytes, &tmB, (kt_lo + i) * kStageX, nb * 128, fb);
                        if (!kW8)
                            bulk_load(sA + 2 * kTileBytes + 4 * kSfAtom,
                                      p.sfb + (static_cast<size_t>(nb) * num_kb + kb0) * kSfAtom, nkb * kSfAtom, fb);
                        issued |= 1u << i;
                    }
                    WQ_TRACE_AT(2);
                    griddep_wait();
                    WQ_TRACE_AT(3);
                    for (int i = 0; i < pre; ++i) {
                        const int kb0 = (kt_lo + i) * 4, nkb = min(4, num_kb - kb0);
                        const uint32_t fb = bar_full + 8u * i;
                        const uint32_t sA = base + static_cast<uint32_t>(i) * kSB;
                        tma_load_2d(sA, &tmA, (kt_lo + i) * kStageX, mb * 128, fb);
                        if (!kW8)
                            bulk_load(sA + 2 * kTileBytes,
                                      p.sfa + (static_cast<size_t>(mb) * num_kb + kb0) * kSfAtom, nkb * kSfAtom, fb);
                    }
                    kt += pre;
                    stage = pre % S;
                    ph = pre == S ? 1u : 0u;
                }
                for (; kt < kt_hi; ++kt) {
                    if (!mbar_wait(bar_empty + 8u * stage, ph ^ 1u, abort_flag, p.err, 1)) { ok = false; break; }
                    const int kb0 = kt * 4;
                    const int nkb = min(4, num_kb - kb0);
                    const uint32_t fb = bar_full + 8u * stage;
                    const uint32_t sA = base + static_cast<uint32_t>(stage) * kSB;
                    mbar_arrive_expect_tx(fb, 2 * kTileBytes + (kW8 ? 0u : 2u * nkb * kSfAtom));
                    tma_load_2d(sA, &tmA, kt * kStageX, mb * 128, fb);
                    tma_load_2d(sA + kTileBytes, &tmB, kt * kStageX, nb * 128, fb);
                    if (!kW8) {
                        bulk_load(sA + 2 * kTileBytes, p.sfa + (static_cast<size_t>(mb) * num_kb + kb0) * kSfAtom,
                                  nkb * kSfAtom, fb);
                        bulk_load(sA + 2 * kTileBytes + 4 * kSfAtom,
                                  p.sfb + (static_cast<size_t>(nb) * num_kb + kb0) * kSfAtom, nkb * kSfAtom, fb);
                    }
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
            const uint32_t idesc_f8 = (1u << 4) | mn;                          // e4m3 x e4m3 -> f32
            int stage = 0;
            uint32_t ph = 0, sph = 0;
            int tl = 0;
            bool ok = true;
            for (int tile = tile_first; tile < tiles && ok; tile += tile_step, ++tl) {
                const int buf = tl & 1;
                const uint32_t aph = (static_cast<uint32_t>(tl) >> 1) & 1u;
                if (!mbar_wait(bar_tempty + 8u * buf, aph ^ 1u, abort_flag, p.err, 4)) { ok = false; break; }
                WQ_TILE_AT(tl, 0);
                tc_fence_after();
                const uint32_t d_acc = tmem + 128u * buf;
                // The scale factors of stage k+1 are copied into TMEM right after the MMAs of stage k
                // are issued, so the copies overlap the MMAs instead of sitting in front of them.
                auto copy_scales = [&](int stg, int ktx) {
                    if (kW8) return;
                    const int nkbx = min(4, num_kb - ktx * 4);
                    const uint32_t sAx = base + static_cast<uint32_t>(stg) * kSB;
                    const uint32_t sfx = tmem + p.sf_col + 32u * stg;
                    for (int kb = 0; kb < nkbx; ++kb) {
                        tmem_cp_32x128b_x4(sfx + 4u * kb, smem_desc(sAx + 2 * kTileBytes + kSfAtom * kb, 0, 128, 0));
                        tmem_cp_32x128b_x4(sfx + 16u + 4u * kb,
                                           smem_desc(sAx + 2 * kTileBytes + 4 * kSfAtom + kSfAtom * kb, 0, 128, 0));
                    }
                };
                for (int kt = kt_lo; kt < kt_hi; ++kt) {
                    // (TMA-filled stages need no tcgen05 fence: the mbarrier completion orders them)
                    if (!mbar_wait(bar_full + 8u * stage, ph, abort_flag, p.err, 5)) { ok = false; break; }
                    if (tl == 0 && kt == kt_lo) WQ_TRACE_AT(4);
                    const int nkb = kW8 ? (p.fp8 ? min(4, (p.K - kt * 128) / 32) : 4) : min(4, num_kb - kt * 4);
                    const uint32_t sA = base + static_cast<uint32_t>(stage) * kSB;
                    const uint32_t sf_t = tmem + p.sf_col + 32u * stage;
                    if (kt == kt_lo) copy_scales(stage, kt);
                    const uint64_t ad = smem_desc(sA, 16, 1024, 2);
                    const uint64_t bd = smem_desc(sA + kTileBytes, 16, 1024, 2);
                    for (int kb = 0; kb < nkb; ++kb) {
                        const uint32_t accum = (kt != kt_lo || kb != 0) ? 1u : 0u;
                        if (kW8 && p.fp8)
                            mma_f8(d_acc, ad + 2u * kb, bd + 2u * kb, idesc_f8, accum);
                        else if (kW8)
                            mma_f16(d_acc, ad + 2u * kb, bd + 2u * kb, idesc_bf16, accum);
                        else
                            mma_nvf4(d_acc, ad + 2u * kb, bd + 2u * kb, idesc_fp4, sf_t + 4u * kb,
                                     sf_t + 16u + 4u * kb, accum);
                    }
                    tc_commit(bar_empty + 8u * stage);
                    if (++stage == S) { stage = 0; ph ^= 1u; }
                    if (kt + 1 < kt_hi) {
                        if (!mbar_wait(bar_full + 8u * stage, ph, abort_flag, p.err, 5)) { ok = false; break; }
                        copy_scales(stage, kt + 1);
                    }
                }
                if (!ok) break;
                WQ_TILE_AT(tl, 1);
                if (has_side) {
                    if (!mbar_wait(bar_sfull, sph, abort_flag, p.err, 6)) { ok = false; break; }
                    WQ_TILE_AT(tl, 2);
                    if (!mbar_wait(bar_stempty, sph ^ 1u, abort_flag, p.err, 7)) { ok = false; break; }
                    WQ_TILE_AT(tl, 3);
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
                if (tl == 0) WQ_TRACE_AT(5);
            }
            // every MMA this thread issued has completed before TMEM is released
            tc_commit(bar_final);
            mbar_wait(bar_final, 0, abort_flag, p.err, 8);
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 2..9)
        const int q = warp & 3;                        // TMEM lane quadrant of this warp
        const int hh = (warp - 2) >> 2;                // column half: 0 -> cols 0..63, 1 -> 64..127
        const uint32_t ystage = base + p.off_y + static_cast<uint32_t>(warp - 2) * kYHalfBytes;
        const uint32_t t_lane = static_cast<uint32_t>(q * 32) << 16;
        const int row_t = q * 32 + lane;
        int tl = 0;
        griddep_wait();                                // gA is written by the previous grid
        for (int tile = tile_first; tile < tiles; tile += tile_step, ++tl) {
            const int mb = tile / n_tiles, nb = tile % n_tiles;
            const int buf = tl & 1;
            const uint32_t aph = (static_cast<uint32_t>(tl) >> 1) & 1u;
            const int row = mb * 128 + row_t;
            const float alpha = row < M ? __fmul_rn(__ldg(p.gA + row), p.gW) : 0.0f;
            const bool add_bias = p.bias != nullptr && !split;
            if (!mbar_wait(bar_tfull + 8u * buf, aph, abort_flag, p.err, 9)) break;
            if (tl == 0 && threadIdx.x == 64) WQ_TRACE_AT(6);
            if (threadIdx.x == 64) WQ_TILE_AT(tl, 4);
            tc_fence_after();
            if (!split) {
                if (lane == 0) bulk_wait_group_read0(); // staging free again
                __syncwarp();
            }
            for (int ch = 0; ch < 2; ++ch) {
                const int c0 = hh * 64 + ch * 32;       // first column of this chunk in the tile
                float4 bv[8], cv[8];
                if (p.colscale != nullptr) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int n = nb * 128 + c0 + 4 * j;
                        cv[j] = n < N ? __ldg(reinterpret_cast<const float4*>(p.colscale + n)) : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
                if (add_bias) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int n = nb * 128 + c0 + 4 * j;
                        bv[j] = n < N ? __ldg(reinterpret_cast<const float4*>(p.bias + n)) : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
                uint32_t acc[32], sd[32];
                tmem_ld_32x32b_x32(tmem + 128u * buf + static_cast<uint32_t>(c0) + t_lane, acc);
                if (has_side) tmem_ld_32x32b_x32(tmem + 256u + static_cast<uint32_t>(c0) + t_lane, sd);
                tmem_wait_ld();
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    v[i] = alpha * __uint_as_float(acc[i]);
                    if (p.colscale != nullptr) {
                        const float4& cq = cv[i / 4];
                        v[i] *= (i % 4 == 0) ? cq.x : (i % 4 == 1) ? cq.y : (i % 4 == 2) ? cq.z : cq.w;
                    }
                    if (has_side) v[i] += __uint_as_float(sd[i]);
                }
                if (add_bias) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        v[4 * j] += bv[j].x; v[4 * j + 1] += bv[j].y; v[4 * j + 2] += bv[j].z; v[4 * j + 3] += bv[j].w;
                    }
                }
                if (split) {
                    // fp32 partial of this CTA's K slice, rows swizzled by 16 B: pushed to the
                    // slot (this rank, row) of the rank that reduces the row, or kept here
                    if (row < M) {
                        if (push) {
                            if (!start_waited) {
                                cluster_wait();            // every CTA of the cluster has started
                                start_waited = true;
                            }
                            const int valid = min(128, M - mb * 128);
                            const int per = (valid + p.split - 1) / p.split;
                            const int owner = row_t / per;
                            const uint32_t drow = static_cast<uint32_t>(static_cast<int>(rank) * per + row_t - owner * per);
                            const uint32_t prow = base + p.off_recv + drow * 512u;
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const uint32_t c4 = static_cast<uint32_t>(c0 / 4 + j);
                                st_dsmem_v4f(mapa_shared(prow + ((c4 ^ (drow & 7u)) << 4), static_cast<uint32_t>(owner)),
                                             v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                            }
                        } else {
                            const uint32_t prow = base + static_cast<uint32_t>(row_t) * 512u;
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const uint32_t c4 = static_cast<uint32_t>(c0 / 4 + j);
                                st_shared_v4f(prow + ((c4 ^ (static_cast<uint32_t>(row_t) & 7u)) << 4), v[4 * j],
                                              v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                            }
                        }
                    } else if (push && !start_waited) {
                        cluster_wait();
                        start_waited = true;
                    }
                } else {
                    const uint32_t hb = ystage + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const uint32_t j = static_cast<uint32_t>(ch * 4 + jj);
                        st_shared_v4(hb + ((j ^ (static_cast<uint32_t>(lane) & 7u)) << 4),
                                     pack_bf16x2(v[8 * jj], v[8 * jj + 1]), pack_bf16x2(v[8 * jj + 2], v[8 * jj + 3]),
                                     pack_bf16x2(v[8 * jj + 4], v[8 * jj + 5]), pack_bf16x2(v[8 * jj + 6], v[8 * jj + 7]));
                    }
                }
            }
            tc_fence_before();
            if (split) {
                if (threadIdx.x == 64) WQ_TRACE_AT(7);
                break;                                 // one tile per cluster
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar_tempty + 8u * buf);
                if (has_side) mbar_arrive(bar_stempty);
            }
            if (threadIdx.x == 64) WQ_TILE_AT(tl, 5);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                const int y0 = mb * 128 + q * 32;
                if (y0 < M && nb * 128 + hh * 64 < N) tma_store_2d(&tmY, ystage, nb * 128 + hh * 64, y0);
                bulk_commit_group();
            }
        }
        if (lane == 0) bulk_wait_group0();
    }

    if (split) {
        if (push && !start_waited) cluster_wait();     // the start barrier, for every other thread
        cluster_sync();                                // every partial of the cluster is in place
        if (threadIdx.x == 64) WQ_TRACE_AT(8);
        if (warp >= 2 && tile_first < tiles) {
            const int t = threadIdx.x - 64;             // 0 .. 255
            const int mb = tile_first / n_tiles, nb = tile_first % n_tiles;
            const int valid = min(128, M - mb * 128);
            const int per = (valid + p.split - 1) / p.split;
            const int r0 = static_cast<int>(rank) * per;
            const int r1 = min(valid, r0 + per);
            for (int it = t; it < (r1 - r0) * 32; it += 32 * kEpiWarps) {
                const int row_t = r0 + it / 32;
                const uint32_t c4 = static_cast<uint32_t>(it % 32);
                float4 pv[16];
                if (push) {
                    // the slots (sender qr, row) of this rank's receive area
#pragma unroll
                    for (int qr = 0; qr < 16; ++qr)
                        if (qr < p.split) {
                            const uint32_t drow = static_cast<uint32_t>(qr * per + it / 32);
                            pv[qr] = lds_v4f(base + p.off_recv + drow * 512u + ((c4 ^ (drow & 7u)) << 4));
                        }
                } else {
                    // every peer's partial is requested before any is added, so the remote
                    // reads overlap
                    const uint32_t off = base + static_cast<uint32_t>(row_t) * 512u +
                                         ((c4 ^ (static_cast<uint32_t>(row_t) & 7u)) << 4);
#pragma unroll
                    for (int qr = 0; qr < 16; ++qr)
                        if (qr < p.split) pv[qr] = ld_dsmem_v4(mapa_shared(off, static_cast<uint32_t>(qr)));
                }
                // the sum is taken in rank order either way
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int qr = 0; qr < 16; ++qr)
                    if (qr < p.split) {
                        a.x += pv[qr].x; a.y += pv[qr].y; a.z += pv[qr].z; a.w += pv[qr].w;
                    }
                const int n0 = nb * 128 + static_cast<int>(c4) * 4;
                if (n0 < N) {
                    if (p.bias != nullptr) {
                        const float4 b = __ldg(reinterpret_cast<const float4*>(p.bias + n0));
                        a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
                    }
                    uint2 o;
                    o.x = pack_bf16x2(a.x, a.y);
                    o.y = pack_bf16x2(a.z, a.w);
                    *reinterpret_cast<uint2*>(p.y + static_cast<size_t>(mb * 128 + row_t) * N + n0) = o;
                }
            }
        }
        if (threadIdx.x == 64) WQ_TRACE_AT(9);
        if (!push) cluster_sync();                     // peers are done reading this CTA's partial
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (threadIdx.x == 0) WQ_TRACE_AT(10);
}

// Largest cluster size (power of two, <= 16, <= number of K stages) that keeps every tile's
// cluster resident at once; 1 when the tiles alone fill the GPU.
template <bool kW8>
int choose_split_uncached(int tiles, int num_kt, int num_sms, size_t smem) {
    if (tiles * 2 > num_sms) return 1;
    for (int s = 16; s >= 2; s >>= 1) {
        if (s > num_kt || tiles * s > num_sms) continue;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(static_cast<unsigned>(tiles * s));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = static_cast<unsigned>(s);
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, nvfp4_gemm_kernel<kW8>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            continue;
        }
        if (n >= tiles) return s;
    }
    return 1;
}

template <bool kW8>
int choose_split(int tiles, int num_kt, int num_sms, size_t smem) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, size_t>, int> cache;
    const auto key = std::make_tuple(tiles, num_kt, num_sms, smem);
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    const int s = choose_split_uncached<kW8>(tiles, num_kt, num_sms, smem);
    cache[key] = s;
    return s;
}

template <bool kW8>
cudaError_t gemm_attributes() {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(nvfp4_gemm_kernel<kW8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kMaxSmem));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(nvfp4_gemm_kernel<kW8>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    return cudaSuccess;
}

template <bool kW8>
Plan gemm_plan(const GemmArgs& a) {
    // the WQ_GEMM_STAGES knob caps the shared-memory ring depth (tuning)
    const int ms = tune(kTuneGemmStages);
    return make_plan(a.r, a.n_out, ms > 0 ? ms : 8, kW8);
}

// CTAs per output tile of the single-CTA schedule: the forced value, or the largest cluster
// that keeps every tile's cluster resident (1 = persistent).
template <bool kW8>
int gemm_split(const GemmArgs& a, const Plan& pl) {
    const int tiles = ((a.M + 127) / 128) * ((a.N + 127) / 128);
    const int num_kt = kW8 ? (a.fp8 ? (a.K / 64 + 1) / 2 : a.K / 64) : (a.K / 64 + 3) / 4;
    return a.force_split > 0 ? a.force_split : choose_split<kW8>(tiles, num_kt, a.num_sms, pl.total);
}

template <bool kW8>
cudaError_t launch_gemm_t(const GemmArgs& a, cudaStream_t st) {
    const Plan pl = gemm_plan<kW8>(a);
    if (pl.stages < 2) return cudaErrorInvalidConfiguration;
    const cudaError_t ea = gemm_attributes<kW8>();
    if (ea != cudaSuccess) return ea;
    const int tiles = ((a.M + 127) / 128) * ((a.N + 127) / 128);
    const int num_kt = kW8 ? (a.fp8 ? (a.K / 64 + 1) / 2 : a.K / 64) : (a.K / 64 + 3) / 4;
    const int split = gemm_split<kW8>(a, pl);
    if (split > num_kt || split > 16 || (split & (split - 1))) return cudaErrorInvalidValue;
    // split-K push form: the receive slots (per rows x split senders x 512 B) go in ring stages
    // no CTA of the cluster fills; the WQ_GEMM_PUSH knob at 0 keeps the pull form (tests and tuning)
    uint32_t off_recv = 0;
    if (split > 1) {
        const int valid = a.M < 128 ? a.M : 128;
        const int per = (valid + split - 1) / split;
        const int used = (num_kt + split - 1) / split;
        const uint32_t need = static_cast<uint32_t>(per * split) * 512u;
        if (used < pl.stages && static_cast<uint32_t>(pl.stages - used) * stage_bytes(kW8) >= need)
            off_recv = static_cast<uint32_t>(used) * stage_bytes(kW8);
        if (tune(kTuneGemmPush) == 0) off_recv = 0;
    }
    KParams kp{};
    kp.split = split;
    kp.off_recv = off_recv;
    kp.y = static_cast<__nv_bfloat16*>(a.y);
    kp.M = a.M; kp.N = a.N; kp.K = a.K; kp.r = a.r; kp.n_out = a.n_out; kp.stages = pl.stages;
    kp.u_bytes = pl.u_bytes; kp.xo_bytes = pl.xo_bytes; kp.off_side = pl.off_side; kp.off_y = pl.off_y;
    kp.off_bar = pl.off_bar; kp.sf_col = pl.sf_col;
    kp.sfa = a.sfa; kp.sfb = a.sfb; kp.gA = a.gA; kp.gW = a.gW; kp.bias = a.bias; kp.colscale = a.colscale;
    kp.err = a.err;
    kp.fp8 = a.fp8 ? 1 : 0;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(split > 1 ? tiles * split : (tiles < a.num_sms ? tiles : a.num_sms)));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = pl.total;
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    int na = 0;
    at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (split > 1) {
        at[na].id = cudaLaunchAttributeClusterDimension;
        at[na].val.clusterDim.x = static_cast<unsigned>(split);
        at[na].val.clusterDim.y = 1;
        at[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = at;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, nvfp4_gemm_kernel<kW8>, *a.tmA, *a.tmB, *a.tmU, *a.tmQ, *a.tmXO, *a.tmWO,
                              *a.tmY, kp);
}

}  // namespace

// The pair schedule or not (see launch_gemm).
bool use_wide(const GemmArgs& a) {
    bool wide = !a.w8 && a.force_split == 0 && a.K >= 1024 && wide_gemm_tiles(a.M, a.N) >= a.num_sms / 2;
    const int fw = tune(kTuneGemmWide);
    if (fw >= 0) wide = fw == 1 && a.force_split == 0;
    return wide;
}

// Within the pair schedule, the two-accumulator form (256 x 192 tiles): 4-bit layers without a
// fused next-layer quantiser, with K <= 4096 (where the per-tile drain and side branch of the
// single-buffered 256-column form are a large part of a tile) and at least 16 row tiles.
// Measured on B300: M = 16384, K = 1536: 131 -> 107 us (N = 4608), 240 -> 197 us (N = 8960),
// 55 -> 43 us (N = 1536); K = 8960 equal (172 us); M = 768, K = 2048, N = 32768 4% slower.
// The WQ_GEMM_DB knob pins it.
bool use_wide_db(const GemmArgs& a) {
    if (a.w8 || a.chain != nullptr) return false;
    const int f = tune(kTuneGemmDb);
    if (f >= 0) return f == 1;
    return a.K <= 4096 && a.M >= 4096;
}

int gemm_schedule(const GemmArgs& a) {
    if (use_wide(a)) return use_wide_db(a) ? 3 : 2;
    if (a.w8) {
        if (gemm_attributes<true>() != cudaSuccess) return -1;
        return gemm_split<true>(a, gemm_plan<true>(a)) > 1 ? 1 : 0;
    }
    if (gemm_attributes<false>() != cudaSuccess) return -1;
    return gemm_split<false>(a, gemm_plan<false>(a)) > 1 ? 1 : 0;
}

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t st) {
    if (a.M <= 0) return cudaSuccess;
    // Two schedules.  128 x 128 tiles on single CTAs (split-K over clusters when the tiles
    // alone cannot fill the GPU), bound by the tcgen05 issue of one N = 128 MMA and two scale
    // copies per 64-deep K block.  256 x 256 tiles on CTA pairs: an MMA costs the same issue
    // time at N = 128 and N = 256, and the pair kernel feeds its scale copies from a warp of
    // their own, so its MMA stream runs at the instruction rate; the accumulator is
    // single-buffered, so each tile pays the drain and the side branch before the next main
    // loop.  It is chosen for 4-bit layers with K >= 1024 whose 256 x 256 tiles fill every SM
    // pair.  The WQ_GEMM_WIDE knob pins the choice (tests and tuning).  Within the pair schedule the
    // two-accumulator form (256 x 192 tiles, wq_gemm3.cu) takes the layers with K <= 4096: it
    // costs a quarter of each MMA's columns but no MMA waits for an epilogue.
    if (a.chain == nullptr && use_wide(a) && use_wide_db(a)) return launch_gemm_wide_db(a, st);
    if (a.chain != nullptr || use_wide(a)) return launch_gemm_wide(a, st);
    return a.w8 ? launch_gemm_t<true>(a, st) : launch_gemm_t<false>(a, st);
}

}  // namespace wq
