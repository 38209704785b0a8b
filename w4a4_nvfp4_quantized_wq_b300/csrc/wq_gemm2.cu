// wq_gemm2.cu -- the block-scaled NVFP4 GEMM on CTA pairs: 256 x 256 output tiles computed by
// tcgen05.mma.cta_group::2 (M = 256 over the two CTAs of a cluster, N = 256), for batches
// with enough tiles to fill the GPU.  Same operation and epilogue as wq_gemm.cu:
//     y = gA[m] gW acc4 + (U Q + x_O W_O) + b        -> bf16
// (QuantWAMs sec. 4.2 "Backend"; Q-WAM abstract for the 16-bit low-rank branch).
//
// Per CTA of a pair (rank c), 10 warps:
//   warp 0    TMA producer: its 128 rows of the A tile and its 128 of the 256 B rows, its A
//             scale atoms and all 256 rows' B scale atoms (each CTA's TMEM needs the whole
//             tile's B scales), into an S-stage ring; after the K stages of a tile, the side
//             operands (U with this CTA's Q^T rows; x_O with its W_O^T rows) as extra stages.
//             Both CTAs' copies complete rank 0's barriers directly (cta_group::2 TMA): one
//             barrier per stage for the scale atoms, issued first, and one for the operand
//             tiles, so the scales can go to TMEM while the tiles are still landing.
//   warp 1    rank 0: TMEM (collective over the pair) and the single MMA-issuing thread: the
//             pair MMAs of a stage once its tiles have landed and its scales are in TMEM; their
//             completion frees the stage in both CTAs (multicast commit).
//   warp 10   rank 0: the scale feeder.  Once both CTAs' scale atoms of a stage have landed it
//             issues the stage's tcgen05.cp.cta_group::2 copies (each CTA copies its own shared
//             memory into its own TMEM) and commits them to the stage's "scales ready" barrier.
//             A tcgen05.cp issued by the MMA thread itself stalls its MMA stream (~60-90 ns per
//             copy on B300); from another warp it costs the MMAs nothing.
//   warps 2-9 epilogue: two warps per TMEM lane quadrant, 128 columns each.  The 256-column
//             accumulator fills TMEM's first half (the other half holds five stages of scale
//             factors), so it is single-buffered: the epilogue drains it into registers and
//             releases it at once; with a side branch the pair MMAs then compute U Q + x_O W_O
//             into the same columns, which the epilogue adds chunk by chunk before the bf16
//             tile leaves through per-warp staging and TMA stores.
// Every wait is bounded (see ptx.cuh); a CTA that gives up records its error code and the
// pair still meets at the final cluster barrier before TMEM is released.
//
// kW8 = true runs the selective 8-bit layers (int8 values held as bf16) through
// kind::f16 pair MMAs, 64 K per stage, no scale factors.
#include <cuda_bf16.h>

#include <cstdlib>

#include "ptx.cuh"
#include "quant_block.cuh"
#include "quant_math.cuh"
#include "wq_internal.h"

#ifdef WQ_TRACE
// Wait-time counters for kernel development builds only (never defined in the product build).
__device__ unsigned long long g_wq_wtrace[16];   // 10: drain, 11: side read, 12: stores, 13: scales ready
extern "C" WQ_API int wq_wtrace_read(void* host, size_t bytes) {
    return static_cast<int>(cudaMemcpyFromSymbol(host, g_wq_wtrace, bytes));
}
#define WT_T0(v) const unsigned long long v = wq::global_timer_ns()
#define WT_ADD(i, t0) atomicAdd(&g_wq_wtrace[i], wq::global_timer_ns() - (t0))
#else
#define WT_T0(v) ((void)0)
#define WT_ADD(i, t0) ((void)0)
#endif

namespace wq {
namespace {

constexpr int kThreads = 352;
constexpr int kEpiWarps = 8;
constexpr int kScaleWarp = 10;
constexpr uint32_t kHalf = 128 * 128;                   // 128 rows x 128 bytes
constexpr uint32_t kSfaOff = 2 * kHalf;                 // 4 A atoms (this CTA's rows)
constexpr uint32_t kSfbOff = kSfaOff + 4 * kSfAtom;     // 4 atoms of B rows 0..127, then 4 of 128..255
constexpr uint32_t kSfStage = 12 * kSfAtom;             // one CTA's scale boxes of a stage (fixed: 4 K blocks)
constexpr uint32_t kStage4 = kSfbOff + 8 * kSfAtom;     // 38 KiB, a multiple of 1 KiB
constexpr uint32_t kStage8 = 2 * kHalf;
constexpr uint32_t kSideB = 16384;                      // offset of the B-side operand in a side stage
constexpr uint32_t kYWarp = 32 * 128;                   // per-warp staging: 32 rows x 64 bf16
constexpr uint32_t kYBytes = kEpiWarps * kYWarp;
constexpr uint32_t kMaxSmem = 232448;
constexpr uint32_t kSfCol = 256;                        // first scale-factor column
constexpr uint32_t kSfSlot = 48;                        // columns per stage: 4 x 4 (A) + 4 x 8 (B)
constexpr int kMaxStages = 5;                           // 256 + 5 x 48 <= 512 TMEM columns

struct WParams {
    int M, N, K, r, n_out, stages;
    int num_kb, num_kt;
    uint32_t off_y, off_bar;
    const float* gA;
    float gW;
    const float* bias;
    const float* colscale;
    int* err;
    int chain;               // 1: quantise the tile for the next layer instead of storing y
    ChainArgs ch;
    int fp8;                 // 8-bit layer with e4m3 values (kind::f8f6f4, 128 K per stage)
};

__host__ __device__ constexpr uint32_t stage_bytes(bool w8) { return w8 ? kStage8 : kStage4; }

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

// ---------------------------------------------------------------- chain epilogue
// One row's 64-column block held as two 32-value halves (x: columns 0..31, y: 32..63), in place.
__device__ __forceinline__ float& cv(uint32_t (&x)[32], uint32_t (&y)[32], int i) {
    return *reinterpret_cast<float*>(i < 32 ? &x[i] : &y[i - 32]);
}

// The next layer's input transform of one 64-block (FoldQuantVLA Key Contribution 2 / QuantWAMs
// Eq. (1)): smoothing before or after the Walsh-Hadamard butterflies at strides 1..32 (the pages'
// order, one fp32 add or subtract each), then the exact 1/8.  inv_pairs: the block's 64 inv_s in
// pair order (per 32-channel half, channels k and k + 16 side by side).
__device__ __forceinline__ void chain_transform(uint32_t (&x)[32], uint32_t (&y)[32], const float* inv_pairs,
                                                int rotate) {
    const bool after = (rotate & 3) == 3;
    auto smooth = [&]() {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const float2 sv = __ldg(reinterpret_cast<const float2*>(inv_pairs + 32 * hf + 2 * k));
                cv(x, y, 32 * hf + k) = __fmul_rn(cv(x, y, 32 * hf + k), sv.x);
                cv(x, y, 32 * hf + k + 16) = __fmul_rn(cv(x, y, 32 * hf + k + 16), sv.y);
            }
    };
    if (inv_pairs != nullptr && !after) smooth();
    if (rotate & 1) {
#pragma unroll
        for (int h = 1; h < 64; h <<= 1)
#pragma unroll
            for (int i = 0; i < 64; ++i)
                if ((i & h) == 0) {
                    const float a = cv(x, y, i), b = cv(x, y, i + h);
                    cv(x, y, i) = __fadd_rn(a, b);
                    cv(x, y, i + h) = __fsub_rn(a, b);
                }
#pragma unroll
        for (int i = 0; i < 64; ++i) cv(x, y, i) = __fmul_rn(cv(x, y, i), 0.125f);
        if (inv_pairs != nullptr && after) smooth();
    }
}

// Kept channels of the block to x_O (fp16) and +0 in the values; NVFP4 codes and e4m3 scales of
// the block with the fixed g (the same rounding steps as the activation quantiser), stored in the
// layouts the next layer's GEMM reads.
__device__ __forceinline__ void chain_emit(uint32_t (&x)[32], uint32_t (&y)[32], const ChainArgs& c, int m,
                                           bool row_ok, int kb, int K) {
    if (c.n_out) {
        const uint32_t m0 = __ldg(c.omega_blk + 4 * kb), m1 = __ldg(c.omega_blk + 4 * kb + 1);
        uint32_t idx = __ldg(c.omega_blk + 4 * kb + 2);
#pragma unroll
        for (int i = 0; i < 64; ++i) {
            const uint32_t bit = i < 32 ? (m0 >> i) & 1u : (m1 >> (i - 32)) & 1u;
            if (bit) {
                if (row_ok) c.xo[static_cast<size_t>(m) * c.xo_ld + idx] = __half_as_ushort(__float2half_rn(cv(x, y, i)));
                cv(x, y, i) = 0.0f;
                ++idx;
            }
        }
    }
    const float g = c.g, rg = __frcp_rn(c.g);
    uint32_t words[8], sc4 = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        float vals[16];
        float bm = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            vals[i] = cv(x, y, 16 * b + i);
            bm = fmaxf(bm, fabsf(vals[i]));
        }
        const uint32_t sc = scale_code<false>(bm, g, rg);
        const float d = __fmul_rn(dec_e4m3(sc), g);
        const float r = __frcp_rn(d);
        words[2 * b] = d != 0.0f ? e2m1_codes8_r<false>(vals, d, r) : 0u;
        words[2 * b + 1] = d != 0.0f ? e2m1_codes8_r<false>(vals + 8, d, r) : 0u;
        sc4 |= sc << (8 * b);
    }
    if (row_ok) {
        uint4* dst = reinterpret_cast<uint4*>(c.codes + static_cast<size_t>(m) * (K / 2) + kb * 32);
        dst[0] = make_uint4(words[0], words[1], words[2], words[3]);
        dst[1] = make_uint4(words[4], words[5], words[6], words[7]);
        const size_t off = (static_cast<size_t>(m / 128) * (K / 64) + kb) * kSfAtom + (m % 32) * 16 + ((m % 128) / 32) * 4;
        *reinterpret_cast<uint32_t*>(c.sf + off) = sc4;
    }
}

template <bool kW8>
__global__ void __launch_bounds__(kThreads, 1)
wide_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmU, const __grid_constant__ CUtensorMap tmQ,
                 const __grid_constant__ CUtensorMap tmXO, const __grid_constant__ CUtensorMap tmWO,
                 const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmSFA,
                 const __grid_constant__ CUtensorMap tmSFB, const WParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw_addr);
    constexpr uint32_t SB = stage_bytes(kW8);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();
    const int S = p.stages;
    const uint32_t bar_full = base + p.off_bar;
    const uint32_t bar_scf = bar_full + 8u * S;          // rank 0: both CTAs' scale atoms of the stage landed
    const uint32_t bar_empty = bar_scf + 8u * S;
    const uint32_t bar_tfull = bar_empty + 8u * S;
    const uint32_t bar_tempty = bar_tfull + 8u;          // rank 0: both epilogues drained the accumulator
    const uint32_t bar_sfull = bar_tempty + 8u;
    const uint32_t bar_sempty = bar_sfull + 8u;          // rank 0: both epilogues read the side results
    const uint32_t bar_final = bar_sempty + 8u;
    const uint32_t bar_sready = bar_final + 8u;          // rank 0: the stage's scales are in TMEM
    const uint32_t bar_sfinal = bar_sready + 8u * S;     // rank 0: the feeder's copies have all completed
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base_ptr + p.off_bar + 8u * (4 * S + 6));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int M = p.M, N = p.N;
    const int nnt = (N + 255) / 256;
    const int tiles = ((M + 255) / 256) * nnt;
    const int pair = static_cast<int>(blockIdx.x) / 2, npairs = static_cast<int>(gridDim.x) / 2;
    const bool has_side = (p.r + p.n_out) > 0;
    const int side_stages = (p.r > 0 ? 1 : 0) + (p.n_out > 0 ? 1 : 0);
    const int num_kt = p.num_kt;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_full + 8u * s, 1);
            mbar_init(bar_scf + 8u * s, 1);
            mbar_init(bar_empty + 8u * s, 1);
        }
        mbar_init(bar_tfull, 1);
        mbar_init(bar_tempty, 2 * kEpiWarps);
        mbar_init(bar_sfull, 1);
        mbar_init(bar_sempty, 2 * kEpiWarps);
        mbar_init(bar_final, 1);
        for (int s = 0; s < S; ++s) mbar_init(bar_sready + 8u * s, 1);
        mbar_init(bar_sfinal, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (!kW8) {
            tma_prefetch_desc(&tmSFA);
            tma_prefetch_desc(&tmSFB);
        }
        if (!p.chain) tma_prefetch_desc(&tmY);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_holder), 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();                 // both CTAs' barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    griddep_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer (each CTA)
        if (lane == 0) {
            // rank 0's barriers as cluster addresses: both CTAs' copies complete them, and rank 0
            // alone arms them with the pair's byte counts
            const uint32_t full0 = mapa_shared(bar_full, 0), scf0 = mapa_shared(bar_scf, 0);
            const bool lead = rank == 0;
            uint32_t q = 0;
            bool ok = true, dep = false;
            for (int tile = pair; ok && tile < tiles; tile += npairs) {
                const int mb = tile / nnt, nb = tile % nnt;
                const int mrow = mb * 256 + static_cast<int>(rank) * 128, nrow = nb * 256 + static_cast<int>(rank) * 128;
                for (int kt = 0; kt < num_kt + side_stages; ++kt, ++q) {
                    const uint32_t s = q % static_cast<uint32_t>(S);
                    WT_T0(tw0);
                    if (q >= static_cast<uint32_t>(S) &&
                        !mbar_wait(bar_empty + 8u * s, ((q / S) - 1u) & 1u, abort_flag, p.err, 31)) {
                        ok = false;
                        break;
                    }
                    WT_ADD(0, tw0);
                    const uint32_t sA = base + s * SB, fb = full0 + 8u * s, sb = scf0 + 8u * s;
                    if (kt < num_kt) {
                        if (kW8) {
                            const int x0 = kt * (p.fp8 ? 128 : 64);     // 128-byte rows either way
                            if (lead) mbar_arrive_expect_tx(bar_full + 8u * s, 4 * kHalf);
                            tma_load_2d_pair(sA + kHalf, &tmB, x0, nrow, fb);
                            if (!dep) { griddep_wait(); dep = true; }
                            tma_load_2d_pair(sA, &tmA, x0, mrow, fb);
                        } else {
                            // scale boxes first (4 K blocks each; blocks past K and rows past M or N
                            // read as zeros), the weight side before the wait on the previous grid
                            const int kb0 = kt * 4;
                            if (lead) {
                                mbar_arrive_expect_tx(bar_scf + 8u * s, 2 * kSfStage);
                                mbar_arrive_expect_tx(bar_full + 8u * s, 4 * kHalf);
                            }
                            tma_load_3d_pair(sA + kSfbOff, &tmSFB, 0, kb0, 2 * nb, sb);
                            tma_load_2d_pair(sA + kHalf, &tmB, kt * 128, nrow, fb);
                            if (!dep) { griddep_wait(); dep = true; }
                            tma_load_3d_pair(sA + kSfaOff, &tmSFA, 0, kb0, 2 * mb + static_cast<int>(rank), sb);
                            tma_load_2d_pair(sA, &tmA, kt * 128, mrow, fb);
                        }
                    } else {
                        const bool lowrank = kt == num_kt && p.r > 0;
                        if (lead) {
                            mbar_arrive_expect_tx(bar_full + 8u * s, 1024u * static_cast<uint32_t>(lowrank ? p.r : p.n_out));
                            if (!kW8) mbar_arrive(bar_scf + 8u * s);      // no scales: the phase still turns
                        }
                        tma_load_2d_pair(sA, lowrank ? &tmU : &tmXO, 0, mrow, fb);
                        tma_load_2d_pair(sA + kSideB, lowrank ? &tmQ : &tmWO, 0, nrow, fb);
                    }
                }
            }
            // never leave with copies still landing in shared memory: a stage is released (in both
            // CTAs) only after the MMAs that read it, which waited for its bytes
            const uint32_t first = q > static_cast<uint32_t>(S) ? q - S : 0u;
            for (uint32_t t = first; t < q; ++t)
                mbar_wait(bar_empty + 8u * (t % S), (t / S) & 1u, abort_flag, p.err, 32);
        }
    } else if (warp == kScaleWarp) {
        // ------------------------------------------------------------ rank 0: scale feeder
        if (!kW8 && lane == 0 && rank == 0) {
            uint32_t q = 0;
            bool ok = true;
            // one arrival per use of a stage, side-operand stages included (no copies there), so
            // the barrier's phase follows the same sequence number as the ring
            for (int tile = pair; ok && tile < tiles; tile += npairs) {
                for (int kt = 0; kt < num_kt + side_stages; ++kt, ++q) {
                    const uint32_t s = q % static_cast<uint32_t>(S), ph = (q / S) & 1u;
                    // the stage's MMAs of S uses ago completed before the producer refilled it,
                    // so the stage's TMEM slot is free once its scale atoms have landed
                    if (!mbar_wait(bar_scf + 8u * s, ph, abort_flag, p.err, 43)) { ok = false; break; }
                    if (kt < num_kt) {
                        const uint32_t sA = base + s * SB;
                        const int nkb = min(4, p.num_kb - kt * 4);
                        const uint32_t slot = tmem + kSfCol + kSfSlot * s;
                        for (int kb = 0; kb < nkb; ++kb) {
                            tmem_cp_pair_32x128b_x4(slot + 4u * kb, smem_desc(sA + kSfaOff + kSfAtom * kb, 0, 128, 0));
                            tmem_cp_pair_32x128b_x4(slot + 16u + 8u * kb,
                                                    smem_desc(sA + kSfbOff + kSfAtom * kb, 0, 128, 0));
                            tmem_cp_pair_32x128b_x4(slot + 20u + 8u * kb,
                                                    smem_desc(sA + kSfbOff + 4 * kSfAtom + kSfAtom * kb, 0, 128, 0));
                        }
                    }
                    tc_commit_pair(bar_sready + 8u * s);
                }
            }
            // every copy this thread issued has completed before TMEM is released
            tc_commit_pair(bar_sfinal);
            mbar_wait(bar_sfinal, 0, abort_flag, p.err, 46);
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ------------------------------------------------------------ rank 0: MMA issuer
            const uint32_t mn = ((256u >> 3) << 17) | ((256u >> 4) << 24);   // M = 256 (pair), N = 256
            const uint32_t idesc_fp4 = (1u << 7) | (1u << 10) | mn;
            const uint32_t idesc_bf16 = (1u << 4) | (1u << 7) | (1u << 10) | mn;
            const uint32_t idesc_f16 = (1u << 4) | mn;
            const uint32_t idesc_f8 = (1u << 4) | mn;                        // e4m3 x e4m3 -> f32
            uint32_t q = 0;
            int tl = 0;
            bool ok = true;
            for (int tile = pair; ok && tile < tiles; tile += npairs, ++tl) {
                WT_T0(tw0);
                if (tl > 0) {
                    // the accumulator columns are free once both epilogues have read the last tile
                    if (!mbar_wait(has_side ? bar_sempty : bar_tempty, static_cast<uint32_t>(tl - 1) & 1u, abort_flag,
                                   p.err, 34)) { ok = false; break; }
                }
                WT_ADD(2, tw0);
                WT_T0(tmain);
                tc_fence_after();
                for (int kt = 0; kt < num_kt; ++kt, ++q) {
                    const uint32_t s = q % static_cast<uint32_t>(S), ph = (q / S) & 1u;
                    WT_T0(tw1);
                    if (!mbar_wait(bar_full + 8u * s, ph, abort_flag, p.err, 35)) { ok = false; break; }
                    WT_ADD(3, tw1);
                    // (TMA-filled stages need no tcgen05 fence: the mbarrier completion orders them)
                    const uint32_t sA = base + s * SB;
                    const uint64_t ad = smem_desc(sA, 16, 1024, 2), bd = smem_desc(sA + kHalf, 16, 1024, 2);
                    if (kW8 && p.fp8) {
                        const int nmma = min(4, (p.K - kt * 128) / 32);
                        for (int kb = 0; kb < nmma; ++kb)
                            mma_f8_pair(tmem, ad + 2u * kb, bd + 2u * kb, idesc_f8, (kt | kb) != 0 ? 1u : 0u);
                    } else if (kW8) {
#pragma unroll
                        for (int kb = 0; kb < 4; ++kb)
                            mma_f16_pair(tmem, ad + 2u * kb, bd + 2u * kb, idesc_bf16, (kt | kb) != 0 ? 1u : 0u);
                    } else {
                        const int nkb = min(4, p.num_kb - kt * 4);
                        const uint32_t slot = tmem + kSfCol + kSfSlot * s;
                        // the scale feeder's copies of this stage have completed
                        WT_T0(tw5);
                        if (!mbar_wait(bar_sready + 8u * s, ph, abort_flag, p.err, 45)) { ok = false; break; }
                        WT_ADD(13, tw5);
                        tc_fence_after();
                        for (int kb = 0; kb < nkb; ++kb)
                            mma_nvf4_pair(tmem, ad + 2u * kb, bd + 2u * kb, idesc_fp4, slot + 4u * kb, slot + 16u + 8u * kb,
                                          (kt | kb) != 0 ? 1u : 0u);
                    }
                    tc_commit_pair_mc(bar_empty + 8u * s, 0x3);
                }
                if (!ok) break;
                tc_commit_pair_mc(bar_tfull, 0x3);
                WT_ADD(5, tmain);
                if (has_side) {
                    WT_T0(tw3);
                    if (!mbar_wait(bar_tempty, static_cast<uint32_t>(tl) & 1u, abort_flag, p.err, 37)) { ok = false; break; }
                    WT_ADD(6, tw3);
                    tc_fence_after();
                    uint32_t acc = 0;
                    for (int st = 0; st < side_stages; ++st, ++q) {
                        const uint32_t s = q % static_cast<uint32_t>(S), ph = (q / S) & 1u;
                        if (!mbar_wait(bar_full + 8u * s, ph, abort_flag, p.err, 38)) { ok = false; break; }
                        const uint32_t sA = base + s * SB;
                        const bool lowrank = st == 0 && p.r > 0;
                        const uint32_t rb = 2u * static_cast<uint32_t>(lowrank ? p.r : p.n_out);
                        const uint32_t sw = swizzle_mode_for_row_bytes(rb);
                        const uint64_t xd = smem_desc(sA, 16, 8 * rb, sw), wd = smem_desc(sA + kSideB, 16, 8 * rb, sw);
                        for (uint32_t j = 0; j < rb / 32u; ++j, acc = 1)
                            mma_f16_pair(tmem, xd + 2u * j, wd + 2u * j, lowrank ? idesc_bf16 : idesc_f16, acc);
                        tc_commit_pair_mc(bar_empty + 8u * s, 0x3);
                    }
                    if (!ok) break;
                    tc_commit_pair_mc(bar_sfull, 0x3);
                }
            }
            // every MMA this thread issued has completed before TMEM is released
            tc_commit_pair(bar_final);
            mbar_wait(bar_final, 0, abort_flag, p.err, 40);
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 2..9)
        const int qd = warp & 3;                          // TMEM lane quadrant
        const int hh = (warp - 2) >> 2;                   // column half of the 256-wide tile
        const uint32_t ystage = base + p.off_y + static_cast<uint32_t>(warp - 2) * kYWarp;
        const uint32_t t_lane = static_cast<uint32_t>(qd * 32) << 16;
        const uint32_t tempty0 = mapa_shared(bar_tempty, 0), sempty0 = mapa_shared(bar_sempty, 0);
        griddep_wait();                                   // gA is written by the previous grid
        int tl = 0;
        for (int tile = pair; tile < tiles; tile += npairs, ++tl) {
            const int mb = tile / nnt, nb = tile % nnt;
            const int row0 = mb * 256 + static_cast<int>(rank) * 128 + qd * 32;
            const int row = row0 + lane;
            const float alpha = row < M ? __fmul_rn(__ldg(p.gA + row), p.gW) : 0.0f;
            // this warp's 128 bias (and column-scale) values, one float4 per lane, fetched before
            // the accumulator wait so that their latency hides behind the main loop; the column
            // loop below takes them from the owning lane by shuffle
            const int nl = nb * 256 + 128 * hh + 4 * lane;
            const float4 bias4 = (p.bias != nullptr && nl < N) ? __ldg(reinterpret_cast<const float4*>(p.bias + nl))
                                                               : make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 cs4 = (p.colscale != nullptr && nl < N)
                                   ? __ldg(reinterpret_cast<const float4*>(p.colscale + nl))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
            WT_T0(te0);
            if (!mbar_wait(bar_tfull, static_cast<uint32_t>(tl) & 1u, abort_flag, p.err, 41)) break;
            if (lane == 0) WT_ADD(7, te0);
            WT_T0(te1);
            tc_fence_after();
            uint32_t a0[32], a1[32], a2[32], a3[32];
            const uint32_t tcol = tmem + t_lane + 128u * hh;
            tmem_ld_32x32b_x32(tcol, a0);
            tmem_ld_32x32b_x32(tcol + 32u, a1);
            tmem_ld_32x32b_x32(tcol + 64u, a2);
            tmem_ld_32x32b_x32(tcol + 96u, a3);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty0);
            if (lane == 0) WT_ADD(10, te1);
            if (has_side) {
                // alpha acc while the side MMAs run (the same RN(alpha acc) the combine below adds to)
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    a0[i] = __float_as_uint(__fmul_rn(alpha, __uint_as_float(a0[i])));
                    a1[i] = __float_as_uint(__fmul_rn(alpha, __uint_as_float(a1[i])));
                    a2[i] = __float_as_uint(__fmul_rn(alpha, __uint_as_float(a2[i])));
                    a3[i] = __float_as_uint(__fmul_rn(alpha, __uint_as_float(a3[i])));
                }
                WT_T0(te2);
                if (!mbar_wait(bar_sfull, static_cast<uint32_t>(tl) & 1u, abort_flag, p.err, 42)) break;
                if (lane == 0) WT_ADD(8, te2);
                tc_fence_after();
            }
            // before the accumulator goes back only the side results are folded in (v = RN(alpha acc)
            // + side, chunk by chunk as they are read); column scales, bias and the bf16 stores
            // follow after the release and overlap the next tile's main loop
            WT_T0(te3);
            if (has_side) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t* acc = j == 0 ? a0 : (j == 1 ? a1 : (j == 2 ? a2 : a3));
                    uint32_t sd[32];
                    tmem_ld_32x32b_x32(tmem + t_lane + static_cast<uint32_t>(128 * hh + 32 * j), sd);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        acc[i] = __float_as_uint(__fadd_rn(__uint_as_float(acc[i]), __uint_as_float(sd[i])));
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(sempty0);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t* acc = j == 0 ? a0 : (j == 1 ? a1 : (j == 2 ? a2 : a3));
#pragma unroll
                for (int g4 = 0; g4 < 8; ++g4) {
                    const int src = 8 * j + g4;                    // lane holding columns 32 j + 4 g4 ..
                    float v[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        v[e] = has_side ? __uint_as_float(acc[4 * g4 + e]) : __fmul_rn(alpha, __uint_as_float(acc[4 * g4 + e]));
                    if (p.colscale != nullptr) {
                        v[0] = __fmul_rn(v[0], __shfl_sync(0xFFFFFFFFu, cs4.x, src));
                        v[1] = __fmul_rn(v[1], __shfl_sync(0xFFFFFFFFu, cs4.y, src));
                        v[2] = __fmul_rn(v[2], __shfl_sync(0xFFFFFFFFu, cs4.z, src));
                        v[3] = __fmul_rn(v[3], __shfl_sync(0xFFFFFFFFu, cs4.w, src));
                    }
                    if (p.bias != nullptr) {
                        v[0] = __fadd_rn(v[0], __shfl_sync(0xFFFFFFFFu, bias4.x, src));
                        v[1] = __fadd_rn(v[1], __shfl_sync(0xFFFFFFFFu, bias4.y, src));
                        v[2] = __fadd_rn(v[2], __shfl_sync(0xFFFFFFFFu, bias4.z, src));
                        v[3] = __fadd_rn(v[3], __shfl_sync(0xFFFFFFFFu, bias4.w, src));
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[4 * g4 + e] = __float_as_uint(v[e]);
                }
            }
            if (lane == 0) WT_ADD(11, te3);
            WT_T0(te4);
            if (!kW8 && p.chain) {
                // the next layer's NVFP4 input from this row's 128 columns (two 64-blocks), from
                // the bf16 value the output would have stored
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    a0[i] = __float_as_uint(__bfloat162float(__float2bfloat16_rn(__uint_as_float(a0[i]))));
                    a1[i] = __float_as_uint(__bfloat162float(__float2bfloat16_rn(__uint_as_float(a1[i]))));
                    a2[i] = __float_as_uint(__bfloat162float(__float2bfloat16_rn(__uint_as_float(a2[i]))));
                    a3[i] = __float_as_uint(__bfloat162float(__float2bfloat16_rn(__uint_as_float(a3[i]))));
                }
                const bool row_ok = row < M;
                const int c0 = nb * 256 + 128 * hh;
                if (c0 < N) {
                    const int kb = c0 / 64;
                    chain_transform(a0, a1, p.ch.inv_s ? p.ch.inv_s + 64 * kb : nullptr, p.ch.rotate);
                    chain_emit(a0, a1, p.ch, row, row_ok, kb, N);
                }
                if (c0 + 64 < N) {
                    const int kb = c0 / 64 + 1;
                    chain_transform(a2, a3, p.ch.inv_s ? p.ch.inv_s + 64 * kb : nullptr, p.ch.rotate);
                    chain_emit(a2, a3, p.ch, row, row_ok, kb, N);
                }
                if (row_ok && nb == 0 && hh == 0) {
                    p.ch.g_out[row] = p.ch.g;
                    for (int cc = p.ch.n_out; cc < p.ch.xo_ld; ++cc) p.ch.xo[static_cast<size_t>(row) * p.ch.xo_ld + cc] = 0;
                }
                if (lane == 0) WT_ADD(12, te4);
                if (lane == 0) WT_ADD(9, te1);
                continue;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t* acc = j == 0 ? a0 : (j == 1 ? a1 : (j == 2 ? a2 : a3));
                if ((j & 1) == 0) {
                    if (lane == 0) bulk_wait_group_read0();   // the staging buffer is free again
                    __syncwarp();
                }
                const uint32_t hb = ystage + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const uint32_t ch = static_cast<uint32_t>((j & 1) * 4 + jj);
                    const float* f = reinterpret_cast<const float*>(acc) + 8 * jj;
                    st_shared_v4(hb + ((ch ^ (static_cast<uint32_t>(lane) & 7u)) << 4), pack_bf16x2(f[0], f[1]),
                                 pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
                }
                if (j & 1) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const int x0 = nb * 256 + 128 * hh + 64 * (j >> 1);
                        if (row0 < M && x0 < N) tma_store_2d(&tmY, ystage, x0, row0);
                        bulk_commit_group();
                    }
                }
            }
            if (lane == 0) WT_ADD(12, te4);
            if (lane == 0) WT_ADD(9, te1);
        }
        if (lane == 0) bulk_wait_group0();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();                 // the pair's MMAs (issued by rank 0) are complete in both TMEMs
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, 512);
}

}  // namespace

int wide_gemm_tiles(int M, int N) { return ((M + 255) / 256) * ((N + 255) / 256); }

cudaError_t launch_gemm_wide(const GemmArgs& a, cudaStream_t st) {
    if (a.M <= 0) return cudaSuccess;
    const bool w8 = a.w8;
    const uint32_t SB = stage_bytes(w8);
    int S = static_cast<int>((kMaxSmem - kYBytes - 2048) / SB);
    if (S > kMaxStages && !w8) S = kMaxStages;
    if (S > 8) S = 8;
    if (S < 2) return cudaErrorInvalidConfiguration;
    WParams p{};
    p.M = a.M; p.N = a.N; p.K = a.K; p.r = a.r; p.n_out = a.n_out; p.stages = S;
    p.num_kb = a.K / 64;
    p.num_kt = w8 ? (a.fp8 ? (p.num_kb + 1) / 2 : a.K / 64) : (p.num_kb + 3) / 4;
    p.fp8 = a.fp8 ? 1 : 0;
    p.off_y = static_cast<uint32_t>(S) * SB;
    p.off_bar = p.off_y + kYBytes;
    if (!w8 && (a.tmSFA == nullptr || a.tmSFB == nullptr)) return cudaErrorInvalidValue;
    p.gA = a.gA; p.gW = a.gW; p.bias = a.bias; p.colscale = a.colscale;
    p.err = a.err;
    if (a.chain != nullptr) {
        if (w8 || (a.N % 64) != 0) return cudaErrorInvalidValue;
        p.chain = 1;
        p.ch = *a.chain;
    }
    const uint32_t total = p.off_bar + 8u * (4 * S + 6) + 16u + 1024u;
    static bool attr_set[2] = {false, false};
    if (!attr_set[w8]) {
        const cudaError_t e = w8 ? cudaFuncSetAttribute(wide_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                        static_cast<int>(kMaxSmem))
                                 : cudaFuncSetAttribute(wide_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                        static_cast<int>(kMaxSmem));
        if (e != cudaSuccess) return e;
        attr_set[w8] = true;
    }
    const int tiles = wide_gemm_tiles(a.M, a.N);
    const int pairs = tiles < a.num_sms / 2 ? tiles : a.num_sms / 2;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = total;
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = 2;
    at[1].val.clusterDim.y = 1;
    at[1].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    // the 8-bit layers carry no scale boxes: any map fills the unused parameters
    const CUtensorMap& sfa = w8 ? *a.tmA : *a.tmSFA;
    const CUtensorMap& sfb = w8 ? *a.tmB : *a.tmSFB;
    if (w8)
        return cudaLaunchKernelEx(&cfg, wide_gemm_kernel<true>, *a.tmA, *a.tmB, *a.tmU, *a.tmQ, *a.tmXO, *a.tmWO,
                                  *a.tmY, sfa, sfb, p);
    return cudaLaunchKernelEx(&cfg, wide_gemm_kernel<false>, *a.tmA, *a.tmB, *a.tmU, *a.tmQ, *a.tmXO, *a.tmWO, *a.tmY,
                              sfa, sfb, p);
}

}  // namespace wq
