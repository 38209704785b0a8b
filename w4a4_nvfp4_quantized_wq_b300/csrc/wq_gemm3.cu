// wq_gemm3.cu -- the block-scaled NVFP4 GEMM on CTA pairs with two accumulators: 256 x 192 output
// tiles (tcgen05.mma.cta_group::2, M = 256 over the two CTAs of a cluster, N = 192), for batches
// with enough tiles to fill the GPU and a K short enough that the per-tile drain matters.  Same
// operation and epilogue as wq_gemm.cu and wq_gemm2.cu:
//     y = gA[m] gW acc4 + (U Q + x_O W_O) + b        -> bf16
// (QuantWAMs sec. 4.2 "Backend"; Q-WAM abstract for the 16-bit low-rank branch).
//
// Why 192 columns.  One MMA costs the same issue time at N = 192 as at N = 256, but two 192-column
// accumulators (384 TMEM columns) leave room for the block scales, where two 256-column ones
// would fill TMEM.  With two of them nothing on the tensor pipe waits for the epilogue: tile t's
// main loop runs into one accumulator while the other is drained and then takes tile t + 1's side
// branch.  Accumulator b's k-th use is tile k's main product (k odd for b = 1, even for b = 0)
// or tile k's side product (the other parity), so every tile has its main product in buffer t % 2
// and its side product in buffer (t + 1) % 2, each written once and read once.
//
// Per CTA of a pair (rank c), 11 warps:
//   warp 0    TMA producer: per K stage its 128 rows of the A tile and its 96 of the 192 B rows,
//             with the stage's scale boxes (A: its 128 rows; B: the tile's 192 rows, from the
//             weights' 192-row tile layout) on a barrier of their own, issued first; per tile the
//             side operands (U and x_O rows, this CTA's 96 rows of Q^T and W_O^T) into a buffer of
//             their own once the previous tile's side MMAs have completed.  Both CTAs' copies
//             complete rank 0's barriers (cta_group::2 TMA).
//   warp 1    rank 0: TMEM (collective over the pair) and the single MMA-issuing thread.  Between
//             the stages of tile t's main loop it issues tile t's side MMAs as soon as their
//             operands have landed and the other accumulator has been drained.
//   warp 10   rank 0: the scale feeder.  The scales go to TMEM in half stages (two 64-deep K
//             blocks, 24 columns) through a ring of four half slots: a copy waits for its slot's
//             MMAs of two stages before; a tcgen05.cp issued by another warp than the MMA thread
//             costs the MMA stream nothing.
//   warps 2-9 epilogue: two warps per TMEM lane quadrant, 96 columns each.  Per tile: the side
//             product into registers (release), then the main product 32 columns at a time,
//             v = RN(RN(alpha acc) + side) (release after the last), then column scales, bias and
//             bf16 out through per-warp staging and TMA stores.
// Every wait is bounded (see ptx.cuh); a CTA that gives up records its error code and the pair
// still meets at the final cluster barrier before TMEM is released.
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "quant_block.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int kThreads = 352;
constexpr int kEpiWarps = 8;
constexpr int kScaleWarp = 10;
constexpr int kN = 192;                                  // tile columns (pair MMA N)
constexpr int kStages = 4;
constexpr uint32_t kAHalf = 128 * 128;                   // this CTA's 128 A rows x 128 bytes
constexpr uint32_t kBHalf = 96 * 128;                    // this CTA's 96 B rows x 128 bytes
constexpr uint32_t kSfaOff = kAHalf + kBHalf;            // 4 A atoms (this CTA's rows)
constexpr uint32_t kSfbOff = kSfaOff + 4 * kSfAtom;      // 4 atoms of tile rows 0..127, then 4 of 128..191
constexpr uint32_t kSfStage = 12 * kSfAtom;
constexpr uint32_t kStage = kSfbOff + 8 * kSfAtom;       // 34 KiB, a multiple of 1 KiB
// side buffer: U | Q^T rows | x_O | W_O^T rows, each at a 1 KiB boundary, sized for width 64
constexpr uint32_t kSideU = 0, kSideQ = 16384, kSideX = 28672, kSideW = 45056, kSideBytes = 57344;
constexpr uint32_t kYWarp = 32 * 64;                     // per-warp staging: 32 rows x 32 bf16
constexpr uint32_t kOffSide = kStages * kStage;
constexpr uint32_t kOffY = kOffSide + kSideBytes;
constexpr uint32_t kOffBar = kOffY + kEpiWarps * kYWarp;
// barriers (8 bytes each): full[S], scf[S], empty[S], hready[4], hfree[4], done[2], bfree[2],
// sidefull, sidefree, final, sfinal; then the TMEM holder and the abort flag
constexpr uint32_t kNumBars = 3 * kStages + 4 + 4 + 2 + 2 + 4;
constexpr uint32_t kSmemBytes = kOffBar + 8 * kNumBars + 16 + 1024;
constexpr uint32_t kAcc1 = 192;                          // second accumulator's first column
constexpr uint32_t kHalfSlot0 = 384;                     // four half slots of 24 columns
constexpr uint32_t kHalfSlotCols = 24;

struct DParams {
    int M, N, K, r, n_out;
    int num_kb, num_kt;
    const float* gA;
    float gW;
    const float* bias;
    const float* colscale;
    int* err;
};

__device__ __forceinline__ uint32_t swizzle_for(uint32_t row_bytes) {
    return row_bytes == 128 ? 2u : (row_bytes == 64 ? 4u : 6u);
}
__device__ __forceinline__ void st_shared_v4u(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

__global__ void __launch_bounds__(kThreads, 1)
wide_db_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB96,
                    const __grid_constant__ CUtensorMap tmU, const __grid_constant__ CUtensorMap tmQ96,
                    const __grid_constant__ CUtensorMap tmXO, const __grid_constant__ CUtensorMap tmWO96,
                    const __grid_constant__ CUtensorMap tmY32, const __grid_constant__ CUtensorMap tmSFA,
                    const __grid_constant__ CUtensorMap tmSFB192, const DParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw_addr);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();
    constexpr uint32_t S = kStages;
    const uint32_t bar_full = base + kOffBar;
    const uint32_t bar_scf = bar_full + 8u * S;          // rank 0: both CTAs' scale boxes of a stage landed
    const uint32_t bar_empty = bar_scf + 8u * S;         // both CTAs: the stage's MMAs completed
    const uint32_t bar_hready = bar_empty + 8u * S;      // rank 0: a half slot's scales are in TMEM
    const uint32_t bar_hfree = bar_hready + 32u;         // rank 0: a half slot's MMAs completed
    const uint32_t bar_done = bar_hfree + 32u;           // both CTAs: an accumulator's product is complete
    const uint32_t bar_bfree = bar_done + 16u;           // rank 0: both epilogues have read an accumulator
    const uint32_t bar_sidefull = bar_bfree + 16u;       // rank 0: both CTAs' side operands landed
    const uint32_t bar_sidefree = bar_sidefull + 8u;     // both CTAs: the side MMAs completed
    const uint32_t bar_final = bar_sidefree + 8u;
    const uint32_t bar_sfinal = bar_final + 8u;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base_ptr + kOffBar + 8u * kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int M = p.M, N = p.N;
    const int nnt = (N + kN - 1) / kN;
    const int tiles = ((M + 255) / 256) * nnt;
    const int pair = static_cast<int>(blockIdx.x) / 2, npairs = static_cast<int>(gridDim.x) / 2;
    const bool has_side = (p.r + p.n_out) > 0;
    const int num_kt = p.num_kt;

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < S; ++s) {
            mbar_init(bar_full + 8u * s, 1);
            mbar_init(bar_scf + 8u * s, 1);
            mbar_init(bar_empty + 8u * s, 1);
        }
        for (uint32_t h = 0; h < 4; ++h) {
            mbar_init(bar_hready + 8u * h, 1);
            mbar_init(bar_hfree + 8u * h, 1);
        }
        for (uint32_t b = 0; b < 2; ++b) {
            mbar_init(bar_done + 8u * b, 1);
            mbar_init(bar_bfree + 8u * b, 2 * kEpiWarps);
        }
        mbar_init(bar_sidefull, 1);
        mbar_init(bar_sidefree, 1);
        mbar_init(bar_final, 1);
        mbar_init(bar_sfinal, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB96);
        tma_prefetch_desc(&tmSFA);
        tma_prefetch_desc(&tmSFB192);
        tma_prefetch_desc(&tmY32);
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
            const uint32_t full0 = mapa_shared(bar_full, 0), scf0 = mapa_shared(bar_scf, 0);
            const uint32_t side0 = mapa_shared(bar_sidefull, 0);
            const bool lead = rank == 0;
            const uint32_t side_bytes = 448u * static_cast<uint32_t>(p.r + p.n_out);   // (128 + 96) rows x 2 bytes
            uint32_t q = 0;
            int tl = 0;
            bool ok = true, dep = false;
            for (int tile = pair; ok && tile < tiles; tile += npairs, ++tl) {
                const int mb = tile / nnt, nb = tile % nnt;
                const int mrow = mb * 256 + static_cast<int>(rank) * 128, nrow = nb * kN + static_cast<int>(rank) * 96;
                if (has_side) {
                    // the side buffer is free once the previous tile's side MMAs have completed
                    if (tl > 0 && !mbar_wait(bar_sidefree, static_cast<uint32_t>(tl - 1) & 1u, abort_flag, p.err, 61)) {
                        ok = false;
                        break;
                    }
                    if (!dep) { griddep_wait(); dep = true; }      // U and x_O come from the previous grid
                    if (lead) mbar_arrive_expect_tx(bar_sidefull, 2u * side_bytes);
                    const uint32_t sb = base + kOffSide;
                    if (p.r > 0) {
                        tma_load_2d_pair(sb + kSideU, &tmU, 0, mrow, side0);
                        tma_load_2d_pair(sb + kSideQ, &tmQ96, 0, nrow, side0);
                    }
                    if (p.n_out > 0) {
                        tma_load_2d_pair(sb + kSideX, &tmXO, 0, mrow, side0);
                        tma_load_2d_pair(sb + kSideW, &tmWO96, 0, nrow, side0);
                    }
                }
                for (int kt = 0; kt < num_kt; ++kt, ++q) {
                    const uint32_t s = q % S;
                    if (q >= S && !mbar_wait(bar_empty + 8u * s, ((q / S) - 1u) & 1u, abort_flag, p.err, 62)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sA = base + s * kStage, fb = full0 + 8u * s, sc = scf0 + 8u * s;
                    // scale boxes first (4 K blocks each; blocks past K and rows past M or N read as
                    // zeros), the weight side before the wait on the previous grid
                    const int kb0 = kt * 4;
                    if (lead) {
                        mbar_arrive_expect_tx(bar_scf + 8u * s, 2 * kSfStage);
                        mbar_arrive_expect_tx(bar_full + 8u * s, 2 * (kAHalf + kBHalf));
                    }
                    tma_load_3d_pair(sA + kSfbOff, &tmSFB192, 0, kb0, 2 * nb, sc);
                    tma_load_2d_pair(sA + kAHalf, &tmB96, kt * 128, nrow, fb);
                    if (!dep) { griddep_wait(); dep = true; }
                    tma_load_3d_pair(sA + kSfaOff, &tmSFA, 0, kb0, 2 * mb + static_cast<int>(rank), sc);
                    tma_load_2d_pair(sA, &tmA, kt * 128, mrow, fb);
                }
            }
            // never leave with copies still landing in shared memory: stages and the side buffer
            // are released (in both CTAs) only after the MMAs that read them
            const uint32_t first = q > S ? q - S : 0u;
            for (uint32_t t = first; t < q; ++t)
                mbar_wait(bar_empty + 8u * (t % S), (t / S) & 1u, abort_flag, p.err, 63);
            if (has_side && tl > 0) mbar_wait(bar_sidefree, static_cast<uint32_t>(tl - 1) & 1u, abort_flag, p.err, 64);
        }
    } else if (warp == kScaleWarp) {
        // ------------------------------------------------------------ rank 0: scale feeder
        if (lane == 0 && rank == 0) {
            uint32_t q = 0, hq = 0;
            bool ok = true;
            for (int tile = pair; ok && tile < tiles; tile += npairs)
                for (int kt = 0; ok && kt < num_kt; ++kt, ++q) {
                    const uint32_t s = q % S;
                    if (!mbar_wait(bar_scf + 8u * s, (q / S) & 1u, abort_flag, p.err, 65)) { ok = false; break; }
                    const uint32_t sA = base + s * kStage;
                    for (int h = 0; h < 2; ++h, ++hq) {
                        const uint32_t hs = hq % 4u;
                        // the half slot's MMAs of two stages before have completed
                        if (hq >= 4u && !mbar_wait(bar_hfree + 8u * hs, ((hq / 4u) - 1u) & 1u, abort_flag, p.err, 66)) {
                            ok = false;
                            break;
                        }
                        const uint32_t slot = tmem + kHalfSlot0 + kHalfSlotCols * hs;
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            const uint32_t kb = static_cast<uint32_t>(2 * h + j);
                            tmem_cp_pair_32x128b_x4(slot + 4u * j, smem_desc(sA + kSfaOff + kSfAtom * kb, 0, 128, 0));
                            tmem_cp_pair_32x128b_x4(slot + 8u + 8u * j, smem_desc(sA + kSfbOff + kSfAtom * kb, 0, 128, 0));
                            tmem_cp_pair_32x128b_x4(slot + 12u + 8u * j,
                                                    smem_desc(sA + kSfbOff + 4 * kSfAtom + kSfAtom * kb, 0, 128, 0));
                        }
                        tc_commit_pair(bar_hready + 8u * hs);
                    }
                }
            // every copy this thread issued has completed before TMEM is released
            tc_commit_pair(bar_sfinal);
            mbar_wait(bar_sfinal, 0, abort_flag, p.err, 67);
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ------------------------------------------------------------ rank 0: MMA issuer
            const uint32_t mn = ((static_cast<uint32_t>(kN) >> 3) << 17) | ((256u >> 4) << 24);   // M = 256 (pair)
            const uint32_t idesc_fp4 = (1u << 7) | (1u << 10) | mn;
            const uint32_t idesc_bf16 = (1u << 4) | (1u << 7) | (1u << 10) | mn;
            const uint32_t idesc_f16 = (1u << 4) | mn;
            const uint32_t sb = base + kOffSide;
            uint32_t q = 0, hq = 0;
            int tl = 0;
            bool ok = true;
            // tile tl's side product into accumulator (tl + 1) % 2, once its operands have landed and
            // that accumulator's previous product (tile tl - 1's main) has been read
            auto side_ready = [&](int t, bool block) -> bool {
                const uint32_t x = static_cast<uint32_t>(t + 1) & 1u;
                if (block) {
                    if (has_side && !mbar_wait(bar_sidefull, static_cast<uint32_t>(t) & 1u, abort_flag, p.err, 68)) return false;
                    if (t > 0 && !mbar_wait(bar_bfree + 8u * x, static_cast<uint32_t>(t - 1) & 1u, abort_flag, p.err, 69))
                        return false;
                    return true;
                }
                if (has_side && !mbar_try_wait(bar_sidefull, static_cast<uint32_t>(t) & 1u)) return false;
                return t == 0 || mbar_try_wait(bar_bfree + 8u * x, static_cast<uint32_t>(t - 1) & 1u);
            };
            auto issue_side = [&](int t) {
                const uint32_t x = static_cast<uint32_t>(t + 1) & 1u;
                const uint32_t dacc = tmem + (x ? kAcc1 : 0u);
                tc_fence_after();
                uint32_t acc = 0;
                if (p.r > 0) {
                    const uint32_t rb = 2u * static_cast<uint32_t>(p.r), sw = swizzle_for(rb);
                    const uint64_t xd = smem_desc(sb + kSideU, 16, 8 * rb, sw), wd = smem_desc(sb + kSideQ, 16, 8 * rb, sw);
                    for (uint32_t j = 0; j < rb / 32u; ++j, acc = 1) mma_f16_pair(dacc, xd + 2u * j, wd + 2u * j, idesc_bf16, acc);
                }
                if (p.n_out > 0) {
                    const uint32_t rb = 2u * static_cast<uint32_t>(p.n_out), sw = swizzle_for(rb);
                    const uint64_t xd = smem_desc(sb + kSideX, 16, 8 * rb, sw), wd = smem_desc(sb + kSideW, 16, 8 * rb, sw);
                    for (uint32_t j = 0; j < rb / 32u; ++j, acc = 1) mma_f16_pair(dacc, xd + 2u * j, wd + 2u * j, idesc_f16, acc);
                }
                tc_commit_pair_mc(bar_done + 8u * x, 0x3);
                if (has_side) tc_commit_pair_mc(bar_sidefree, 0x3);
            };
            for (int tile = pair; ok && tile < tiles; tile += npairs, ++tl) {
                const uint32_t y = static_cast<uint32_t>(tl) & 1u;
                const uint32_t dacc = tmem + (y ? kAcc1 : 0u);
                // accumulator y's previous product (tile tl - 1's side) has been read
                if (tl > 0 && !mbar_wait(bar_bfree + 8u * y, static_cast<uint32_t>(tl - 1) & 1u, abort_flag, p.err, 70)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                bool side_done = false;
                for (int kt = 0; kt < num_kt; ++kt, ++q) {
                    const uint32_t s = q % S, ph = (q / S) & 1u;
                    if (!mbar_wait(bar_full + 8u * s, ph, abort_flag, p.err, 71)) { ok = false; break; }
                    const uint32_t sA = base + s * kStage;
                    const uint64_t ad = smem_desc(sA, 16, 1024, 2), bd = smem_desc(sA + kAHalf, 16, 1024, 2);
                    const int nkb = min(4, p.num_kb - kt * 4);
                    for (int h = 0; h < 2; ++h, ++hq) {
                        const uint32_t hs = hq % 4u;
                        if (!mbar_wait(bar_hready + 8u * hs, (hq / 4u) & 1u, abort_flag, p.err, 72)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t slot = tmem + kHalfSlot0 + kHalfSlotCols * hs;
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            const int kb = 2 * h + j;
                            if (kb < nkb)
                                mma_nvf4_pair(dacc, ad + 2u * static_cast<uint32_t>(kb), bd + 2u * static_cast<uint32_t>(kb),
                                              idesc_fp4, slot + 4u * j, slot + 8u + 8u * j, (kt | kb) != 0 ? 1u : 0u);
                        }
                        tc_commit_pair(bar_hfree + 8u * hs);
                    }
                    if (!ok) break;
                    tc_commit_pair_mc(bar_empty + 8u * s, 0x3);
                    if (!side_done && side_ready(tl, false)) {
                        issue_side(tl);
                        side_done = true;
                    }
                }
                if (!ok) break;
                tc_commit_pair_mc(bar_done + 8u * y, 0x3);
                if (!side_done) {
                    if (!side_ready(tl, true)) { ok = false; break; }
                    issue_side(tl);
                }
            }
            // every MMA this thread issued has completed before TMEM is released
            tc_commit_pair(bar_final);
            mbar_wait(bar_final, 0, abort_flag, p.err, 73);
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 2..9)
        const int qd = warp & 3;                          // TMEM lane quadrant
        const int hh = (warp - 2) >> 2;                   // column half of the 192-wide tile
        const uint32_t ystage = base + kOffY + static_cast<uint32_t>(warp - 2) * kYWarp;
        const uint32_t t_lane = static_cast<uint32_t>(qd * 32) << 16;
        const uint32_t bfree0 = mapa_shared(bar_bfree, 0);
        griddep_wait();                                   // gA is written by the previous grid
        int tl = 0;
        for (int tile = pair; tile < tiles; tile += npairs, ++tl) {
            const int mb = tile / nnt, nb = tile % nnt;
            const int row0 = mb * 256 + static_cast<int>(rank) * 128 + qd * 32;
            const int row = row0 + lane;
            const float alpha = row < M ? __fmul_rn(__ldg(p.gA + row), p.gW) : 0.0f;
            const uint32_t y = static_cast<uint32_t>(tl) & 1u, x = y ^ 1u;
            const uint32_t col0 = static_cast<uint32_t>(96 * hh);
            // this warp's 96 bias (and column-scale) values, one float4 per lane for lanes 0..23,
            // fetched before the waits; the column loop takes them from the owning lane by shuffle
            const int nl = nb * kN + 96 * hh + 4 * lane;
            const bool bl = lane < 24 && nl < N;
            const float4 bias4 = (p.bias != nullptr && bl) ? __ldg(reinterpret_cast<const float4*>(p.bias + nl))
                                                           : make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 cs4 = (p.colscale != nullptr && bl) ? __ldg(reinterpret_cast<const float4*>(p.colscale + nl))
                                                             : make_float4(0.f, 0.f, 0.f, 0.f);
            // the side product (accumulator x), read whole and released
            uint32_t sd0[32], sd1[32], sd2[32];
            if (!mbar_wait(bar_done + 8u * x, static_cast<uint32_t>(tl) & 1u, abort_flag, p.err, 74)) break;
            tc_fence_after();
            if (has_side) {
                const uint32_t tcol = tmem + t_lane + (x ? kAcc1 : 0u) + col0;
                tmem_ld_32x32b_x32(tcol, sd0);
                tmem_ld_32x32b_x32(tcol + 32u, sd1);
                tmem_ld_32x32b_x32(tcol + 64u, sd2);
                tmem_wait_ld();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(bfree0 + 8u * x);
            // the main product (accumulator y), 32 columns at a time: v = RN(RN(alpha acc) + side)
            if (!mbar_wait(bar_done + 8u * y, static_cast<uint32_t>(tl) & 1u, abort_flag, p.err, 75)) break;
            tc_fence_after();
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                uint32_t* sd = j == 0 ? sd0 : (j == 1 ? sd1 : sd2);
                uint32_t a[32];
                tmem_ld_32x32b_x32(tmem + t_lane + (y ? kAcc1 : 0u) + col0 + 32u * static_cast<uint32_t>(j), a);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float v = __fmul_rn(alpha, __uint_as_float(a[i]));
                    sd[i] = __float_as_uint(has_side ? __fadd_rn(v, __uint_as_float(sd[i])) : v);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(bfree0 + 8u * y);
            // column scales, bias, bf16 and the stores (32 x 32 boxes) overlap the next products
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                uint32_t* sd = j == 0 ? sd0 : (j == 1 ? sd1 : sd2);
#pragma unroll
                for (int g4 = 0; g4 < 8; ++g4) {
                    const int src = 8 * j + g4;                    // lane holding columns 32 j + 4 g4 ..
                    float v[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) v[e] = __uint_as_float(sd[4 * g4 + e]);
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
                    for (int e = 0; e < 4; ++e) sd[4 * g4 + e] = __float_as_uint(v[e]);
                }
                if (lane == 0) bulk_wait_group_read0();   // the staging buffer is free again
                __syncwarp();
                const uint32_t hb = ystage + static_cast<uint32_t>(lane) * 64u;   // row lane, 64 bytes, no swizzle
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float* f = reinterpret_cast<const float*>(&sd[8 * c]);
                    st_shared_v4u(hb + 16u * static_cast<uint32_t>(c), bf16x2(f[0], f[1]), bf16x2(f[2], f[3]),
                                  bf16x2(f[4], f[5]), bf16x2(f[6], f[7]));
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const int x0 = nb * kN + 96 * hh + 32 * j;
                    if (row0 < M && x0 < N) tma_store_2d(&tmY32, ystage, x0, row0);
                    bulk_commit_group();
                }
            }
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

int wide_db_tiles(int M, int N) { return ((M + 255) / 256) * ((N + kN - 1) / kN); }

cudaError_t launch_gemm_wide_db(const GemmArgs& a, cudaStream_t st) {
    if (a.M <= 0) return cudaSuccess;
    if (a.w8 || a.chain != nullptr || a.r > 64 || a.n_out > 64 || a.tmSFA == nullptr || a.tmB96 == nullptr ||
        a.tmSFB192 == nullptr || a.tmY32 == nullptr || (a.r > 0 && a.tmQ96 == nullptr) || (a.n_out > 0 && a.tmWO96 == nullptr))
        return cudaErrorInvalidValue;
    DParams p{};
    p.M = a.M; p.N = a.N; p.K = a.K; p.r = a.r; p.n_out = a.n_out;
    p.num_kb = a.K / 64;
    p.num_kt = (p.num_kb + 3) / 4;
    p.gA = a.gA; p.gW = a.gW; p.bias = a.bias; p.colscale = a.colscale; p.err = a.err;
    static bool attr_set = false;
    if (!attr_set) {
        const cudaError_t e = cudaFuncSetAttribute(wide_db_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int tiles = wide_db_tiles(a.M, a.N);
    const int pairs = tiles < a.num_sms / 2 ? tiles : a.num_sms / 2;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
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
    // maps a layer without the branch does not use stand in for the unused parameters
    const CUtensorMap& tu = a.r > 0 ? *a.tmU : *a.tmA;
    const CUtensorMap& tq = a.r > 0 ? *a.tmQ96 : *a.tmA;
    const CUtensorMap& tx = a.n_out > 0 ? *a.tmXO : *a.tmA;
    const CUtensorMap& tw = a.n_out > 0 ? *a.tmWO96 : *a.tmA;
    return cudaLaunchKernelEx(&cfg, wide_db_gemm_kernel, *a.tmA, *a.tmB96, tu, tq, tx, tw, *a.tmY32, *a.tmSFA,
                              *a.tmSFB192, p);
}

}  // namespace wq
