// wq_fused.cu -- the whole W4A4 forward of a small batch (M <= 64 rows) in one kernel.
//
// Same operation as wq_quant.cu followed by wq_gemm.cu (FoldQuantVLA, Key Contributions 1-2;
// QuantWAMs sec. 3.1 and sec. 4.2 "Backend"; Q-WAM abstract), but the activation codes never
// leave shared memory: a thread-block cluster of `cs` CTAs owns one 128-column tile of y and
// splits K between its ranks; each rank quantises its own K slice of x (the row maxima and the
// low-rank partial sums meet across the cluster through distributed shared memory), writes the
// codes and scales straight into the MMA operand layout in its shared memory, multiplies them
// with the weight slice its producer streamed in since launch, and the ranks' fp32 partials are
// summed in rank order through distributed shared memory.  At batch 1 the two kernels of the
// two-launch path are latency-bound; this path removes one launch, the global round trip of
// the codes, and the wait for the whole quantiser grid.
//
// CTA (rank k of the cluster for column tile nt), 10 warps:
//   warp 0     producer: weight tile (128 rows x nb 64-blocks), its scale atoms and (rank 0)
//              the Q^T and W_O^T tiles at launch; after griddepcontrol.wait the x boxes
//              (16 rows x 64 channels each), the inv_s slice and the Omega table slice.
//   warp 1     TMEM and the single MMA-issuing thread: scale copies, nb block-scaled MMAs,
//              (rank 0) the 16-bit side MMAs, one commit.
//   warps 2-9  quantiser (pass 1: transform, kept channels out to rank 0, maxima, U share;
//              exchange; pass 2: codes and scales into the operand tile), then the split-K
//              epilogue (fp32 partials, cluster barrier, rank-ordered sum, bias, bf16).
// Work item t = g nb + i is row group g (16 rows) of block i; warp w takes items w and w + 8,
// whose transformed values stay in its registers between the passes.
// A CTA allocates all 512 TMEM columns, so the launch asks for enough shared memory that no
// two CTAs share an SM: two CTAs of one cluster on one SM would each wait for the other (one in
// tcgen05.alloc, the other at a cluster barrier).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdlib>
#include <mutex>
#include <vector>

#include "ptx.cuh"
#include "quant_block.cuh"
#include "wq_internal.h"

#ifdef WQ_TRACE
// Timeline probes for kernel development builds only (never defined in the product build).
__device__ unsigned long long g_wq_ftrace[1024 * 32];
#define WQ_FTRACE_AT(slot) do { if (blockIdx.x < 1024) g_wq_ftrace[blockIdx.x * 32 + (slot)] = wq::global_timer_ns(); } while (0)
extern "C" WQ_API int wq_ftrace_read(void* host, size_t bytes) {
    return static_cast<int>(cudaMemcpyFromSymbol(host, g_wq_ftrace, bytes));
}
#else
#define WQ_FTRACE_AT(slot) ((void)0)
#endif

namespace wq {
namespace {

constexpr int kThreads = 320;
constexpr int kQWarps = 8;
constexpr uint32_t kBox = 2048;          // one x box: 16 rows x 64 bf16
constexpr int kMaxItems = 16;
constexpr uint32_t kOneCtaPerSm = 120 * 1024;   // more than half of an SM's shared memory

struct FParams {
    int M, K, N, r, n_out;
    int nblk, nb, cs, R16;
    const float* inv_s;              // pair order
    int rotate;
    const uint32_t* omega_blk;
    const uint32_t* pfrag;
    const uint8_t* sfb;
    float gW;
    const float* bias;
    __nv_bfloat16* y;
    int* err;
    // shared-memory layout (offsets from the 1 KiB-aligned base)
    uint32_t off_a, off_b, off_sfa, off_sfb, off_u, off_xo, off_q, off_wo, off_pf, off_amax, off_rmax, off_uc, off_ga,
        off_invs, off_omega, off_bar, total;
};

// Byte offset of byte `b` of row `row` in a K-major tile of `rb`-byte rows stored with the
// shared-memory swizzle of the same width (128, 64 or 32 bytes): the 16-byte chunk index is
// XORed with address bits 7.. of the row start.
__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t b, uint32_t rb) {
    const uint32_t chunk = (b >> 4) ^ (((row * rb) >> 7) & (rb / 16u - 1u));
    return row * rb + (chunk << 4) + (b & 15u);
}
__device__ __forceinline__ uint32_t smem_layout_for(uint32_t rb) {
    return rb == 128 ? 2u : (rb == 64 ? 4u : 6u);
}
__device__ __forceinline__ void st_shared_v4u(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" :: "r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared::cluster.b16 [%0], %1;" :: "r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_v2(uint32_t addr, uint32_t a, uint32_t b) {
    asm volatile("st.shared::cluster.v2.b32 [%0], {%1, %2};" :: "r"(addr), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Kept channels of this lane's half (bit e of `mine`: channel e in the pair order of P) to rank
// 0's x_O tile, row `row`, from slot `idx` on.
__device__ __forceinline__ void send_kept(const f2 (&P)[16], uint32_t mine, uint32_t idx, uint32_t row,
                                          uint32_t xo0, uint32_t rb) {
#pragma unroll
    for (int e = 0; e < 32; ++e)
        if ((mine >> e) & 1u) {
            const float v = e < 16 ? lo2(P[e]) : hi2(P[e - 16]);
            st_cluster_u16(xo0 + swz(row, 2u * idx, rb), __half_as_ushort(__float2half_rn(v)));
            ++idx;
        }
}

template <int R>
__global__ void __launch_bounds__(kThreads, 1)
fused_forward_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmWO,
                     const FParams p) {
    constexpr int NT = R / 8;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw_addr);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();
    const int cs = p.cs, nb = p.nb, R16 = p.R16, M = p.M, N = p.N;
    const int nt = static_cast<int>(blockIdx.x) / cs;
    const int kb_lo = static_cast<int>(rank) * nb;
    const int items = R16 * nb;
    const uint32_t rb_a = static_cast<uint32_t>(nb) * 32u;   // operand row bytes (64 or 128)
    const uint32_t rb_u = 2u * static_cast<uint32_t>(p.r), rb_o = 2u * static_cast<uint32_t>(p.n_out);
    const bool has_side = (p.r + p.n_out) > 0;
    const bool side = rank == 0 && has_side;
    if (threadIdx.x == 0) WQ_FTRACE_AT(0);

    const uint32_t bar_w = base + p.off_bar, bar_c = bar_w + 8, bar_x = bar_w + 16, bar_a = bar_w + 24,
                   bar_s = bar_w + 32, bar_t = bar_w + 40, bar_p = bar_w + 48;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base_ptr + p.off_bar + 56);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    float* s_amax = reinterpret_cast<float*>(base_ptr + p.off_amax);   // [item][16 rows]
    float* s_rmax = reinterpret_cast<float*>(base_ptr + p.off_rmax);   // [64 rows]: this CTA's row maxima
    float* s_uc = reinterpret_cast<float*>(base_ptr + p.off_uc);       // [64 rows][R]: this CTA's U partial
    float* s_ga = reinterpret_cast<float*>(base_ptr + p.off_ga);       // [64 rows]: gA
    const uint32_t* s_omega = reinterpret_cast<const uint32_t*>(base_ptr + p.off_omega);

    if (threadIdx.x == 0) {
        mbar_init(bar_w, 1);
        mbar_init(bar_c, 1);
        mbar_init(bar_x, 1);
        mbar_init(bar_a, kQWarps);
        mbar_init(bar_s, static_cast<uint32_t>(cs * kQWarps));   // (rank 0) every warp of every rank
        mbar_init(bar_t, 1);
        mbar_init(bar_p, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    // the operand tile and scale atoms of the rows no item covers, and rank 0's side tiles,
    // start as zeros (rows >= M of the covered groups are zeros from the TMA fill)
    for (uint32_t o = threadIdx.x * 16u; o < 128u * rb_a; o += kThreads * 16u)
        if (o >= static_cast<uint32_t>(R16) * 16u * rb_a) st_shared_v4u(base + p.off_a + o, 0u, 0u, 0u, 0u);
    for (uint32_t o = threadIdx.x * 16u; o < static_cast<uint32_t>(nb) * kSfAtom; o += kThreads * 16u)
        st_shared_v4u(base + p.off_sfa + o, 0u, 0u, 0u, 0u);
    if (side) {
        for (uint32_t o = threadIdx.x * 16u; o < 128u * rb_u; o += kThreads * 16u) st_shared_v4u(base + p.off_u + o, 0u, 0u, 0u, 0u);
        for (uint32_t o = threadIdx.x * 16u; o < 128u * rb_o; o += kThreads * 16u) st_shared_v4u(base + p.off_xo + o, 0u, 0u, 0u, 0u);
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), 512);   // accumulator 0..127, side 128..255, scales 256..
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    cluster_arrive();               // the peers' barriers and zeroed tiles exist before remote stores
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    griddep_launch_dependents();
    if (threadIdx.x == 0) WQ_FTRACE_AT(1);

    if (warp < 2) {
        // nothing of these two warps is read across the cluster: they pass the first two
        // cluster barriers (the exchange) without waiting for their role work
        cluster_wait();
        cluster_arrive();
    }
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            // the weights are this layer's own: stream them before the previous grid finishes
            if constexpr (R > 0) {
                const uint32_t pbytes = static_cast<uint32_t>(nb * NT) * 1024u;   // P fragments of the CTA's blocks
                mbar_arrive_expect_tx(bar_p, pbytes);
                bulk_load(base + p.off_pf, p.pfrag + static_cast<size_t>(kb_lo) * NT * 256, pbytes, bar_p);
            }
            const uint32_t wbytes = 128u * rb_a + static_cast<uint32_t>(nb) * kSfAtom +
                                    (side ? 128u * (rb_u + rb_o) : 0u);
            mbar_arrive_expect_tx(bar_w, wbytes);
            tma_load_2d(base + p.off_b, &tmB, kb_lo * 32, nt * 128, bar_w);
            bulk_load(base + p.off_sfb, p.sfb + (static_cast<size_t>(nt) * p.nblk + kb_lo) * kSfAtom,
                      static_cast<uint32_t>(nb) * kSfAtom, bar_w);
            if (side && p.r) tma_load_2d(base + p.off_q, &tmQ, 0, nt * 128, bar_w);
            if (side && p.n_out) tma_load_2d(base + p.off_wo, &tmWO, 0, nt * 128, bar_w);
            griddep_wait();         // x belongs to the previous grid
            WQ_FTRACE_AT(2);
            const uint32_t cbytes = (p.inv_s ? 256u * nb : 0u) + (p.n_out ? 16u * nb : 0u);
            mbar_arrive_expect_tx(bar_c, cbytes);
            if (p.inv_s) bulk_load(base + p.off_invs, p.inv_s + kb_lo * 64, 256u * nb, bar_c);
            if (p.n_out) bulk_load(base + p.off_omega, p.omega_blk + kb_lo * 4, 16u * nb, bar_c);
            mbar_arrive_expect_tx(bar_x, static_cast<uint32_t>(items) * kBox);
            for (int t = 0; t < items; ++t)
                tma_load_2d(base + static_cast<uint32_t>(t) * kBox, &tmX, (kb_lo + t % nb) * 64, (t / nb) * 16, bar_x);
            // never leave with copies still landing in shared memory
            mbar_wait(bar_w, 0, abort_flag, p.err, 51);
            mbar_wait(bar_c, 0, abort_flag, p.err, 52);
            mbar_wait(bar_x, 0, abort_flag, p.err, 53);
            if constexpr (R > 0) mbar_wait(bar_p, 0, abort_flag, p.err, 61);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t mn = ((128u >> 3) << 17) | ((128u >> 4) << 24);
            const uint32_t idesc_fp4 = (1u << 7) | (1u << 10) | mn;
            const uint32_t idesc_bf16 = (1u << 4) | (1u << 7) | (1u << 10) | mn;
            const uint32_t idesc_f16 = (1u << 4) | mn;
            bool ok = mbar_wait(bar_w, 0, abort_flag, p.err, 54) && mbar_wait(bar_a, 0, abort_flag, p.err, 55);
            WQ_FTRACE_AT(8);
            if (ok) {
                tc_fence_after();
                const uint32_t sf = tmem + 256u;   // scale atoms: A at +4 i, B at +16 + 4 i
                for (int i = 0; i < nb; ++i) {
                    tmem_cp_32x128b_x4(sf + 4u * i, smem_desc(base + p.off_sfa + kSfAtom * i, 0, 128, 0));
                    tmem_cp_32x128b_x4(sf + 16u + 4u * i, smem_desc(base + p.off_sfb + kSfAtom * i, 0, 128, 0));
                }
                const uint32_t lay = smem_layout_for(rb_a);
                const uint64_t ad = smem_desc(base + p.off_a, 16, 8 * rb_a, lay);
                const uint64_t bd = smem_desc(base + p.off_b, 16, 8 * rb_a, lay);
                for (int i = 0; i < nb; ++i)
                    mma_nvf4(tmem, ad + 2u * i, bd + 2u * i, idesc_fp4, sf + 4u * i, sf + 16u + 4u * i, i ? 1u : 0u);
                if (side) {
                    ok = mbar_wait_cluster(bar_s, 0, abort_flag, p.err, 56);
                    if (ok) {
                        tc_fence_after();
                        uint32_t acc = 0;
                        if (p.r) {
                            const uint32_t sw = smem_layout_for(rb_u);
                            const uint64_t ud = smem_desc(base + p.off_u, 16, 8 * rb_u, sw);
                            const uint64_t qd = smem_desc(base + p.off_q, 16, 8 * rb_u, sw);
                            for (int j = 0; j < p.r / 16; ++j, acc = 1)
                                mma_f16(tmem + 128u, ud + 2u * j, qd + 2u * j, idesc_bf16, acc);
                        }
                        if (p.n_out) {
                            const uint32_t sw = smem_layout_for(rb_o);
                            const uint64_t xd = smem_desc(base + p.off_xo, 16, 8 * rb_o, sw);
                            const uint64_t wd = smem_desc(base + p.off_wo, 16, 8 * rb_o, sw);
                            for (int c = 0; c < p.n_out / 16; ++c, acc = 1)
                                mma_f16(tmem + 128u, xd + 2u * c, wd + 2u * c, idesc_f16, acc);
                        }
                    }
                }
            }
            tc_commit(bar_t);       // every MMA issued here is complete when bar_t flips
            mbar_wait(bar_t, 0, abort_flag, p.err, 60);
            WQ_FTRACE_AT(9);
        }
    } else {
        // ------------------------------------------------------------ quantiser, then epilogue
        const int wi = warp - 2;
        const int r = lane & 15, half = lane >> 4;
        const int nmine = (wi < items) + (wi + kQWarps < items);
        cluster_wait();
        bool ok = __all_sync(kQFullMask, mbar_wait(bar_c, 0, abort_flag, p.err, 57));
        ok = ok && __all_sync(kQFullMask, mbar_wait(bar_x, 0, abort_flag, p.err, 58));
        if constexpr (R > 0) ok = ok && __all_sync(kQFullMask, mbar_wait(bar_p, 0, abort_flag, p.err, 62));
        if (threadIdx.x == 64) WQ_FTRACE_AT(3);
        const uint32_t xo0 = p.n_out ? mapa_shared(base + p.off_xo, 0) : 0u;
        f2 P0[16], P1[16];
        float bm[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
        // ---- pass 1
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            if (s >= nmine || !ok) break;
            f2 (&P)[16] = s == 0 ? P0 : P1;
            const int t = wi + kQWarps * s, g = t / nb, i = t % nb;
            const uint32_t box = base + static_cast<uint32_t>(t) * kBox;
            load_transform(box, r, half, p.inv_s ? base + p.off_invs + static_cast<uint32_t>(i) * 256u : 0u, p.rotate, P);
            if (threadIdx.x == 64 && s == 0) WQ_FTRACE_AT(14);
            if constexpr (R > 0)   // the partial lands in the box
                u_step_smem<NT>(box, lane, base + p.off_pf + static_cast<uint32_t>(i * NT) * 1024u, box, true);
            if (threadIdx.x == 64 && s == 0) WQ_FTRACE_AT(15);
            const uint32_t m0 = p.n_out ? s_omega[4 * i] : 0u, m1 = p.n_out ? s_omega[4 * i + 1] : 0u;
            const uint32_t mine = half ? m1 : m0;
            if (mine != 0u) {
                send_kept(P, mine, s_omega[4 * i + 2] + (half ? static_cast<uint32_t>(__popc(m0)) : 0u),
                          static_cast<uint32_t>(g * 16 + r), xo0, rb_o);
                apply_keep(P, mine);
            }
            absmax_pairs(P, bm[s][0], bm[s][1]);
            const float am = fmaxf(fmaxf(bm[s][0], bm[s][1]), __shfl_xor_sync(kQFullMask, fmaxf(bm[s][0], bm[s][1]), 16));
            if (half == 0) s_amax[t * 16 + r] = am;
            if (threadIdx.x == 64 && s == 0) WQ_FTRACE_AT(16);
        }
        if (threadIdx.x == 64) WQ_FTRACE_AT(17);
        named_bar_sync(1, kQWarps * 32);
        if (threadIdx.x == 64) WQ_FTRACE_AT(4);
        // ---- this CTA's row maxima and U partial (blocks summed in order)
        for (int row = threadIdx.x - 64; row < R16 * 16; row += kQWarps * 32) {
            float a = 0.0f;
            for (int i = 0; i < nb; ++i) a = fmaxf(a, s_amax[((row / 16) * nb + i) * 16 + row % 16]);
            s_rmax[row] = a;
        }
        if constexpr (R > 0) {
            for (int idx = threadIdx.x - 64; idx < R16 * NT * 128; idx += kQWarps * 32) {
                const int g = idx / (NT * 128), e = idx % (NT * 128);
                float sum = 0.0f;
                for (int i = 0; i < nb; ++i) sum = __fadd_rn(sum, ld_shared_f32(base + static_cast<uint32_t>(g * nb + i) * kBox + 4u * e));
                int rr, cc;
                frag_pos(e, rr, cc);
                s_uc[(g * 16 + rr) * R + cc] = sum;
            }
        }
        cluster_arrive();
        cluster_wait();
        if (threadIdx.x == 64) WQ_FTRACE_AT(5);
        // ---- the row amax over the cluster (every rank) and U (rank 0)
        for (int row = threadIdx.x - 64; row < R16 * 16; row += kQWarps * 32) {
            float pv[16];
            const uint32_t la = smem_u32(s_rmax + row);
#pragma unroll
            for (int q = 0; q < 16; ++q)
                if (q < cs) pv[q] = ld_dsmem_f32(mapa_shared(la, static_cast<uint32_t>(q)));
            float a = 0.0f;
#pragma unroll
            for (int q = 0; q < 16; ++q)
                if (q < cs) a = fmaxf(a, pv[q]);
            s_ga[row] = __fdiv_rn(a, 2688.0f);
        }
        if constexpr (R > 0) {
            // every rank sums its slice of U over the ranks (in rank order) and writes it as
            // bf16 into rank 0's operand tile
            const int e4 = R16 * 16 * R / 4;
            const int per4 = (e4 + cs - 1) / cs;
            const int v0 = static_cast<int>(rank) * per4, v1 = min(e4, v0 + per4);
            const uint32_t u0 = mapa_shared(base + p.off_u, 0);
            for (int v = v0 + static_cast<int>(threadIdx.x) - 64; v < v1; v += kQWarps * 32) {
                float4 pv[16];
                const uint32_t la = smem_u32(s_uc) + 16u * static_cast<uint32_t>(v);
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    if (q < cs) pv[q] = ld_dsmem_v4(mapa_shared(la, static_cast<uint32_t>(q)));
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    if (q < cs) {
                        a.x += pv[q].x; a.y += pv[q].y; a.z += pv[q].z; a.w += pv[q].w;
                    }
                const int row = (4 * v) / R, j = (4 * v) % R;
                st_cluster_v2(u0 + swz(static_cast<uint32_t>(row), 2u * j, rb_u), pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w));
            }
        }
        if (has_side) {
            // U slices and kept channels (sent before the exchange) -> rank 0's tensor-core reads
            fence_proxy_async_all();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(bar_s, 0));
        }
        named_bar_sync(1, kQWarps * 32);                 // s_ga complete
        if (threadIdx.x == 64) WQ_FTRACE_AT(6);
        if (threadIdx.x == 64) WQ_FTRACE_AT(18);
        // ---- pass 2: codes and scales into the operand tile
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            if (s >= nmine || !ok) break;
            const f2 (&P)[16] = s == 0 ? P0 : P1;
            const int t = wi + kQWarps * s, g = t / nb, i = t % nb;
            const uint32_t row = static_cast<uint32_t>(g * 16 + r);
            const float gsc = s_ga[row];
            uint32_t w[4], sa, sb;
            nvfp4_half_codes<true>(P, bm[s][0], bm[s][1], gsc, __frcp_rn(gsc), w, sa, sb);
            if (threadIdx.x == 64 && s == 0) WQ_FTRACE_AT(19);
            st_shared_v4u(base + p.off_a + swz(row, static_cast<uint32_t>(32 * i + 16 * half), rb_a), w[0], w[1], w[2], w[3]);
            const uint32_t s2 = sa | (sb << 8);
            const uint32_t s2o = __shfl_xor_sync(kQFullMask, s2, 16);
            if (half == 0)
                st_shared_u32(base + p.off_sfa + kSfAtom * i + (row % 32u) * 16u + (row / 32u) * 4u, s2 | (s2o << 16));
            if (threadIdx.x == 64 && s == 0) WQ_FTRACE_AT(20);
        }
        if (threadIdx.x == 64) WQ_FTRACE_AT(21);
        fence_proxy_async_smem();                        // codes and scales -> the MMA's reads
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_a);
        if (threadIdx.x == 64) WQ_FTRACE_AT(7);

        // ---- epilogue: this rank's fp32 partial, then the rank-ordered sum
        const int q4 = warp & 3, hh = (warp - 2) >> 2;
        const uint32_t t_lane = static_cast<uint32_t>(q4 * 32) << 16;
        const int row_t = q4 * 32 + lane;
        const bool have = __all_sync(kQFullMask, mbar_wait(bar_t, 0, abort_flag, p.err, 59));
        tc_fence_after();
        if (threadIdx.x == 64) WQ_FTRACE_AT(10);
        const uint32_t part = base;                      // fp32 partials reuse the x boxes: row stride 512 B
        // tcgen05.ld is a warp-wide instruction: the whole warp loads (the condition is uniform
        // over the warp), and only the lanes of covered rows store
        if (have && q4 * 32 < R16 * 16) {
            const bool mine_row = row_t < R16 * 16;
            const float alpha = mine_row ? __fmul_rn(s_ga[row_t], p.gW) : 0.0f;
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
                const int c0 = hh * 64 + ch * 32;
                uint32_t acc[32], sd[32];
                tmem_ld_32x32b_x32(tmem + static_cast<uint32_t>(c0) + t_lane, acc);
                if (side) tmem_ld_32x32b_x32(tmem + 128u + static_cast<uint32_t>(c0) + t_lane, sd);
                tmem_wait_ld();
                if (mine_row) {
                    const uint32_t prow = part + static_cast<uint32_t>(row_t) * 512u;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        float v[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            v[e] = alpha * __uint_as_float(acc[4 * j + e]);
                            if (side) v[e] += __uint_as_float(sd[4 * j + e]);
                        }
                        const uint32_t c4 = static_cast<uint32_t>(c0 / 4 + j);
                        st_shared_v4f(prow + ((c4 ^ (static_cast<uint32_t>(row_t) & 7u)) << 4), v[0], v[1], v[2], v[3]);
                    }
                }
            }
        }
        tc_fence_before();
    }

    if (warp < 2) {
        __syncwarp();
        cluster_wait();
    }
    cluster_sync();                                      // every rank's partial is in its shared memory
    if (threadIdx.x == 64) WQ_FTRACE_AT(11);
    if (warp >= 2) {
        const int t = threadIdx.x - 64;
        const int per = (M + cs - 1) / cs;
        const int r0 = static_cast<int>(rank) * per, r1 = min(M, r0 + per);
        for (int it = t; it < (r1 - r0) * 32; it += kQWarps * 32) {
            const int row = r0 + it / 32;
            const uint32_t c4 = static_cast<uint32_t>(it % 32);
            const uint32_t off = base + static_cast<uint32_t>(row) * 512u + ((c4 ^ (static_cast<uint32_t>(row) & 7u)) << 4);
            float4 pv[16];
#pragma unroll
            for (int q = 0; q < 16; ++q)
                if (q < cs) pv[q] = ld_dsmem_v4(mapa_shared(off, static_cast<uint32_t>(q)));
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int q = 0; q < 16; ++q)
                if (q < cs) {
                    a.x += pv[q].x; a.y += pv[q].y; a.z += pv[q].z; a.w += pv[q].w;
                }
            const int n0 = nt * 128 + static_cast<int>(c4) * 4;
            if (n0 < N) {
                if (p.bias != nullptr) {
                    const float4 b = __ldg(reinterpret_cast<const float4*>(p.bias + n0));
                    a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
                }
                uint2 o;
                o.x = pack_bf16x2(a.x, a.y);
                o.y = pack_bf16x2(a.z, a.w);
                *reinterpret_cast<uint2*>(p.y + static_cast<size_t>(row) * N + n0) = o;
            }
        }
    }
    if (threadIdx.x == 64) WQ_FTRACE_AT(12);
    cluster_sync();                                      // peers are done reading this CTA's partials
    if (threadIdx.x == 0) WQ_FTRACE_AT(13);
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

using FusedKernel = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, FParams);

FusedKernel fused_kernel_for(int r) {
    switch (r) {
        case 0: return fused_forward_kernel<0>;
        case 16: return fused_forward_kernel<16>;
        case 32: return fused_forward_kernel<32>;
        default: return nullptr;
    }
}

// Shared-memory layout of one CTA (offsets from the 1 KiB-aligned base).
void fused_layout(FParams& p, int nb, int r, int n_out) {
    const uint32_t rb_a = 32u * static_cast<uint32_t>(nb);
    uint32_t off = 16u * kBox;                          // x boxes (also the fp32 partials: 64 rows x 512 B)
    auto take = [&](uint32_t bytes, uint32_t align) {
        off = (off + align - 1) / align * align;
        const uint32_t o = off;
        off += bytes;
        return o;
    };
    p.off_a = take(128u * rb_a, 1024);
    p.off_b = take(128u * rb_a, 1024);
    p.off_sfa = take(nb * kSfAtom, 1024);
    p.off_sfb = take(nb * kSfAtom, 1024);
    p.off_u = take(128u * 2u * r, 1024);
    p.off_xo = take(128u * 2u * n_out, 1024);
    p.off_q = take(128u * 2u * r, 1024);
    p.off_wo = take(128u * 2u * n_out, 1024);
    p.off_pf = take(static_cast<uint32_t>(nb) * static_cast<uint32_t>(r / 8) * 1024u, 128);
    p.off_amax = take(kMaxItems * 16 * 4, 16);
    p.off_rmax = take(64 * 4, 16);
    p.off_uc = take(64u * 4u * (r > 0 ? r : 1), 16);
    p.off_ga = take(64 * 4, 16);
    p.off_invs = take(256u * nb, 128);
    p.off_omega = take(16u * nb, 16);
    p.off_bar = take(64, 16);
    p.total = off + 1024;
    if (p.total < kOneCtaPerSm) p.total = kOneCtaPerSm;
}

cudaError_t ensure_attributes(int r) {
    // the three instantiations share one function type: each keeps its own flag
    static bool attr_set[3] = {false, false, false};
    const int slot = r == 0 ? 0 : (r == 16 ? 1 : 2);
    FusedKernel kern = fused_kernel_for(r);
    if (kern == nullptr) return cudaErrorInvalidValue;
    if (!attr_set[slot]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        attr_set[slot] = true;
    }
    return cudaSuccess;
}

// How many clusters of `cs` CTAs with `smem` bytes each can be resident at once (cached).
int max_resident_clusters(int r, int cs, uint32_t smem) {
    struct Entry { int r, cs; uint32_t smem; int n; };
    static std::mutex mu;
    static std::vector<Entry> cache;
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry& e : cache)
        if (e.r == r && e.cs == cs && e.smem == smem) return e.n;
    int n = 0;
    if (ensure_attributes(r) == cudaSuccess) {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(static_cast<unsigned>(cs));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = static_cast<unsigned>(cs);
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, fused_kernel_for(r), &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            n = 0;
        }
    }
    cache.push_back(Entry{r, cs, smem, n});
    return n;
}

}  // namespace

// Blocks per CTA and cluster size for a fused forward, or false when the batch or the shape
// is outside its range (M <= 64 rows, rank <= 32, K a multiple of 128 up to 64 blocks per
// cluster) or when the grid's clusters could not all be resident at once (a second wave would
// cost more than the two-kernel path).
bool fused_plan(int M, int K, int N, int r, int n_out, int& nb, int& cs) {
    if (M < 1 || M > 64 || (r != 0 && r != 16 && r != 32)) return false;
    const int nblk = K / 64, nt = (N + 127) / 128;
    for (int cand : {2, 4}) {
        if (nblk % cand) continue;
        const int c = nblk / cand;
        if (c > 16) continue;
        if (((M + 15) / 16) * cand > kMaxItems) continue;
        FParams p{};
        fused_layout(p, cand, r, n_out);
        if (max_resident_clusters(r, c, p.total) < nt) continue;
        nb = cand;
        cs = c;
        return true;
    }
    return false;
}

cudaError_t launch_fused(const FusedArgs& a, cudaStream_t st) {
    FParams p{};
    p.M = a.M; p.K = a.K; p.N = a.N; p.r = a.r; p.n_out = a.n_out;
    p.nblk = a.K / 64; p.nb = a.nb; p.cs = a.cs; p.R16 = (a.M + 15) / 16;
    p.inv_s = a.inv_s; p.rotate = a.rotate; p.omega_blk = a.omega_blk; p.pfrag = a.pfrag; p.sfb = a.sfb;
    p.gW = a.gW; p.bias = a.bias; p.y = static_cast<__nv_bfloat16*>(a.y); p.err = a.err;
    fused_layout(p, a.nb, a.r, a.n_out);
    const cudaError_t ea = ensure_attributes(a.r);
    if (ea != cudaSuccess) return ea;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(((a.N + 127) / 128) * a.cs));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = p.total;
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = static_cast<unsigned>(a.cs);
    at[1].val.clusterDim.y = 1;
    at[1].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, fused_kernel_for(a.r), *a.tmX, *a.tmB, *a.tmQ, *a.tmWO, p);
}

}  // namespace wq
