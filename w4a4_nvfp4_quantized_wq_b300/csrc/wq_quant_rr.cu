// wq_quant_rr.cu -- the activation quantiser for many rows of a layer with K <= 1536, with each
// row tile's transformed values kept in registers between its two passes: x is read from HBM once
// and transformed once.
//
// Same operation as wq_quant.cu (FoldQuantVLA, Key Contribution 2: channel scaling, block
// Hadamard via the FWHT with beta = 64, dynamic per-token NVFP4; QuantWAMs sec. 3.1 Eq. (1): the
// Top-K channels of the rotated basis stay in FP16; Q-WAM: the 16-bit low-rank branch U = x P):
//   xs = fp32(x) * inv_s;  xt = FWHT64(xs) * 1/8 (strides 1, 2, .., 32, in that order);
//   x_O = fp16(xt[O]), xt[O] = 0;  g = amax|xt| / 2688;  sc_b = e4m3((bmax_b / 6) / g);
//   code = e2m1(xt / (dec(sc_b) g));  U = bf16(x P).
// Every rounding is an explicit _rn operation, so the codes equal the stream and cluster
// schedules' bit for bit.
//
// Mapping.  Rows go in tiles of 16 and the 64-channel blocks of K in pairs; one persistent CTA per
// SM owns every pair of its tiles: warp w owns pair w in every tile, and lane l holds all 64
// channels of row l % 16 of the pair's block l / 16, as 32 packed pairs (channel k, channel k +
// 32).  So every FWHT stride runs in the lane's registers: strides 1..16 as packed fp32x2
// butterflies between pairs, stride 32 inside each pair.
//   pass 1    the pair's share of U (mma.sync on the two raw boxes, P staged in shared memory),
//             the transform, the kept channels, the four 16-element maxima and the row maximum;
//   exchange  row maxima and U partial sums over the warps (shared memory, warp order; the partials
//             alternate between two buffers, so one barrier a tile suffices);
//   pass 2    scales and codes from the registers.
// Each warp streams its own pair: once it has read a tile's two boxes from its shared-memory slot,
// its lane 0 issues the TMA loads of the next tile's boxes into the same slot, so the copy runs
// under the rest of the tile's work.
// (A K range wider than one CTA's goes to the stream schedule: spreading it over a cluster and
// exchanging the row maxima and U sums every tile measured slower than streaming it twice.)
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "ptx.cuh"
#include "quant_block.cuh"
#include "quant_math.cuh"
#include "wq_internal.h"

#ifdef WQ_TRACE
// Per-phase cycle counters for kernel development builds only (never defined in the product build).
__device__ unsigned long long g_wq_rtrace[16];
extern "C" WQ_API int wq_rtrace_read(void* host, size_t bytes) {
    return static_cast<int>(cudaMemcpyFromSymbol(host, g_wq_rtrace, bytes));
}
#define RT_DECL unsigned long long rt_acc[8] = {0, 0, 0, 0, 0, 0, 0, 0}; long long rt_t = clock64(), rt_n = 0
#define RT(i) do { const long long t_ = clock64(); rt_acc[i] += static_cast<unsigned long long>(t_ - rt_t); rt_t = t_; } while (0)
#define RT_TILE() (++rt_n)
#define RT_FLUSH() do { if (lane == 0) { for (int i_ = 0; i_ < 8; ++i_) atomicAdd(&g_wq_rtrace[i_], rt_acc[i_]); \
                                           atomicAdd(&g_wq_rtrace[8], static_cast<unsigned long long>(rt_n)); } } while (0)
#else
#define RT_DECL
#define RT(i) ((void)0)
#define RT_TILE() ((void)0)
#define RT_FLUSH() ((void)0)
#endif

namespace wq {
namespace {

constexpr int kRTile = 16;                          // rows per tile
constexpr int kMaxPairs = 12;                       // warps per CTA (one CTA per SM)
constexpr uint32_t kRBox = kRTile * 128;            // one TMA box: 16 rows x 64 bf16
constexpr uint32_t kRSlot = 2 * kRBox;              // a pair's two boxes
constexpr uint32_t kSmemBudget = 226 * 1024;
constexpr unsigned kRMask = 0xFFFFFFFFu;

struct RParams {
    int M, K, nblk, npairs;
    int W;                  // pairs (warps) per CTA
    int row_tiles;
    const float* inv_s;     // [K] in (k, k + 32) pair order per block, or null
    int rotate;             // bit 0: FWHT; bit 1: smoothing after it
    const uint32_t* omega_blk;
    int n_out, xo_ld;
    uint16_t* xo;
    const uint32_t* pfrag;  // P in mma.sync B-fragment order
    int p_smem;             // 1: pfrag is staged in shared memory
    uint16_t* u;
    uint8_t* codes;
    uint8_t* sf;
    int sf_layout;
    float* g;
    int* err;
};

struct RLayout {
    uint32_t off_p, off_invs, off_omega, off_upart, off_amax, off_bar, off_abort, total;
};

__host__ __device__ inline RLayout make_rlayout(int W, int R, bool p_smem) {
    RLayout l{};
    const uint32_t nb = 2u * static_cast<uint32_t>(W), nt = static_cast<uint32_t>(R / 8);
    l.off_p = static_cast<uint32_t>(W) * kRSlot;                       // slots first (1024-aligned)
    l.off_invs = l.off_p + (p_smem ? nb * nt * 1024u : 0u);
    l.off_omega = l.off_invs + 256u * nb;
    // per tile parity: the warps' U partials (fragment order) and row maxima
    l.off_upart = l.off_omega + 16u * nb;
    l.off_amax = l.off_upart + 2u * static_cast<uint32_t>(W) * nt * 512u;
    l.off_bar = (l.off_amax + 2u * 4u * kRTile * static_cast<uint32_t>(W) + 7u) & ~7u;
    l.off_abort = l.off_bar + 8u * (static_cast<uint32_t>(W) + 1u);
    l.total = l.off_abort + 16u + 1024u;                               // + alignment slack
    return l;
}

// The pair's share of U for the tile's 16 rows: every n-tile of P over the pair's 128 channels
// accumulated on the tensor cores, then stored to the warp's partial (fragment order, NT x 512 B).
template <int NT>
__device__ __forceinline__ void u_pair(uint32_t slot, int lane, int nblocks, const RParams& p, int kb0, uint32_t pf_s,
                                       uint32_t upart) {
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;
#pragma unroll
    for (int bb = 0; bb < 2; ++bb) {
        if (bb < nblocks) {
            uint32_t a[4][4];
            u_frags(slot + static_cast<uint32_t>(bb) * kRBox, lane, a);
            // n-tiles in groups of up to four: the group's P fragments, then its tensor-core
            // chains issued interleaved (independent chains; each runs its four k-steps in order
            // from zero, so the accumulation depth is 64 as in the other schedules), then one
            // fp32 add per partial
            constexpr int NG = NT < 4 ? NT : (NT > 4 ? 2 : 4);   // rank 64: pairs, for registers
#pragma unroll
            for (int n0 = 0; n0 < NT; n0 += NG) {
                uint4 q[NG][2];
                if (p.p_smem) {
#pragma unroll
                    for (int g = 0; g < NG; ++g) {
                        const uint32_t pb =
                            pf_s + ((static_cast<uint32_t>(bb * NT + n0 + g)) * 32u + static_cast<uint32_t>(lane)) * 32u;
                        q[g][0] = ld_shared_v4(pb);
                        q[g][1] = ld_shared_v4(pb + 16u);
                    }
                } else {
#pragma unroll
                    for (int g = 0; g < NG; ++g) {
                        const uint4* pb = reinterpret_cast<const uint4*>(
                            p.pfrag + (static_cast<size_t>((kb0 + bb) * NT + n0 + g) * 32 + lane) * 8);
                        q[g][0] = __ldg(pb);
                        q[g][1] = __ldg(pb + 1);
                    }
                }
                float t[NG][4];
#pragma unroll
                for (int g = 0; g < NG; ++g) t[g][0] = t[g][1] = t[g][2] = t[g][3] = 0.0f;
#pragma unroll
                for (int f = 0; f < 4; ++f)
#pragma unroll
                    for (int g = 0; g < NG; ++g) {
                        const uint4& qq = q[g][f >> 1];
                        mma_bf16_16816(t[g], a[f][0], a[f][1], a[f][2], a[f][3], (f & 1) ? qq.z : qq.x,
                                       (f & 1) ? qq.w : qq.y);
                    }
#pragma unroll
                for (int g = 0; g < NG; ++g)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[n0 + g][e] = __fadd_rn(acc[n0 + g][e], t[g][e]);
            }
        }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
        st_shared_v4f(upart + (static_cast<uint32_t>(nt) * 32u + static_cast<uint32_t>(lane)) * 16u, acc[nt][0],
                      acc[nt][1], acc[nt][2], acc[nt][3]);
}

// Row r of a raw box (128-byte swizzle: 16-byte chunk c of row r at c ^ (r % 8)) as 32 pairs
// (channel k, channel k + 32) in fp32.
__device__ __forceinline__ void load_row64(uint32_t box, int r, f2 (&V)[32]) {
    const uint32_t rb = box + static_cast<uint32_t>(r) * 128u, sw = static_cast<uint32_t>(r) & 7u;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint4 lo = ld_shared_v4(rb + ((static_cast<uint32_t>(c) ^ sw) << 4));
        const uint4 hi = ld_shared_v4(rb + ((static_cast<uint32_t>(c + 4) ^ sw) << 4));
        const uint32_t wl[4] = {lo.x, lo.y, lo.z, lo.w}, wh[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint32_t a = wl[e / 2], b = wh[e / 2];
            V[8 * c + e] = (e & 1) ? pk2(__uint_as_float(a & 0xFFFF0000u), __uint_as_float(b & 0xFFFF0000u))
                                   : pk2(__uint_as_float(a << 16), __uint_as_float(b << 16));
        }
    }
}

// V *= inv_s (the block's 64 values in pair order at shared address invs).
__device__ __forceinline__ void smooth64(f2 (&V)[32], uint32_t invs) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const float4 sv = ld_shared_v4f(invs + 16u * j);
        V[2 * j] = mul2(V[2 * j], pk2(sv.x, sv.y));
        V[2 * j + 1] = mul2(V[2 * j + 1], pk2(sv.z, sv.w));
    }
}

// The block-64 FWHT in the pages' order (strides 1, 2, 4, 8, 16 between pairs, 32 inside each
// pair; position k takes a + b and k + h takes a - b), then the exact 1/8.
__device__ __forceinline__ void fwht64(f2 (&V)[32]) {
#pragma unroll
    for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
        for (int k = 0; k < 32; ++k)
            if ((k & h) == 0) {
                const f2 a = V[k], b = V[k + h];
                V[k] = add2(a, b);
                V[k + h] = sub2(a, b);
            }
    }
    const f2 c8 = pk2(0.125f, 0.125f);
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        const float a = lo2(V[k]), b = hi2(V[k]);
        V[k] = mul2(pk2(__fadd_rn(a, b), __fsub_rn(a, b)), c8);
    }
}

// Zero the kept channels (bit k of m0: channel k, of m1: channel k + 32); every other value keeps
// all its bits, the sign of a zero included.  bfe.s32 of one bit gives the all-ones mask of a kept
// channel, which the and-not clears.
__device__ __forceinline__ void keep64(f2 (&V)[32], uint32_t m0, uint32_t m1) {
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        uint32_t a, b, ka, kb2;
        asm("mov.b64 {%0, %1}, %2;" : "=r"(a), "=r"(b) : "l"(V[k]));
        asm("bfe.s32 %0, %1, %2, 1;" : "=r"(ka) : "r"(m0), "r"(k));
        asm("bfe.s32 %0, %1, %2, 1;" : "=r"(kb2) : "r"(m1), "r"(k));
        a &= ~ka;
        b &= ~kb2;
        asm("mov.b64 %0, {%1, %2};" : "=l"(V[k]) : "r"(a), "r"(b));
    }
}

// Scales and codes of one row's block: bm[i] is the maximum of 16-block i (channels 16 i ..
// 16 i + 15); 32 code bytes (element 2j in the low nibble of byte j) and the four scale bytes.
// Codes by the reciprocal-and-bracket argument of e2m1_codes8_r for all 64 values; a lane whose
// brackets straddle a rounding point anywhere (or whose scale is zero or tiny) redoes its block
// with the exact quotients.
__device__ __forceinline__ void codes64(const f2 (&V)[32], const float (&bm)[4], float gsc, float rg, uint32_t (&w)[8],
                                        uint32_t& scales) {
    uint32_t sc[4];
    float d[4], rc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        sc[i] = scale_code<false>(bm[i], gsc, rg);
        d[i] = __fmul_rn(dec_e4m3(sc[i]), gsc);
        rc[i] = __frcp_rn(d[i]);
    }
    scales = sc[0] | (sc[1] << 8) | (sc[2] << 16) | (sc[3] << 24);
    uint32_t bad = fmaxf(fmaxf(rc[0], rc[1]), fmaxf(rc[2], rc[3])) < 3.0e38f ? 0u : 1u;
    const f2 mlo = pk2(0.99999952316284180f, 0.99999952316284180f);
    const f2 mhi = pk2(1.00000047683715820f, 1.00000047683715820f);
    const f2 rA = pk2(rc[0], rc[2]), rB = pk2(rc[1], rc[3]);   // 16-blocks of channels k, k + 32
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const f2 rr = j < 2 ? rA : rB;
        uint32_t lb[4], hb[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int k = 8 * j + 2 * e;
            const f2 q0 = mul2(V[k], rr), q1 = mul2(V[k + 1], rr);
            const f2 l0 = mul2(q0, mlo), l1 = mul2(q1, mlo), h0 = mul2(q0, mhi), h1 = mul2(q1, mhi);
            const uint32_t alo = cvt_e2m1x2(lo2(l0), lo2(l1)), ahi = cvt_e2m1x2(lo2(h0), lo2(h1));
            const uint32_t blo = cvt_e2m1x2(hi2(l0), hi2(l1)), bhi = cvt_e2m1x2(hi2(h0), hi2(h1));
            bad |= (alo ^ ahi) | (blo ^ bhi);
            lb[e] = alo;
            hb[e] = blo;
        }
        w[j] = __byte_perm(__byte_perm(lb[0], lb[1], 0x0040), __byte_perm(lb[2], lb[3], 0x0040), 0x5410);
        w[4 + j] = __byte_perm(__byte_perm(hb[0], hb[1], 0x0040), __byte_perm(hb[2], hb[3], 0x0040), 0x5410);
    }
    if (bad != 0u) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float v[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = i < 2 ? lo2(V[16 * i + e]) : hi2(V[16 * (i - 2) + e]);
            w[2 * i] = d[i] != 0.0f ? e2m1_codes8_r<true>(v, d[i], rc[i]) : 0u;
            w[2 * i + 1] = d[i] != 0.0f ? e2m1_codes8_r<true>(v + 8, d[i], rc[i]) : 0u;
        }
    }
}

// 144 registers a thread: three warps on each SM sub-partition's 16K registers.
template <int R>
__global__ void __maxnreg__(144) quantize_resident_kernel(const __grid_constant__ CUtensorMap tmX, const RParams p) {
    constexpr int NT = R / 8;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw_addr);
    const RLayout lay = make_rlayout(p.W, R, p.p_smem != 0);
    const uint32_t bar_full = base + lay.off_bar;
    const uint32_t bar_const = bar_full + 8u * static_cast<uint32_t>(p.W);
    const uint32_t s_omega = base + lay.off_omega;     // shared-space accesses only (ld/st.shared)
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + lay.off_abort);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int nb = p.nblk;                                   // the CTA owns every block

    griddep_launch_dependents();          // the GEMM may start streaming its weights now
    if (threadIdx.x == 0) {
        for (int i = 0; i < p.W; ++i) mbar_init(bar_full + 8u * i, 1);
        mbar_init(bar_const, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    const int r = lane & 15, b = lane >> 4;
    const int kb0 = 2 * warp;                                // the pair's first block
    const int nblocks = min(2, nb - kb0);
    const int kb = kb0 + b;                                  // this lane's block
    const bool blk_ok = b < nblocks;
    const int nthr = p.W * 32;
    const uint32_t slot = base + static_cast<uint32_t>(warp) * kRSlot;
    const uint32_t box = slot + static_cast<uint32_t>(b) * kRBox;
    const uint32_t invs = p.inv_s ? base + lay.off_invs + 256u * static_cast<uint32_t>(kb) : 0u;
    const uint32_t upart_stride = static_cast<uint32_t>(p.W * NT) * 512u;       // one tile parity
    const uint32_t pf_s = base + lay.off_p + static_cast<uint32_t>(kb0 * NT) * 1024u;
    const bool after = (p.rotate & 3) == 3;

    griddep_wait();                       // x and this grid's outputs belong to the previous grid
    // this pair's boxes of one row tile into the warp's slot
    auto load_tile = [&](int tile) {
        mbar_arrive_expect_tx(bar_full + 8u * warp, nblocks == 2 ? kRSlot : kRBox);
        tma_load_2d(slot, &tmX, kb0 * 64, tile * kRTile, bar_full + 8u * warp);
        if (nblocks == 2) tma_load_2d(slot + kRBox, &tmX, (kb0 + 1) * 64, tile * kRTile, bar_full + 8u * warp);
    };
    if (lane == 0) {
        if (warp == 0) {
            // inv_s, the kept-channel table and P
            const uint32_t pbytes = p.p_smem ? static_cast<uint32_t>(nb * NT) * 1024u : 0u;
            const uint32_t cbytes = (p.inv_s ? 256u * nb : 0u) + (p.n_out ? 16u * nb : 0u) + pbytes;
            mbar_arrive_expect_tx(bar_const, cbytes);
            if (p.inv_s) bulk_load(base + lay.off_invs, p.inv_s, 256u * nb, bar_const);
            if (p.n_out) bulk_load(base + lay.off_omega, p.omega_blk, 16u * nb, bar_const);
            if (pbytes) bulk_load(base + lay.off_p, p.pfrag, pbytes, bar_const);
        }
        tma_prefetch_desc(&tmX);
        if (static_cast<int>(blockIdx.x) < p.row_tiles) load_tile(blockIdx.x);
    }
    bool ok = __all_sync(kRMask, mbar_wait_sleep<false>(bar_const, 0, abort_flag, p.err, 44));
    int issued = static_cast<int>(blockIdx.x) < p.row_tiles ? 0 : -1;  // iteration of the last load issued
    const uint32_t m0 = (p.n_out && blk_ok) ? ld_shared_u32(s_omega + 16u * kb) : 0u;
    const uint32_t m1 = (p.n_out && blk_ok) ? ld_shared_u32(s_omega + 16u * kb + 4u) : 0u;

    int it = 0;
    RT_DECL;
    for (int tile = blockIdx.x; tile < p.row_tiles; tile += gridDim.x, ++it) {
        RT(7);
        RT_TILE();
        const int row = tile * kRTile + r;
        const bool row_ok = row < p.M;
        const uint32_t par = static_cast<uint32_t>(it) & 1u;
        const uint32_t upart_t = base + lay.off_upart + par * upart_stride;     // this tile's partials
        const uint32_t s_amax = base + lay.off_amax + par * static_cast<uint32_t>(4 * kRTile * p.W);
        f2 V[32];
        float bm[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        // ---- pass 1
        if (ok) ok = __all_sync(kRMask, mbar_wait_sleep<false>(bar_full + 8u * warp, par, abort_flag, p.err, 45));
        RT(0);
        if (ok) {
            if constexpr (R > 0) u_pair<NT>(slot, lane, nblocks, p, kb0, pf_s, upart_t + static_cast<uint32_t>(warp * NT) * 512u);
            RT(1);
            if (blk_ok) {
                load_row64(box, r, V);
                if (invs != 0u && !after) smooth64(V, invs);
                if (p.rotate & 1) {
                    fwht64(V);
                    if (invs != 0u && after) smooth64(V, invs);
                }
                if ((m0 | m1) != 0u) {
                    // kept channels: the row's fp16 values into its own (consumed) row of the box,
                    // pair k in 16-byte chunk k / 4 swizzled by the row (chunk ^ r % 8), for the
                    // warp's copy-out below; +0 in the registers
                    const uint32_t rb = box + static_cast<uint32_t>(r) * 128u;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint32_t hw[4];
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const __half2 h2 = __floats2half2_rn(lo2(V[4 * j + t]), hi2(V[4 * j + t]));
                            hw[t] = *reinterpret_cast<const uint32_t*>(&h2);
                        }
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                                     :: "r"(rb + 16u * (static_cast<uint32_t>(j) ^ (static_cast<uint32_t>(r) & 7u))),
                                        "r"(hw[0]), "r"(hw[1]), "r"(hw[2]), "r"(hw[3]) : "memory");
                    }
                    keep64(V, m0, m1);
                }
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    bm[0] = fmaxf(bm[0], fabsf(lo2(V[k])));
                    bm[1] = fmaxf(bm[1], fabsf(lo2(V[16 + k])));
                    bm[2] = fmaxf(bm[2], fabsf(hi2(V[k])));
                    bm[3] = fmaxf(bm[3], fabsf(hi2(V[16 + k])));
                }
            }
            if (p.n_out) {
                // the kept channels of the pair's blocks out to x_O by the whole warp: lane l takes
                // channels l and l + 32 of a block (the pair at 4 l of each row) for its 16 rows,
                // so a block with many kept channels costs its warp a few row sweeps and the
                // stores of a row are contiguous
                __syncwarp();
                bool wrote = false;
                for (int bb = 0; bb < nblocks; ++bb) {
                    const uint32_t om = s_omega + 16u * static_cast<uint32_t>(kb0 + bb);
                    const uint32_t mb0 = ld_shared_u32(om), mb1 = ld_shared_u32(om + 4u);
                    if ((mb0 | mb1) == 0u) continue;
                    wrote = true;
                    const uint32_t below = (1u << lane) - 1u;
                    const bool k0 = (mb0 >> lane) & 1u, k1 = (mb1 >> lane) & 1u;
                    const uint32_t i0 = ld_shared_u32(om + 8u) + static_cast<uint32_t>(__popc(mb0 & below));
                    const uint32_t i1 = ld_shared_u32(om + 8u) + static_cast<uint32_t>(__popc(mb0) + __popc(mb1 & below));
                    const uint32_t bx = slot + static_cast<uint32_t>(bb) * kRBox + 4u * (static_cast<uint32_t>(lane) & 3u);
                    if (k0 || k1) {
#pragma unroll 4
                        for (int rr = 0; rr < kRTile; ++rr) {
                            const int rw = tile * kRTile + rr;
                            const uint32_t a = bx + static_cast<uint32_t>(rr) * 128u +
                                               16u * ((static_cast<uint32_t>(lane) >> 2) ^ (static_cast<uint32_t>(rr) & 7u));
                            const uint32_t hv = ld_shared_u32(a);
                            if (rw < p.M) {
                                uint16_t* xr = p.xo + static_cast<size_t>(rw) * p.xo_ld;
                                if (k0) xr[i0] = static_cast<uint16_t>(hv & 0xFFFFu);
                                if (k1) xr[i1] = static_cast<uint16_t>(hv >> 16);
                            }
                        }
                    }
                }
                if (wrote) fence_proxy_async_smem();   // the scratch precedes the next tile's TMA into the slot
            }
            __syncwarp();                 // the slot is read: the next tile's boxes may land in it
            if (lane == 0 && tile + static_cast<int>(gridDim.x) < p.row_tiles) load_tile(tile + gridDim.x);
            if (tile + static_cast<int>(gridDim.x) < p.row_tiles) issued = it + 1;
        }
        // ---- exchange: the row maximum and U over the warps (warp order)
        float amax = fmaxf(fmaxf(bm[0], bm[1]), fmaxf(bm[2], bm[3]));
        amax = fmaxf(amax, __shfl_xor_sync(kRMask, amax, 16));
        if (b == 0) st_shared_f32(s_amax + 4u * static_cast<uint32_t>(warp * kRTile + r), amax);
        RT(2);
        named_bar_sync(1, nthr);
        RT(3);
        amax = 0.0f;
        {
            // every warp's maximum of the row requested before any is used
            float wm[kMaxPairs];
#pragma unroll
            for (int w = 0; w < kMaxPairs; ++w)
                wm[w] = w < p.W ? ld_shared_f32(s_amax + 4u * static_cast<uint32_t>(w * kRTile + r)) : 0.0f;
#pragma unroll
            for (int w = 0; w < kMaxPairs; ++w) amax = fmaxf(amax, wm[w]);
        }
        RT(6);
        if constexpr (R > 0) {
            // pairs of U sums (row rr, columns cc and cc + 1) over the CTA's threads, each summed
            // over the warps' partials in warp order
            for (int pi = static_cast<int>(threadIdx.x); pi < NT * 64; pi += nthr) {
                const uint32_t off = 8u * static_cast<uint32_t>(pi);
                float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
                for (int w = 0; w < kMaxPairs; ++w)
                    if (w < p.W) {
                        const float2 v = ld_shared_v2f(upart_t + static_cast<uint32_t>(w * NT) * 512u + off);
                        s0 = __fadd_rn(s0, v.x);
                        s1 = __fadd_rn(s1, v.y);
                    }
                int rr, cc;
                frag_pos(2 * pi, rr, cc);
                const int rg = tile * kRTile + rr;
                if (rg < p.M) {
                    const __nv_bfloat162 h = __floats2bfloat162_rn(s0, s1);
                    *reinterpret_cast<uint32_t*>(p.u + static_cast<size_t>(rg) * R + cc) = *reinterpret_cast<const uint32_t*>(&h);
                }
            }
        }
        RT(4);
        const float gsc = __fdiv_rn(amax, 2688.0f);
        const float rg_inv = __frcp_rn(gsc);
        RT(7);
        if (warp == 0 && b == 0 && row_ok) p.g[row] = gsc;
        if (p.n_out && p.xo_ld > p.n_out) {
            // x_O's columns beyond the kept channels are zero
            const int pad = p.xo_ld - p.n_out;
            for (int i = threadIdx.x; i < kRTile * pad; i += nthr) {
                const int rw = tile * kRTile + i / pad;
                if (rw < p.M) p.xo[static_cast<size_t>(rw) * p.xo_ld + p.n_out + i % pad] = 0;
            }
        }
        // ---- pass 2
        if (ok && blk_ok) {
            uint32_t w[8], scales;
            codes64(V, bm, gsc, rg_inv, w, scales);
            if (row_ok) {
                const int K = p.K;
                uint4* dst = reinterpret_cast<uint4*>(p.codes + static_cast<size_t>(row) * (K / 2) + kb * 32);
                dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                size_t off;
                if (p.sf_layout == WQ_SCALE_LAYOUT_MMA)
                    off = (static_cast<size_t>(row / kBlockM) * (K / 64) + kb) * kSfAtom + (row % 32) * 16 +
                          ((row % kBlockM) / 32) * 4;
                else
                    off = static_cast<size_t>(row) * (K / 16) + kb * 4;
                *reinterpret_cast<uint32_t*>(p.sf + off) = scales;
            }
        }
        RT(5);
    }
    RT_FLUSH();
    // every copy this warp issued has landed before the CTA can finish
    if (issued >= 0) mbar_wait_sleep<false>(bar_full + 8u * warp, static_cast<uint32_t>(issued) & 1u, abort_flag, p.err, 47);
}

struct RPlan {
    int W = 0;
    bool p_smem = false;
    uint32_t smem = 0;
};

// Every pair of the row on one CTA of W <= kMaxPairs warps (K <= 1536).
bool resident_plan(int K, int R, RPlan& pl) {
    const int nblk = K / 64, npairs = (nblk + 1) / 2;
    if (npairs < 1 || npairs > kMaxPairs) return false;
    pl.W = npairs;
    pl.p_smem = R > 0 && make_rlayout(pl.W, R, true).total <= kSmemBudget;
    pl.smem = make_rlayout(pl.W, R, pl.p_smem).total;
    return pl.smem <= kSmemBudget;
}

template <int R>
cudaError_t launch_rr(const CUtensorMap& tm, const RParams& rp, const RPlan& pl, int num_sms, cudaStream_t st) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(quantize_resident_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(kSmemBudget));
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(quantize_resident_kernel<R>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                            cudaSharedmemCarveoutMaxShared);
    });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(rp.row_tiles < num_sms ? rp.row_tiles : num_sms));
    cfg.blockDim = dim3(static_cast<unsigned>(pl.W * 32));
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, quantize_resident_kernel<R>, tm, rp);
}

}  // namespace

bool quant_resident_eligible(const QuantArgs& a) {
    if (a.int8 || a.act_scale != WQ_ACT_SCALE_ROW || a.vt != nullptr || (a.inv_s != nullptr && a.inv_s_rr == nullptr))
        return false;
    if (a.r != 0 && a.r != 16 && a.r != 32 && a.r != 64) return false;
    RPlan pl;
    return resident_plan(a.K, a.r, pl);
}

cudaError_t launch_quantize_resident(const QuantArgs& a, cudaStream_t st) {
    if (a.M <= 0) return cudaSuccess;
    RPlan pl;
    if (!resident_plan(a.K, a.r, pl)) return cudaErrorInvalidValue;
    RParams rp{};
    rp.M = a.M;
    rp.K = a.K;
    rp.nblk = a.K / 64;
    rp.npairs = (rp.nblk + 1) / 2;
    rp.W = pl.W;
    rp.row_tiles = (a.M + kRTile - 1) / kRTile;
    rp.inv_s = a.inv_s_rr;
    rp.rotate = a.rotate;
    rp.omega_blk = a.omega_blk;
    rp.n_out = a.n_out;
    rp.xo_ld = a.xo_ld > a.n_out ? a.xo_ld : a.n_out;
    rp.xo = a.xo;
    rp.pfrag = a.pfrag;
    rp.p_smem = pl.p_smem ? 1 : 0;
    rp.u = a.u;
    rp.codes = a.codes;
    rp.sf = a.sf;
    rp.sf_layout = a.sf_layout;
    rp.g = a.g;
    rp.err = a.err;
    switch (a.r) {
        case 0: return launch_rr<0>(*a.tmX, rp, pl, a.num_sms, st);
        case 16: return launch_rr<16>(*a.tmX, rp, pl, a.num_sms, st);
        case 32: return launch_rr<32>(*a.tmX, rp, pl, a.num_sms, st);
        case 64: return launch_rr<64>(*a.tmX, rp, pl, a.num_sms, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace wq
