// wq_quant.cu -- fused activation transform + NVFP4 quantiser (x is read from HBM once).
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
// change a bit.
//
// A CTA owns a tile of 32 rows and a range of at most kMaxBlocks 64-column blocks of K (the
// K range of a row tile is split over a thread-block cluster when K is long or the batch is
// small).  Warp 8 streams the tile's blocks into shared memory with TMA (one 4 KiB,
// 128-byte-swizzled box per block, each loaded once, into a 9 KiB slot).  Warps 0-7 make two
// passes over the resident blocks.  Pass 1: the raw bf16 block feeds ldmatrix + mma.sync for
// U; each thread (one row x 8 channels) smooths its channels and runs FWHT strides 1,2,4 in
// registers, the block is transposed through its slot (fp32, rows padded to 72 words so both
// orders are bank-conflict free) for strides 8,16,32, and the transformed fp32 block is left
// in the slot; the row amax is accumulated.  Pass 2 reads the transformed blocks back and
// writes the codes, scales and outlier values.  Across a cluster the row amax and the U
// partial sums are combined through distributed shared memory.
//
// kInt8 = true is the selective 8-bit variant (FoldQuantVLA, Key Contribution 3) in the same
// basis: a = amax / 127 per row, q = round-half-even(xt / a) clamped to [-127, 127], written as
// exact bf16 integers [M, K] for the 8-bit GEMM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdlib>

#include "ptx.cuh"
#include "quant_math.cuh"
#include "wq_internal.h"

#ifdef WQ_TRACE
// Timeline probes for kernel development builds only (never defined in the product build).
__device__ unsigned long long g_wq_qtrace[4096 * 8];
#define WQ_QTRACE_AT(slot) (g_wq_qtrace[blockIdx.x * 8 + (slot)] = wq::global_timer_ns())
extern "C" WQ_API int wq_qtrace_read(void* host, size_t bytes) {
    return static_cast<int>(cudaMemcpyFromSymbol(host, g_wq_qtrace, bytes));
}
#else
#define WQ_QTRACE_AT(slot) ((void)0)
#endif

namespace wq {
namespace {

constexpr int kRows = 32;                 // rows per tile
constexpr int kConsumerWarps = 8;         // 32 rows x 8 chunks = 256 threads
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr uint32_t kBlockBytes = kRows * 128;          // one TMA box: 32 rows x 64 bf16
constexpr uint32_t kRowWords = 72;                      // fp32 row stride of a slot (64 + 8 pad)
constexpr uint32_t kSlotBytes = 9216;                   // 32 x 72 x 4, a multiple of 1024
constexpr int kTargetBlocks = 8;          // blocks per CTA aimed for (74 KiB: three CTAs per SM)
constexpr int kMaxBlocks = 20;
constexpr unsigned kFullMask = 0xFFFFFFFFu;

struct QParams {
    int M, K;
    int nblk;           // 64-column blocks of K
    int csplit;         // CTAs per row tile (cluster size)
    int max_nb;         // largest block count of one CTA
    int row_tiles;
    const float* inv_s;
    int rotate;
    const int16_t* omega_pos;
    int n_out;
    uint16_t* xo;
    const uint32_t* pfrag;   // low-rank factor P in mma.sync B-fragment order
    uint16_t* u;
    uint8_t* codes;
    uint8_t* sf;
    int sf_layout;
    float* g;
    int* err;
};

struct Layout {
    uint32_t off_invs, off_opos, off_bar, off_amax, off_u, off_abort, total;
};

__host__ __device__ inline Layout make_layout(int max_nb, int r) {
    Layout l{};
    l.off_invs = static_cast<uint32_t>(max_nb) * kSlotBytes;            // inv_s slice, 256 B per block
    l.off_opos = l.off_invs + 256u * static_cast<uint32_t>(max_nb);    // Omega slot slice, 128 B per block
    l.off_bar = l.off_opos + 128u * static_cast<uint32_t>(max_nb);
    l.off_amax = l.off_bar + 8u * static_cast<uint32_t>(max_nb + 1);
    l.off_amax = (l.off_amax + 15u) & ~15u;
    l.off_u = l.off_amax + 4u * kRows;
    l.off_abort = l.off_u + 4u * kRows * static_cast<uint32_t>(r > 0 ? r : 1);
    l.total = l.off_abort + 16u + 1024u;
    return l;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& raw, float (&f)[8]) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// Smoothing and FWHT strides 1, 2, 4 of this thread's 8 channels (s_invs: their 8 entries of
// the shared-memory copy of inv_s).
__device__ __forceinline__ void transform_low(const uint4& raw, const float* s_invs, const QParams& p, float (&v)[8]) {
    bf16x8_to_f32(raw, v);
    if (p.inv_s != nullptr) {
        const float4* sp = reinterpret_cast<const float4*>(s_invs);
        const float4 s0 = sp[0], s1 = sp[1];
        const float s[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = __fmul_rn(v[e], s[e]);
    }
    if (p.rotate) {
#pragma unroll
        for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if ((e & h) == 0) {
                    const float a = v[e], b = v[e + h];
                    v[e] = __fadd_rn(a, b);
                    v[e + h] = __fsub_rn(a, b);
                }
        }
    }
}

// FWHT strides 8, 16, 32 and the 1/8 scale, on the 8 channels c, c+8, ..., c+56 of a row
// (the partner of channel c + 8j at stride 8h is channel c + 8 (j ^ h)).
__device__ __forceinline__ void transform_high(float (&w)[8]) {
#pragma unroll
    for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if ((j & h) == 0) {
                const float a = w[j], b = w[j + h];
                w[j] = __fadd_rn(a, b);
                w[j + h] = __fsub_rn(a, b);
            }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = __fmul_rn(w[j], 0.125f);
}

__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
    asm volatile("st.shared.f32 [%0], %1;" :: "r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void ld_shared_v8f(uint32_t addr, float (&v)[8]) {
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]) : "r"(addr) : "memory");
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7]) : "r"(addr + 16u) : "memory");
}

// zero the kept channels; in pass 2 also store their fp16 values (s_opos: the 8 slot entries)
__device__ __forceinline__ void split_outliers(float (&v)[8], const int16_t* s_opos, int row, bool store,
                                               const QParams& p) {
    const uint4 pw = *reinterpret_cast<const uint4*>(s_opos);
    const uint32_t w[4] = {pw.x, pw.y, pw.z, pw.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const int pos = static_cast<int16_t>((w[e / 2] >> (16 * (e & 1))) & 0xFFFFu);
        if (pos >= 0) {
            if (store) p.xo[static_cast<size_t>(row) * p.n_out + pos] = __half_as_ushort(__float2half_rn(v[e]));
            v[e] = 0.0f;
        }
    }
}

template <int R, bool kInt8>
__global__ void __launch_bounds__(kThreads) quantize_kernel(const __grid_constant__ CUtensorMap tmX, const QParams p) {
    constexpr int NT = R / 8 > 0 ? R / 8 : 1;       // n8 tiles of U
    constexpr int NTW = NT > 4 ? NT / 4 : 1;        // n-tiles per warp
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw_addr);
    const Layout lay = make_layout(p.max_nb, R);
    const uint32_t bar_full = base + lay.off_bar;
    const uint32_t bar_const = bar_full + 8u * static_cast<uint32_t>(p.max_nb);
    const float* s_invs = reinterpret_cast<const float*>(base_ptr + lay.off_invs);
    const int16_t* s_opos = reinterpret_cast<const int16_t*>(base_ptr + lay.off_opos);
    float* s_amax = reinterpret_cast<float*>(base_ptr + lay.off_amax);
    float* s_u = reinterpret_cast<float*>(base_ptr + lay.off_u);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + lay.off_abort);

    griddep_launch_dependents();          // the GEMM may start streaming its weights now

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const bool clustered = p.csplit > 1;
    const uint32_t rank = clustered ? cluster_ctarank() : 0u;
    const int tile = clustered ? static_cast<int>(blockIdx.x) / p.csplit : static_cast<int>(blockIdx.x);
    const int kb_lo = static_cast<int>(rank) * p.nblk / p.csplit;
    const int nb = (static_cast<int>(rank) + 1) * p.nblk / p.csplit - kb_lo;
    const int K = p.K;

    if (threadIdx.x == 0) {
        WQ_QTRACE_AT(0);
        for (int i = 0; i < nb; ++i) mbar_init(bar_full + 8u * i, 1);
        mbar_init(bar_const, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ TMA producer
        if (clustered) cluster_arrive();   // nothing of this warp is read across the cluster
        if (lane == 0) {
            tma_prefetch_desc(&tmX);
            griddep_wait();                // x and this grid's outputs belong to the previous grid
            // this CTA's slices of inv_s and of the Omega slot table
            const uint32_t cbytes = (p.inv_s ? 256u * nb : 0u) + (p.n_out ? 128u * nb : 0u);
            mbar_arrive_expect_tx(bar_const, cbytes);
            if (p.inv_s) bulk_load(base + lay.off_invs, p.inv_s + kb_lo * 64, 256u * nb, bar_const);
            if (p.n_out) bulk_load(base + lay.off_opos, p.omega_pos + kb_lo * 64, 128u * nb, bar_const);
            for (int i = 0; i < nb; ++i) {
                const uint32_t fb = bar_full + 8u * i;
                mbar_arrive_expect_tx(fb, kBlockBytes);
                tma_load_2d(base + static_cast<uint32_t>(i) * kSlotBytes, &tmX, (kb_lo + i) * 64, tile * kRows, fb);
            }
            WQ_QTRACE_AT(1);
            // every copy has landed before this CTA can finish
            for (int i = 0; i < nb; ++i) mbar_wait(bar_full + 8u * i, 0, abort_flag, p.err, 11);
            mbar_wait(bar_const, 0, abort_flag, p.err, 13);
        }
        __syncwarp();
        if (clustered) {
            cluster_wait();
            cluster_arrive();
            cluster_wait();
        }
        return;
    }

    // ---------------------------------------------------------------- consumers (warps 0-7)
    const int rloc = warp * 4 + (lane >> 3);            // row of the tile
    const int c = lane & 7;                              // chunk of the block
    const int row = tile * kRows + rloc;
    const bool row_ok = row < p.M;
    const uint32_t my_off = static_cast<uint32_t>(rloc) * 128u + ((static_cast<uint32_t>(c) ^ (rloc & 7u)) << 4);

    // pass 1: row amax and the low-rank projection
    float amax = 0.0f;
    float uacc[NTW][4];
#pragma unroll
    for (int j = 0; j < NTW; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) uacc[j][e] = 0.0f;
    const int mt = warp & 1;                             // 16-row half of the tile for mma
    bool ok = mbar_wait(bar_const, 0, abort_flag, p.err, 14);
    // low-rank B fragments, prefetched one block ahead
    uint4 bq[NTW][2];
    auto load_bq = [&](int kb) {
        if constexpr (R > 0) {
#pragma unroll
            for (int j = 0; j < NTW; ++j) {
                const int nt = (warp >> 1) + 4 * j;
                if (nt < NT) {
                    const uint4* pb = reinterpret_cast<const uint4*>(
                        p.pfrag + (static_cast<size_t>(kb * NT + nt) * 32 + lane) * 8);
                    bq[j][0] = __ldg(pb);
                    bq[j][1] = __ldg(pb + 1);
                }
            }
        }
    };
    load_bq(kb_lo);
    for (int i = 0; ok && i < nb; ++i) {
        if (!mbar_wait(bar_full + 8u * i, 0, abort_flag, p.err, 12)) { ok = false; break; }
        if (i == 0 && threadIdx.x == 0) WQ_QTRACE_AT(2);
        const uint32_t blk = base + static_cast<uint32_t>(i) * kSlotBytes;
        const int kb = kb_lo + i;
        if constexpr (R > 0) {
            uint4 bcur[NTW][2];
#pragma unroll
            for (int j = 0; j < NTW; ++j) {
                bcur[j][0] = bq[j][0];
                bcur[j][1] = bq[j][1];
            }
            if (i + 1 < nb) load_bq(kb + 1);
            // each 64-column block is accumulated on the tensor cores from zero and then added
            // to the running sum with an fp32 add, so the tensor-core accumulation depth stays
            // at 64 products whatever K is
            float blk_acc[NTW][4];
#pragma unroll
            for (int j = 0; j < NTW; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) blk_acc[j][e] = 0.0f;
            const uint32_t arow = static_cast<uint32_t>(16 * mt + (lane & 7) + 8 * ((lane >> 3) & 1));
#pragma unroll
            for (int f = 0; f < 4; ++f) {
                const uint32_t chunk = static_cast<uint32_t>(2 * f + (lane >> 4));
                uint32_t a0, a1, a2, a3;
                ldmatrix_x4(blk + arow * 128u + ((chunk ^ (arow & 7u)) << 4), a0, a1, a2, a3);
#pragma unroll
                for (int j = 0; j < NTW; ++j) {
                    const int nt = (warp >> 1) + 4 * j;
                    if (nt < NT) {
                        const uint4& q = bcur[j][f >> 1];
                        const uint32_t b0 = (f & 1) ? q.z : q.x;
                        const uint32_t b1 = (f & 1) ? q.w : q.y;
                        mma_bf16_16816(blk_acc[j], a0, a1, a2, a3, b0, b1);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < NTW; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) uacc[j][e] = __fadd_rn(uacc[j][e], blk_acc[j][e]);
        }
        const uint4 raw = ld_shared_v4(blk + my_off);
        // every warp has read the slot's bf16 rows before any warp writes fp32 rows over them
        // (fp32 row r spans the bytes of bf16 rows 2.25 r .. 2.25 r + 2, owned by other warps)
        named_bar_sync(1, kConsumerWarps * 32);
        float v[8];
        transform_low(raw, s_invs + i * 64 + c * 8, p, v);
        const uint32_t rowb = blk + static_cast<uint32_t>(rloc) * (kRowWords * 4u);
        if (p.rotate) {
            // transpose through the slot: write channels 8c..8c+7, read c, c+8, ..., c+56
            st_shared_v4f(rowb + c * 32u, v[0], v[1], v[2], v[3]);
            st_shared_v4f(rowb + c * 32u + 16u, v[4], v[5], v[6], v[7]);
            __syncwarp();
            float w[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) w[j] = ld_shared_f32(rowb + (c + 8u * j) * 4u);
            transform_high(w);
#pragma unroll
            for (int j = 0; j < 8; ++j) st_shared_f32(rowb + (c + 8u * j) * 4u, w[j]);
            if (p.n_out == 0) {
#pragma unroll
                for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(w[j]));
            } else {
                __syncwarp();
                ld_shared_v8f(rowb + c * 32u, v);
            }
        } else {
            st_shared_v4f(rowb + c * 32u, v[0], v[1], v[2], v[3]);
            st_shared_v4f(rowb + c * 32u + 16u, v[4], v[5], v[6], v[7]);
        }
        if (!p.rotate || p.n_out > 0) {
            if (p.n_out > 0) split_outliers(v, s_opos + i * 64 + c * 8, row, false, p);
#pragma unroll
            for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(v[e]));
        }
    }
    __syncwarp();
    amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 4));
    if (threadIdx.x == 0) WQ_QTRACE_AT(3);

    const int gq = lane >> 2, cq = lane & 3;             // mma fragment row / column pair
    if (clustered) {
        if (c == 0) s_amax[rloc] = amax;
        if constexpr (R > 0) {
#pragma unroll
            for (int j = 0; j < NTW; ++j) {
                const int nt = (warp >> 1) + 4 * j;
                if (nt < NT) {
                    const int col = 8 * nt + 2 * cq;
                    s_u[(16 * mt + gq) * R + col] = uacc[j][0];
                    s_u[(16 * mt + gq) * R + col + 1] = uacc[j][1];
                    s_u[(16 * mt + gq + 8) * R + col] = uacc[j][2];
                    s_u[(16 * mt + gq + 8) * R + col + 1] = uacc[j][3];
                }
            }
        }
        cluster_arrive();
        cluster_wait();
        float a = 0.0f;
        const uint32_t la = smem_u32(s_amax + rloc);
        for (int qr = 0; qr < p.csplit; ++qr) a = fmaxf(a, ld_dsmem_f32(mapa_shared(la, static_cast<uint32_t>(qr))));
        amax = a;
        if constexpr (R > 0) {
            // every rank reduces an interleaved share of the tile's U entries
            {
                for (int idx = threadIdx.x * p.csplit + static_cast<int>(rank); idx < kRows * R;
                     idx += kConsumerWarps * 32 * p.csplit) {
                    const int rr = idx / R, cc = idx % R;
                    const uint32_t la2 = smem_u32(s_u + idx);
                    float sum = 0.0f;
                    for (int qr = 0; qr < p.csplit; ++qr) sum += ld_dsmem_f32(mapa_shared(la2, static_cast<uint32_t>(qr)));
                    const int rg = tile * kRows + rr;
                    if (rg < p.M) p.u[static_cast<size_t>(rg) * R + cc] = __bfloat16_as_ushort(__float2bfloat16_rn(sum));
                }
            }
        }
    } else if constexpr (R > 0) {
#pragma unroll
        for (int j = 0; j < NTW; ++j) {
            const int nt = (warp >> 1) + 4 * j;
            if (nt < NT) {
                const int col = 8 * nt + 2 * cq;
                const int r0 = tile * kRows + 16 * mt + gq, r1 = r0 + 8;
                if (r0 < p.M)
                    *reinterpret_cast<__nv_bfloat162*>(p.u + static_cast<size_t>(r0) * R + col) =
                        __floats2bfloat162_rn(uacc[j][0], uacc[j][1]);
                if (r1 < p.M)
                    *reinterpret_cast<__nv_bfloat162*>(p.u + static_cast<size_t>(r1) * R + col) =
                        __floats2bfloat162_rn(uacc[j][2], uacc[j][3]);
            }
        }
    }
    const float gsc = __fdiv_rn(amax, kInt8 ? 127.0f : 2688.0f);
    if (threadIdx.x == 0) WQ_QTRACE_AT(4);
    if (rank == 0 && c == 0 && row_ok) p.g[row] = gsc;

    // pass 2: codes, scales and the kept channels, from the resident blocks
    for (int i = 0; ok && i < nb; ++i) {
        const uint32_t blk = base + static_cast<uint32_t>(i) * kSlotBytes;
        const int kb = kb_lo + i;
        float v[8];
        ld_shared_v8f(blk + static_cast<uint32_t>(rloc) * (kRowWords * 4u) + c * 32u, v);
        if (p.n_out > 0) split_outliers(v, s_opos + i * 64 + c * 8, row, row_ok, p);
        if constexpr (kInt8) {
            uint32_t pk[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float t[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float r = gsc != 0.0f ? rintf(__fdiv_rn(v[2 * q + e], gsc)) : 0.0f;
                    t[e] = fminf(fmaxf(r, -127.0f), 127.0f);
                }
                const __nv_bfloat162 h = __floats2bfloat162_rn(t[0], t[1]);
                pk[q] = *reinterpret_cast<const uint32_t*>(&h);
            }
            if (row_ok)
                *reinterpret_cast<uint4*>(p.codes + (static_cast<size_t>(row) * K + kb * 64 + c * 8) * 2) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
            continue;
        }
        float cm = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) cm = fmaxf(cm, fabsf(v[e]));
        const float bm = fmaxf(cm, __shfl_xor_sync(kFullMask, cm, 1));
        uint32_t sc = 0;
        if (gsc != 0.0f) sc = cvt_e4m3(__fdiv_rn(__fdiv_rn(bm, 6.0f), gsc));
        const float d = __fmul_rn(dec_e4m3(sc), gsc);
        const uint32_t word = d != 0.0f ? e2m1_codes8(v, d) : 0u;
        if (row_ok) *reinterpret_cast<uint32_t*>(p.codes + static_cast<size_t>(row) * (K / 2) + kb * 32 + 4 * c) = word;
        const uint32_t s1 = __shfl_down_sync(kFullMask, sc, 2);
        const uint32_t s2 = __shfl_down_sync(kFullMask, sc, 4);
        const uint32_t s3 = __shfl_down_sync(kFullMask, sc, 6);
        if (row_ok && c == 0) {
            const uint32_t w4 = sc | (s1 << 8) | (s2 << 16) | (s3 << 24);
            size_t off;
            if (p.sf_layout == WQ_SCALE_LAYOUT_MMA)
                off = (static_cast<size_t>(row / kBlockM) * (K / 64) + kb) * kSfAtom + (row % 32) * 16 +
                      ((row % kBlockM) / 32) * 4;
            else
                off = static_cast<size_t>(row) * (K / 16) + kb * 4;
            *reinterpret_cast<uint32_t*>(p.sf + off) = w4;
        }
    }
    if (threadIdx.x == 0) WQ_QTRACE_AT(5);
    if (clustered) {
        cluster_arrive();                 // peers are done reading this CTA's s_amax / s_u
        cluster_wait();
    }
    if (threadIdx.x == 0) WQ_QTRACE_AT(6);
}

struct Choice {
    int csplit, max_nb;
};

Choice choose(int M, int K, int num_sms) {
    const int nblk = K / 64;
    const int row_tiles = (M + kRows - 1) / kRows;
    int cs = 1;
    while (cs < 16 && (nblk + cs - 1) / cs > kTargetBlocks) cs <<= 1;
    // small batches: spread a row tile's K range over more CTAs
    while (cs < 16 && row_tiles * cs * 2 <= num_sms && nblk >= 2 * cs) cs <<= 1;
    if (cs > nblk) cs = nblk;
    return Choice{cs, (nblk + cs - 1) / cs};
}

template <int R, bool kInt8>
cudaError_t launch_r(const CUtensorMap& tm, const QParams& qp, cudaStream_t st) {
    const Layout lay = make_layout(qp.max_nb, R);
    static bool attr_set = false;
    if (!attr_set) {
        const Layout worst = make_layout(kMaxBlocks, R);
        cudaError_t e = cudaFuncSetAttribute(quantize_kernel<R, kInt8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(worst.total));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(quantize_kernel<R, kInt8>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(qp.row_tiles * qp.csplit));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = lay.total;
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    int na = 0;
    at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (qp.csplit > 1) {
        at[na].id = cudaLaunchAttributeClusterDimension;
        at[na].val.clusterDim.x = static_cast<unsigned>(qp.csplit);
        at[na].val.clusterDim.y = 1;
        at[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = at;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, quantize_kernel<R, kInt8>, tm, qp);
}

}  // namespace

cudaError_t launch_quantize_act(const QuantArgs& a, cudaStream_t st) {
    if (a.M <= 0) return cudaSuccess;
    Choice ch = choose(a.M, a.K, a.num_sms);
    // WQ_QUANT_SPLIT=<n> pins the CTAs per row tile (tuning and tests)
    if (const char* fs = std::getenv("WQ_QUANT_SPLIT")) {
        const int v = std::atoi(fs);
        const int nblk = a.K / 64;
        if (v >= 1 && v <= 16 && (v & (v - 1)) == 0 && v <= nblk && (nblk + v - 1) / v <= kMaxBlocks)
            ch = Choice{v, (nblk + v - 1) / v};
    }
    if (ch.max_nb > kMaxBlocks) return cudaErrorInvalidValue;
    QParams qp{};
    qp.M = a.M; qp.K = a.K; qp.nblk = a.K / 64; qp.csplit = ch.csplit; qp.max_nb = ch.max_nb;
    qp.row_tiles = (a.M + kRows - 1) / kRows;
    qp.inv_s = a.inv_s; qp.rotate = a.rotate; qp.omega_pos = a.omega_pos; qp.n_out = a.n_out; qp.xo = a.xo;
    qp.pfrag = a.pfrag; qp.u = a.u; qp.codes = a.codes; qp.sf = a.sf; qp.sf_layout = a.sf_layout; qp.g = a.g;
    qp.err = a.err;
    if (a.int8) return a.r == 0 && a.n_out == 0 ? launch_r<0, true>(*a.tmX, qp, st) : cudaErrorInvalidValue;
    switch (a.r) {
        case 0: return launch_r<0, false>(*a.tmX, qp, st);
        case 16: return launch_r<16, false>(*a.tmX, qp, st);
        case 32: return launch_r<32, false>(*a.tmX, qp, st);
        case 64: return launch_r<64, false>(*a.tmX, qp, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace wq
