// wq_quant.cu -- fused activation transform + NVFP4 quantiser: the cluster and stream schedules
// (the register-resident schedule for K <= 1536 is in wq_quant_rr.cu).
//
// Per activation row (FoldQuantVLA, Key Contribution 2: channel scaling, block Hadamard
// via the FWHT with beta = 64, dynamic per-token quantisation; QuantWAMs sec. 3.1 Eq. (1):
// the quantiser sees x R S^-1 and the Top-K channels of that basis stay in FP16):
//   xs   = fp32(x) * inv_s                       (one fp32 multiply)
//   xt   = FWHT64(xs) per 64-block, then * 1/8   (Sylvester order, strides 1..32)
//   x_O  = fp16(xt[O]); xt[O] = 0                (outlier split)
//   g    = amax(|xt|) / 2688                     (fp32 tensor scale of the row)
//   sc_b = e4m3((bmax_b / 6) / g), d_b = dec(sc_b) * g, code = e2m1(xt / d_b)
//   U    = bf16(x P)                             (16-bit low-rank down-projection, Q-WAM ASP)
// Every rounding step is an explicit _rn intrinsic so no multiply-add contraction can
// change a bit.
//
// Rows go in tiles of 16, 64-column blocks of K as 2 KiB TMA boxes (128-byte swizzle).  In a
// warp, lane l owns row l % 16 and half l / 16 of a block (32 channels): FWHT strides 1..16
// run in its registers, stride 32 is one shuffle with lane l ^ 16.  Each block goes through
//   pass 1: smoothing, FWHT, the kept channels (fp16 values out), the 16-element maxima
//           without them, the row amax; the block's share of U (mma.sync on the raw box,
//           every n-tile of P) is added to the warp's partial in shared memory;
//   pass 2: e4m3 scales and e2m1 codes (16 bytes per lane; a row's 32 bytes of a block form
//           one sector), after the row amax of the whole row is known.
// Two schedules:
//   cluster (few rows): a CTA owns one row tile and a K range of at most 16 blocks (the K
//           range of a tile is spread over a thread-block cluster); warp 8 loads every block
//           once, the transformed fp32 block waits in its slot between the passes, and the
//           row amax and U partials are combined through distributed shared memory;
//   stream (many rows): persistent CTAs walk row tiles; warp 8 streams every block of a
//           tile twice through a ring of shared-memory slots (the second time from L2), and
//           pass 2 recomputes the transform instead of keeping it.
//
// kInt8 = true is the selective 8-bit variant (FoldQuantVLA, Key Contribution 3) in the same
// basis: a = amax / 127 per row, q = round-half-even(xt / a) clamped to [-127, 127], written as
// exact bf16 integers [M, K] for the 8-bit GEMM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdlib>

#include "ptx.cuh"
#include "quant_block.cuh"
#include "quant_math.cuh"
#include "wq_internal.h"

#ifdef WQ_TRACE
// Timeline probes for kernel development builds only (never defined in the product build).
__device__ unsigned long long g_wq_qtrace[8192 * 8];
#define WQ_QTRACE_AT(slot) do { if (blockIdx.x < 8192) g_wq_qtrace[blockIdx.x * 8 + (slot)] = wq::global_timer_ns(); } while (0)
extern "C" WQ_API int wq_qtrace_read(void* host, size_t bytes) {
    return static_cast<int>(cudaMemcpyFromSymbol(host, g_wq_qtrace, bytes));
}
__device__ unsigned long long g_wq_qphase[16];
extern "C" WQ_API int wq_qphase_read(void* host, size_t bytes) {
    return static_cast<int>(cudaMemcpyFromSymbol(host, g_wq_qphase, bytes));
}
#define QPH_DECL unsigned long long qph_[8] = {0, 0, 0, 0, 0, 0, 0, 0}; long long qpt_ = clock64()
#define QPH(i) do { const long long n_ = clock64(); qph_[i] += n_ - qpt_; qpt_ = n_; } while (0)
#define QPH_FLUSH do { if (lane == 0) { for (int i_ = 0; i_ < 8; ++i_) atomicAdd(&g_wq_qphase[i_], qph_[i_]); atomicAdd(&g_wq_qphase[8], 1ull); } } while (0)
#else
#define WQ_QTRACE_AT(slot) ((void)0)
#define QPH_DECL ((void)0)
#define QPH(i) ((void)0)
#define QPH_FLUSH ((void)0)
#endif

namespace wq {
namespace {

constexpr int kRows = 16;                 // rows per tile
constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr uint32_t kBoxBytes = kRows * 128;            // one TMA box: 16 rows x 64 bf16
constexpr uint32_t kRowBytes = 272;                     // fp32 row: 64 values + 16 B pad
constexpr uint32_t kF32Off = kBoxBytes;                 // transformed rows (cluster schedule)
constexpr uint32_t kMaxOff = kF32Off + kRows * kRowBytes;   // 6400: four 16-block maxima per row
constexpr uint32_t kSlotBytes = 7168;                   // a multiple of 1024 (TMA swizzle alignment)
constexpr int kMaxBlocks = 16;                          // blocks of one CTA (cluster schedule)
#ifndef WQ_QUANT_RING
#define WQ_QUANT_RING 16
#endif
#ifndef WQ_QUANT_MINB
#define WQ_QUANT_MINB 2
#endif
constexpr int kRing = WQ_QUANT_RING;                    // ring slots (stream schedule)
constexpr unsigned kFullMask = 0xFFFFFFFFu;

struct QParams {
    int M, K;
    int nblk;           // 64-column blocks of K
    int csplit;         // CTAs per row tile (cluster size)
    int max_nb;         // largest block count of one CTA
    int row_tiles;
    const float* inv_s;
    int rotate;
    const uint32_t* omega_blk;   // per block: kept-channel mask (2 words), x_O index of the first
    int n_out;
    int xo_ld;                   // row stride of x_O (columns n_out .. xo_ld-1 are written as zeros)
    uint16_t* xo;
    const uint32_t* pfrag;   // low-rank factor P in mma.sync B-fragment order
    uint16_t* u;
    uint8_t* codes;
    uint8_t* sf;
    int sf_layout;
    float* g;
    int* err;
    // stream kernel phase: 0 both passes with the row's own scale (WQ_ACT_SCALE_ROW); 1 first pass
    // only, row maxima folded into *amax_bits; 2 second pass only, g from *amax_bits; 3 one pass
    // with the fixed g = static_g (WQ_ACT_SCALE_STATIC)
    int phase;
    float static_g;
    unsigned int* amax_bits;
    int fp8;            // 8-bit layer in e4m3 (scale amax / 448, bytes [M, K]) instead of int8
    int fp8_bf16;       // with fp8: the e4m3 values written as exact bf16 [M, K] (A8 steps of a W4 layer)
    // Q-WAM projected complement (phase 6): xt -= u Vt right after each block's transform, u the
    // bf16 U rows written by a first launch (phase 1), Vt bf16 [r_real, K]
    const uint16_t* vt;
    int r_real;
};

// Zero the x_O columns beyond the kept channels for the rows of one tile (they meet zero weight
// rows in the GEMM, which reads the full stored width).
__device__ __forceinline__ void zero_xo_pad(const QParams& p, int tile, int tid, int nthreads) {
    const int pad = p.xo_ld - p.n_out;
    if (p.n_out == 0 || pad <= 0) return;
    for (int i = tid; i < kRows * pad; i += nthreads) {
        const int row = tile * kRows + i / pad;
        if (row < p.M) p.xo[static_cast<size_t>(row) * p.xo_ld + p.n_out + i % pad] = 0;
    }
}

// Pull block kb's slice of the packed P (NT KiB) towards this SM's L1, one 128-byte line per
// lane, ahead of the U step that reads it.
template <int NT>
__device__ __forceinline__ void prefetch_block_consts(const QParams& p, int kb, int lane) {
    if (kb >= p.nblk) return;
    if constexpr (NT > 0) {
        const char* pf = reinterpret_cast<const char*>(p.pfrag) + static_cast<size_t>(kb) * NT * 1024;
#pragma unroll
        for (int l = lane; l < NT * 8; l += 32)
            asm volatile("prefetch.global.L1 [%0];" :: "l"(pf + 128 * l));
    }
}

// Codes and scales of this lane's half row of block kb to global memory.
template <bool kOut>
__device__ __forceinline__ void emit_nvfp4(const f2 (&P)[16], float bma, float bmb, float gsc, float rg, int row,
                                           bool row_ok, int kb, int half, const QParams& p) {
    uint32_t w[4], sa, sb;
    nvfp4_half_codes<kOut>(P, bma, bmb, gsc, rg, w, sa, sb);
    const uint32_t s2 = sa | (sb << 8);
    const uint32_t s2o = __shfl_xor_sync(kFullMask, s2, 16);
    if (row_ok) {
        const int K = p.K;
        *reinterpret_cast<uint4*>(p.codes + static_cast<size_t>(row) * (K / 2) + kb * 32 + 16 * half) =
            make_uint4(w[0], w[1], w[2], w[3]);
        if (half == 0) {
            size_t off;
            if (p.sf_layout == WQ_SCALE_LAYOUT_MMA)
                off = (static_cast<size_t>(row / kBlockM) * (K / 64) + kb) * kSfAtom + (row % 32) * 16 +
                      ((row % kBlockM) / 32) * 4;
            else
                off = static_cast<size_t>(row) * (K / 16) + kb * 4;
            *reinterpret_cast<uint32_t*>(p.sf + off) = s2 | (s2o << 16);
        }
    }
}

// 8-bit values of this lane's half row of block kb as exact bf16 integers (ra = RN(1 / gsc)).
template <bool kOut>
__device__ __forceinline__ void emit_int8(const f2 (&P)[16], float gsc, float ra, int row, bool row_ok, int kb,
                                          int half, const QParams& p) {
    float va[16], vb[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        va[k] = lo2(P[k]);
        vb[k] = hi2(P[k]);
    }
    uint4* dst = reinterpret_cast<uint4*>(p.codes + (static_cast<size_t>(row) * p.K + kb * 64 + 32 * half) * 2);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float q[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (gsc != 0.0f) int8_values8_r<kOut>(j < 2 ? va + 8 * j : vb + 8 * (j - 2), gsc, ra, q);
        uint32_t pkw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(q[2 * e], q[2 * e + 1]);
            pkw[e] = *reinterpret_cast<const uint32_t*>(&h);
        }
        if (row_ok) dst[j] = make_uint4(pkw[0], pkw[1], pkw[2], pkw[3]);
    }
}

// e4m3 codes of this lane's half row of block kb (QuantWAMs sec. 4.2: FP8 W8A8 for the upgraded
// layers): q = e4m3_rn_satfinite(RN(v / a)) with ra = RN(1 / a); the quotient's conversion is
// bracketed as for the e2m1 codes (both ends of t (1 -+ 2^-21), t = RN(v ra), converting to the same
// code prove it; otherwise the exact division).  Bytes in natural channel order.
__device__ __forceinline__ uint32_t e4m3_pair_q(float a0, float a1, float sc, float ra) {
    const float t0 = __fmul_rn(a0, ra), t1 = __fmul_rn(a1, ra);
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(__fmul_rn(t1, 0.99999952316284180f)),
        "f"(__fmul_rn(t0, 0.99999952316284180f)));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(__fmul_rn(t1, 1.00000047683715820f)),
        "f"(__fmul_rn(t0, 1.00000047683715820f)));
    if (lo == hi && ra < 3.0e38f) return lo;
    uint16_t ex;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(ex) : "f"(__fdiv_rn(a1, sc)), "f"(__fdiv_rn(a0, sc)));
    return ex;
}
__device__ __forceinline__ void emit_fp8(const f2 (&P)[16], float gsc, float ra, int row, bool row_ok, int kb,
                                         int half, const QParams& p) {
    // byte c of the half at position c: channels 0..15 are the pairs' first lanes, 16..31 the second
    uint32_t bytes[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        // word q holds channels 4q .. 4q+3 of the half: 0..15 from the pairs' lows, 16..31 from highs
        const int c0 = 4 * q;
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int c = c0 + e;
            v[e] = c < 16 ? lo2(P[c]) : hi2(P[c - 16]);
        }
        uint32_t word = 0u;
        if (gsc != 0.0f) {
            const uint32_t p01 = e4m3_pair_q(v[0], v[1], gsc, ra), p23 = e4m3_pair_q(v[2], v[3], gsc, ra);
            word = (p01 & 0xFFFFu) | (p23 << 16);
        }
        bytes[q] = word;
    }
    if (!row_ok) return;
    if (p.fp8_bf16) {
        // the values of the codes, exact in bf16 (3 mantissa bits, exponents 2^-9 .. 2^8)
        uint32_t vals[16];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
#pragma unroll
            for (int hw = 0; hw < 2; ++hw) {
                const uint16_t pair = static_cast<uint16_t>(bytes[q] >> (16 * hw));
                uint32_t h2;
                asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
                const __half2 hv = *reinterpret_cast<const __half2*>(&h2);
                const __nv_bfloat162 bv = __floats2bfloat162_rn(__low2float(hv), __high2float(hv));
                vals[2 * q + hw] = *reinterpret_cast<const uint32_t*>(&bv);
            }
        }
        uint4* dst = reinterpret_cast<uint4*>(p.codes + (static_cast<size_t>(row) * p.K + kb * 64 + 32 * half) * 2);
#pragma unroll
        for (int j = 0; j < 4; ++j) dst[j] = make_uint4(vals[4 * j], vals[4 * j + 1], vals[4 * j + 2], vals[4 * j + 3]);
        return;
    }
    uint4* dst = reinterpret_cast<uint4*>(p.codes + static_cast<size_t>(row) * p.K + kb * 64 + 32 * half);
    dst[0] = make_uint4(bytes[0], bytes[1], bytes[2], bytes[3]);
    dst[1] = make_uint4(bytes[4], bytes[5], bytes[6], bytes[7]);
}

// xt -= u Vt for this lane's half row of block kb, one fp32 fma per rank term in the order
// j = 0 .. r-1 (the pairs' two lanes are separate IEEE fmas), u from the row's stored bf16 U.
template <int R>
__device__ __forceinline__ void project_block(f2 (&P)[16], const QParams& p, int row, bool row_ok, int kb, int half) {
    if constexpr (R > 0) {
        const uint16_t* urow = p.u + static_cast<size_t>(row) * R;
        const uint16_t* vb = p.vt + kb * 64 + 32 * half;
        for (int j = 0; j < p.r_real; ++j) {
            const float uj = row_ok ? __uint_as_float(static_cast<uint32_t>(urow[j]) << 16) : 0.0f;
            const f2 nu = pk2(-uj, -uj);
            const uint4* v4 = reinterpret_cast<const uint4*>(vb + static_cast<size_t>(j) * p.K);
            const uint4 q0 = __ldg(v4), q1 = __ldg(v4 + 1), q2 = __ldg(v4 + 2), q3 = __ldg(v4 + 3);
            const uint32_t w[16] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w,
                                    q2.x, q2.y, q2.z, q2.w, q3.x, q3.y, q3.z, q3.w};
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const uint32_t a = w[k / 2], b = w[8 + k / 2];
                const float vlo = __uint_as_float((k & 1) ? (a & 0xFFFF0000u) : (a << 16));   // channel k
                const float vhi = __uint_as_float((k & 1) ? (b & 0xFFFF0000u) : (b << 16));   // channel k + 16
                P[k] = fma2(nu, pk2(vlo, vhi), P[k]);
            }
        }
    }
}

// ==================================================================== cluster schedule
struct Layout {
    uint32_t off_invs, off_omega, off_bar, off_amax, off_rmax, off_upart, off_u, off_abort, total;
};

__host__ __device__ inline Layout make_layout(int max_nb, int r) {
    Layout l{};
    const uint32_t nb = static_cast<uint32_t>(max_nb);
    const uint32_t nt = static_cast<uint32_t>(r / 8);
    l.off_invs = nb * kSlotBytes;                  // inv_s slice, 256 B per block
    l.off_omega = l.off_invs + 256u * nb;          // Omega table slice, 16 B per block
    l.off_bar = l.off_omega + 16u * nb;
    l.off_amax = (l.off_bar + 8u * (nb + 1u) + 15u) & ~15u;
    l.off_rmax = l.off_amax + 4u * kRows * kConsumerWarps;
    // per warp, the U partial in mma fragment order (nt x 512 B); up to rank 32 it fits the
    // raw box of the warp's first block, which nothing reads after the warp's own U step
    l.off_upart = l.off_rmax + 4u * kRows;
    l.off_u = l.off_upart + (nt * 512u > kBoxBytes ? kConsumerWarps * nt * 512u : 0u);
    l.off_abort = l.off_u + 4u * kRows * static_cast<uint32_t>(r > 0 ? r : 1);
    l.total = l.off_abort + 16u + 1024u;
    return l;
}

template <int R, bool kInt8>
__global__ void __launch_bounds__(kThreads, R == 64 ? 2 : 3)
quantize_kernel(const __grid_constant__ CUtensorMap tmX, const QParams p) {
    constexpr int NT = R / 8;                       // n8 tiles of U
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw_addr);
    const Layout lay = make_layout(p.max_nb, R);
    const uint32_t bar_full = base + lay.off_bar;
    const uint32_t bar_const = bar_full + 8u * static_cast<uint32_t>(p.max_nb);
    const uint32_t s_invs = base + lay.off_invs;
    // shared-space accesses only (ld/st.shared): a generic access can wait behind the thread's
    // outstanding global stores
    const uint32_t s_omega = base + lay.off_omega;
    const uint32_t s_amax = base + lay.off_amax;
    float* s_rmax = reinterpret_cast<float*>(base_ptr + lay.off_rmax);
    float* s_u = reinterpret_cast<float*>(base_ptr + lay.off_u);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + lay.off_abort);
    auto upart = [&](int w) -> uint32_t {
        return static_cast<uint32_t>(NT) * 512u > kBoxBytes
                   ? base + lay.off_upart + static_cast<uint32_t>(w) * static_cast<uint32_t>(NT) * 512u
                   : base + static_cast<uint32_t>(w) * kSlotBytes;
    };

    griddep_launch_dependents();          // the GEMM may start streaming its weights now

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const bool clustered = p.csplit > 1;
    const uint32_t rank = clustered ? cluster_ctarank() : 0u;
    const int tile = clustered ? static_cast<int>(blockIdx.x) / p.csplit : static_cast<int>(blockIdx.x);
    const int kb_lo = static_cast<int>(rank) * p.nblk / p.csplit;
    const int nb = (static_cast<int>(rank) + 1) * p.nblk / p.csplit - kb_lo;

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
            for (int i = 0; i < nb; ++i) {
                const uint32_t fb = bar_full + 8u * i;
                mbar_arrive_expect_tx(fb, kBoxBytes);
                tma_load_2d(base + static_cast<uint32_t>(i) * kSlotBytes, &tmX, (kb_lo + i) * 64, tile * kRows, fb);
            }
            // this CTA's slices of inv_s and of the Omega table
            const uint32_t cbytes = (p.inv_s ? 256u * nb : 0u) + (p.n_out ? 16u * nb : 0u);
            mbar_arrive_expect_tx(bar_const, cbytes);
            if (p.inv_s) bulk_load(s_invs, p.inv_s + kb_lo * 64, 256u * nb, bar_const);
            if (p.n_out) bulk_load(base + lay.off_omega, p.omega_blk + kb_lo * 4, 16u * nb, bar_const);
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
    const int r = lane & 15, half = lane >> 4;
    const int row = tile * kRows + r;
    const bool row_ok = row < p.M;
    const int active = nb < kConsumerWarps ? nb : kConsumerWarps;   // warps that own blocks
    // waits are made warp-uniform so every shuffle below has all 32 lanes
    bool ok = __all_sync(kFullMask, mbar_wait(bar_const, 0, abort_flag, p.err, 14));

    // ---- pass 1
    float amax = 0.0f;
    for (int i = warp; i < nb; i += kConsumerWarps) prefetch_block_consts<NT>(p, kb_lo + i, lane);
    for (int i = warp; ok && i < nb; i += kConsumerWarps) {
        if (!__all_sync(kFullMask, mbar_wait(bar_full + 8u * i, 0, abort_flag, p.err, 12))) { ok = false; break; }
        if (threadIdx.x == 0) WQ_QTRACE_AT(2);
        const uint32_t slot = base + static_cast<uint32_t>(i) * kSlotBytes;
        f2 P[16];
        load_transform(slot, r, half, p.inv_s ? s_invs + static_cast<uint32_t>(i) * 256u : 0u, p.rotate, P);
        const uint32_t rowb = slot + kF32Off + static_cast<uint32_t>(r) * kRowBytes + 128u * half;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            st_shared_v4f(rowb + 16u * j, lo2(P[2 * j]), hi2(P[2 * j]), lo2(P[2 * j + 1]), hi2(P[2 * j + 1]));
        const uint32_t m0 = p.n_out ? ld_shared_u32(s_omega + 16u * i) : 0u;
        const uint32_t m1 = p.n_out ? ld_shared_u32(s_omega + 16u * i + 4u) : 0u;
        const uint32_t mine = half ? m1 : m0;
        if ((m0 | m1) != 0u) {
            // kept channels out by the whole warp from the stored rows (channel e of a row half is
            // float 2 (e % 16) + e / 16 of it): lane l takes channel l of each half for the 16
            // rows, fp16 value out and +0 in the slot; +0 in the registers
            __syncwarp();
            const uint32_t below = (1u << lane) - 1u;
            const bool k0 = (m0 >> lane) & 1u, k1 = (m1 >> lane) & 1u;
            const uint32_t first = ld_shared_u32(s_omega + 16u * i + 8u);
            const uint32_t i0 = first + static_cast<uint32_t>(__popc(m0 & below));
            const uint32_t i1 = first + static_cast<uint32_t>(__popc(m0) + __popc(m1 & below));
            const uint32_t ce = slot + kF32Off + 4u * (2u * (static_cast<uint32_t>(lane) & 15u) + (static_cast<uint32_t>(lane) >> 4));
            if (k0 || k1) {
#pragma unroll 4
                for (int rr = 0; rr < kRows; ++rr) {
                    const int rw = tile * kRows + rr;
                    const uint32_t a0 = ce + static_cast<uint32_t>(rr) * kRowBytes, a1 = a0 + 128u;
                    const float v0 = k0 ? ld_shared_f32(a0) : 0.0f, v1 = k1 ? ld_shared_f32(a1) : 0.0f;
                    if (k0) st_shared_f32(a0, 0.0f);
                    if (k1) st_shared_f32(a1, 0.0f);
                    if (rw < p.M) {
                        uint16_t* xr = p.xo + static_cast<size_t>(rw) * p.xo_ld;
                        if (k0) xr[i0] = __half_as_ushort(__float2half_rn(v0));
                        if (k1) xr[i1] = __half_as_ushort(__float2half_rn(v1));
                    }
                }
            }
            if (mine != 0u) apply_keep(P, mine);
        }
        float ma, mb;
        absmax_pairs(P, ma, mb);
        st_shared_v2f(slot + kMaxOff + static_cast<uint32_t>(r) * 16u + 8u * half, ma, mb);
        amax = fmaxf(amax, fmaxf(ma, mb));
        if constexpr (R > 0) u_step<NT>(slot, lane, kb_lo + i, p.pfrag, upart(warp), i == warp);
    }

    // ---- row amax and U over the CTA's warps (in warp order), then over the cluster
    if (threadIdx.x == 0) WQ_QTRACE_AT(3);
    if (rank == 0) zero_xo_pad(p, tile, threadIdx.x, kConsumerWarps * 32);
    amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 16));
    if (half == 0) st_shared_f32(s_amax + 4u * static_cast<uint32_t>(warp * kRows + r), amax);
    named_bar_sync(1, kConsumerWarps * 32);
    amax = 0.0f;
    for (int w = 0; w < active; ++w) amax = fmaxf(amax, ld_shared_f32(s_amax + 4u * static_cast<uint32_t>(w * kRows + r)));
    if constexpr (R > 0) {
        for (int idx = threadIdx.x; idx < NT * 128; idx += kConsumerWarps * 32) {
            float sum = 0.0f;
            for (int w = 0; w < active; ++w) sum = __fadd_rn(sum, ld_shared_f32(upart(w) + 4u * idx));
            int rr, cc;
            frag_pos(idx, rr, cc);
            if (clustered) {
                st_shared_f32(smem_u32(s_u + rr * R + cc), sum);
            } else {
                const int rg = tile * kRows + rr;
                if (rg < p.M) p.u[static_cast<size_t>(rg) * R + cc] = __bfloat16_as_ushort(__float2bfloat16_rn(sum));
            }
        }
    }
    if (clustered) {
        if (warp == 0 && half == 0) st_shared_f32(smem_u32(s_rmax + r), amax);
        cluster_arrive();
        cluster_wait();
        // all peers' values are requested before any is used, so the remote reads overlap
        float pv[16];
        const uint32_t la = smem_u32(s_rmax + r);
#pragma unroll
        for (int qr = 0; qr < 16; ++qr)
            if (qr < p.csplit) pv[qr] = ld_dsmem_f32(mapa_shared(la, static_cast<uint32_t>(qr)));
        float a = 0.0f;
#pragma unroll
        for (int qr = 0; qr < 16; ++qr)
            if (qr < p.csplit) a = fmaxf(a, pv[qr]);
        amax = a;
        if constexpr (R > 0) {
            // every rank reduces an interleaved share of the tile's U entries, in rank order
            for (int idx = threadIdx.x * p.csplit + static_cast<int>(rank); idx < kRows * R;
                 idx += kConsumerWarps * 32 * p.csplit) {
                const uint32_t la2 = smem_u32(s_u + idx);
#pragma unroll
                for (int qr = 0; qr < 16; ++qr)
                    if (qr < p.csplit) pv[qr] = ld_dsmem_f32(mapa_shared(la2, static_cast<uint32_t>(qr)));
                float sum = 0.0f;
#pragma unroll
                for (int qr = 0; qr < 16; ++qr)
                    if (qr < p.csplit) sum += pv[qr];
                const int rg = tile * kRows + idx / R;
                if (rg < p.M) p.u[static_cast<size_t>(rg) * R + idx % R] = __bfloat16_as_ushort(__float2bfloat16_rn(sum));
            }
        }
    }
    const float gsc = __fdiv_rn(amax, kInt8 ? (p.fp8 ? 448.0f : 127.0f) : 2688.0f);
    const float rg_inv = __frcp_rn(gsc);
    if (rank == 0 && warp == 0 && half == 0 && row_ok) p.g[row] = gsc;
    if (threadIdx.x == 0) WQ_QTRACE_AT(4);

    // ---- pass 2: codes and scales from the resident transformed rows
    for (int i = warp; ok && i < nb; i += kConsumerWarps) {
        const uint32_t slot = base + static_cast<uint32_t>(i) * kSlotBytes;
        const uint32_t rowb = slot + kF32Off + static_cast<uint32_t>(r) * kRowBytes + 128u * half;
        f2 P[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 t = ld_shared_v4f(rowb + 16u * j);
            P[2 * j] = pk2(t.x, t.y);
            P[2 * j + 1] = pk2(t.z, t.w);
        }
        if constexpr (kInt8) {
            if (p.fp8) emit_fp8(P, gsc, rg_inv, row, row_ok, kb_lo + i, half, p);
            else emit_int8<true>(P, gsc, rg_inv, row, row_ok, kb_lo + i, half, p);
        } else {
            const float2 bm = ld_shared_v2f(slot + kMaxOff + static_cast<uint32_t>(r) * 16u + 8u * half);
            emit_nvfp4<true>(P, bm.x, bm.y, gsc, rg_inv, row, row_ok, kb_lo + i, half, p);
        }
    }
    if (threadIdx.x == 0) WQ_QTRACE_AT(5);
    if (clustered) {
        cluster_arrive();                 // peers are done reading this CTA's s_rmax / s_u
        cluster_wait();
    }
    if (threadIdx.x == 0) WQ_QTRACE_AT(6);
}

// ==================================================================== stream schedule
struct SLayout {
    uint32_t off_invs, off_omega, off_amax, off_upart, off_bar, off_abort, total;
};

__host__ __device__ inline SLayout make_stream_layout(int K, int r) {
    SLayout l{};
    const uint32_t nblk = static_cast<uint32_t>(K / 64);
    l.off_invs = kRing * kBoxBytes;                 // ring of raw boxes
    l.off_omega = l.off_invs + 256u * kRing;        // each ring slot's block of inv_s
    l.off_amax = l.off_omega + 16u * nblk;          // the Omega table
    l.off_upart = l.off_amax + 4u * kRows * kConsumerWarps;
    l.off_bar = l.off_upart + kConsumerWarps * static_cast<uint32_t>(r / 8) * 512u;
    l.off_abort = l.off_bar + 8u * (2 * kRing + 1);
    l.total = l.off_abort + 16u + 1024u;
    return l;
}

template <int R, bool kInt8>
__global__ void __launch_bounds__(kThreads, R == 64 ? 2 : WQ_QUANT_MINB)
quantize_stream_kernel(const __grid_constant__ CUtensorMap tmX, const QParams p) {
    constexpr int NT = R / 8;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw_addr);
    const SLayout lay = make_stream_layout(p.K, R);
    const uint32_t bar_full = base + lay.off_bar;
    const uint32_t bar_empty = bar_full + 8u * kRing;
    const uint32_t bar_const = bar_empty + 8u * kRing;
    const uint32_t s_invs = base + lay.off_invs;
    // shared-space accesses only (ld/st.shared): a generic access can wait behind the thread's
    // outstanding global stores
    const uint32_t s_omega = base + lay.off_omega;
    const uint32_t s_amax = base + lay.off_amax;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + lay.off_abort);
    const int nblk = p.nblk;

    griddep_launch_dependents();

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kRing; ++i) {
            mbar_init(bar_full + 8u * i, 1);
            mbar_init(bar_empty + 8u * i, 1);
        }
        mbar_init(bar_const, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer: every block
        // of each of this CTA's row tiles, twice, in the order the consumer warps take them
        if (lane == 0) {
            tma_prefetch_desc(&tmX);
            griddep_wait();
            const uint32_t cbytes = p.n_out ? 16u * nblk : 0u;
            mbar_arrive_expect_tx(bar_const, cbytes);
            if (p.n_out) bulk_load(base + lay.off_omega, p.omega_blk, 16u * nblk, bar_const);
            uint32_t q = 0;
            bool ok = true;
            const int passes = (p.phase == 0 || p.phase == 6) ? 2 : 1;
            for (int tile = blockIdx.x; ok && tile < p.row_tiles; tile += gridDim.x)
                for (int pass = 0; ok && pass < passes; ++pass)
                    for (int kb = 0; kb < nblk; ++kb, ++q) {
                        const uint32_t s = q % kRing;
                        if (q >= kRing && !mbar_wait(bar_empty + 8u * s, ((q / kRing) - 1u) & 1u, abort_flag, p.err, 21)) {
                            ok = false;
                            break;
                        }
                        // the box and the block's 64 inv_s values travel together
                        mbar_arrive_expect_tx(bar_full + 8u * s, kBoxBytes + (p.inv_s ? 256u : 0u));
                        tma_load_2d(base + s * kBoxBytes, &tmX, kb * 64, tile * kRows, bar_full + 8u * s);
                        if (p.inv_s) bulk_load(s_invs + 256u * s, p.inv_s + 64 * kb, 256u, bar_full + 8u * s);
                    }
            // every copy has landed before this CTA can finish
            for (uint32_t t = q > kRing ? q - kRing : 0u; t < q; ++t)
                mbar_wait(bar_full + 8u * (t % kRing), (t / kRing) & 1u, abort_flag, p.err, 22);
            mbar_wait(bar_const, 0, abort_flag, p.err, 23);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers (warps 0-7)
    const int r = lane & 15, half = lane >> 4;
    const int active = nblk < kConsumerWarps ? nblk : kConsumerWarps;
    const uint32_t upart = base + lay.off_upart + static_cast<uint32_t>(warp * NT) * 512u;
    bool ok = __all_sync(kFullMask, mbar_wait(bar_const, 0, abort_flag, p.err, 24));
    const bool first_pass = p.phase != 2;     // smoothing, FWHT, U, x_O, maxima
    const bool second_pass = p.phase == 0 || p.phase == 2 || p.phase == 6;
    const bool project = p.phase == 6;        // U comes from the previous launch
    // phase 2: the batch maximum was folded in by the previous grid; phase 3: the calibrated g
    float g_fixed = p.static_g;
    if (p.phase == 6) griddep_wait();          // U rows written by the previous grid
    if (p.phase == 2) {
        griddep_wait();
        g_fixed = __fdiv_rn(__uint_as_float(*reinterpret_cast<volatile unsigned int*>(p.amax_bits)), 2688.0f);
    }
    float cta_amax = 0.0f;                             // phase 1: maximum over this CTA's rows
    uint32_t q0 = 0;                                   // ring sequence number of the tile's first block
    QPH_DECL;
    // every warp runs every tile's barriers, also after a failed wait (ok == false skips work)
    for (int tile = blockIdx.x; tile < p.row_tiles; tile += gridDim.x) {
        const int row = tile * kRows + r;
        const bool row_ok = row < p.M;
        float gsc = g_fixed;
        float rg_inv = __frcp_rn(g_fixed);
        if (first_pass) {
            // ---- pass 1 (phase 3: the only pass, codes out with the fixed g)
            float amax = 0.0f;
            if (tile == static_cast<int>(blockIdx.x)) prefetch_block_consts<NT>(p, warp, lane);
            for (int kb = warp; ok && kb < nblk; kb += kConsumerWarps) {
                const uint32_t q = q0 + static_cast<uint32_t>(kb), s = q % kRing;
                prefetch_block_consts<NT>(p, kb + kConsumerWarps < nblk ? kb + kConsumerWarps : warp, lane);
                QPH(3);
                if (!__all_sync(kFullMask, mbar_wait(bar_full + 8u * s, (q / kRing) & 1u, abort_flag, p.err, 25))) {
                    ok = false;
                    break;
                }
                QPH(0);
                const uint32_t box = base + s * kBoxBytes;
                // the block's share of U first (it reads the raw box), so the transformed values
                // are not live across the tensor-core step
                if constexpr (R > 0)
                    if (!project) u_step<NT>(box, lane, kb, p.pfrag, upart, kb == warp);
                QPH(2);
                f2 P[16];
                load_transform(box, r, half, p.inv_s ? s_invs + 256u * s : 0u, p.rotate, P);
                if constexpr (R > 0)
                    if (project) project_block<R>(P, p, row, row_ok, kb, half);
                QPH(1);
                const uint32_t m0 = p.n_out ? ld_shared_u32(s_omega + 16u * kb) : 0u;
                const uint32_t m1 = p.n_out ? ld_shared_u32(s_omega + 16u * kb + 4u) : 0u;
                if ((m0 | m1) != 0u) {
                    // kept channels: fp16 values through a copy in the consumed box (lane l writes its
                    // 32 channels as fp16 pairs at l * 64 B), then out by the whole warp: lane l takes
                    // channel l of each half for the 16 rows, so a block with many kept channels
                    // costs a few row sweeps and a row's stores are contiguous; +0 in the registers
                    __syncwarp();                  // every lane is done reading the box
                    const uint32_t sc = box + static_cast<uint32_t>(lane) * 64u;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t hw[4];
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const __half2 h2 = __floats2half2_rn(lo2(P[4 * j + t]), hi2(P[4 * j + t]));
                            hw[t] = *reinterpret_cast<const uint32_t*>(&h2);
                        }
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(sc + 16u * j), "r"(hw[0]), "r"(hw[1]),
                                     "r"(hw[2]), "r"(hw[3]) : "memory");
                    }
                    __syncwarp();
                    const uint32_t below = (1u << lane) - 1u;
                    const bool k0 = (m0 >> lane) & 1u, k1 = (m1 >> lane) & 1u;
                    const uint32_t first = ld_shared_u32(s_omega + 16u * kb + 8u);
                    const uint32_t i0 = first + static_cast<uint32_t>(__popc(m0 & below));
                    const uint32_t i1 = first + static_cast<uint32_t>(__popc(m0) + __popc(m1 & below));
                    // channel e of a row half sits at 4 (e % 16) + 2 (e / 16) of that lane's copy
                    const uint32_t ce = 4u * (static_cast<uint32_t>(lane) & 15u) + 2u * (static_cast<uint32_t>(lane) >> 4);
                    if (k0 || k1) {
#pragma unroll 4
                        for (int rr = 0; rr < kRows; ++rr) {
                            const int rw = tile * kRows + rr;
                            uint16_t h0 = 0, h1 = 0;
                            if (k0) asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h0) : "r"(box + static_cast<uint32_t>(rr) * 64u + ce) : "memory");
                            if (k1) asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h1) : "r"(box + static_cast<uint32_t>(rr + 16) * 64u + ce) : "memory");
                            if (rw < p.M) {
                                uint16_t* xr = p.xo + static_cast<size_t>(rw) * p.xo_ld;
                                if (k0) xr[i0] = h0;
                                if (k1) xr[i1] = h1;
                            }
                        }
                    }
                    const uint32_t mine = half ? m1 : m0;
                    if (mine != 0u) apply_keep(P, mine);
                    fence_proxy_async_smem();      // the copy precedes the producer's next TMA into the slot
                }
                float ma, mb;
                absmax_pairs(P, ma, mb);
                amax = fmaxf(amax, fmaxf(ma, mb));
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_empty + 8u * s);
                if constexpr (!kInt8)
                    if (p.phase == 3) emit_nvfp4<false>(P, ma, mb, gsc, rg_inv, row, row_ok, kb, half, p);
            }
            QPH(3);
            // ---- row amax and U over the warps, in warp order
            amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 16));
            if (half == 0) st_shared_f32(s_amax + 4u * static_cast<uint32_t>(warp * kRows + r), amax);
            named_bar_sync(1, kConsumerWarps * 32);
            amax = 0.0f;
            for (int w = 0; w < active; ++w)
                amax = fmaxf(amax, ld_shared_f32(s_amax + 4u * static_cast<uint32_t>(w * kRows + r)));
            if constexpr (R > 0) {
                for (int idx = threadIdx.x; idx < (project ? 0 : NT * 128); idx += kConsumerWarps * 32) {
                    float sum = 0.0f;
                    for (int w = 0; w < active; ++w)
                        sum = __fadd_rn(sum, ld_shared_f32(base + lay.off_upart + static_cast<uint32_t>(w * NT) * 512u + 4u * idx));
                    int rr, cc;
                    frag_pos(idx, rr, cc);
                    const int rg = tile * kRows + rr;
                    if (rg < p.M) p.u[static_cast<size_t>(rg) * R + cc] = __bfloat16_as_ushort(__float2bfloat16_rn(sum));
                }
            }
            zero_xo_pad(p, tile, threadIdx.x, kConsumerWarps * 32);
            named_bar_sync(1, kConsumerWarps * 32);        // maxima and partials are free again
            if (p.phase == 0 || p.phase == 6) {
                gsc = __fdiv_rn(amax, kInt8 ? (p.fp8 ? 448.0f : 127.0f) : 2688.0f);
                rg_inv = __frcp_rn(gsc);
            }
            cta_amax = fmaxf(cta_amax, amax);
            q0 += static_cast<uint32_t>(nblk);
        }
        if (warp == 0 && half == 0 && row_ok && p.phase != 1) p.g[row] = gsc;
        QPH(4);
        if (second_pass) {
            // ---- pass 2: the blocks again (from L2), transform recomputed
            for (int kb = warp; ok && kb < nblk; kb += kConsumerWarps) {
                const uint32_t q = q0 + static_cast<uint32_t>(kb), s = q % kRing;
                QPH(7);
                if (!__all_sync(kFullMask, mbar_wait(bar_full + 8u * s, (q / kRing) & 1u, abort_flag, p.err, 26))) {
                    ok = false;
                    break;
                }
                QPH(5);
                f2 P[16];
                load_transform(base + s * kBoxBytes, r, half, p.inv_s ? s_invs + 256u * s : 0u, p.rotate, P);
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_empty + 8u * s);
                if (project) project_block<R>(P, p, row, row_ok, kb, half);
                QPH(6);
                const uint32_t mk = p.n_out ? ld_shared_u32(s_omega + 16u * kb + 4u * static_cast<uint32_t>(half)) : 0u;
                if (mk != 0u) apply_keep(P, mk);
                if constexpr (kInt8) {
                    if (p.fp8) emit_fp8(P, gsc, rg_inv, row, row_ok, kb, half, p);
                    else emit_int8<false>(P, gsc, rg_inv, row, row_ok, kb, half, p);
                } else {
                    float ma, mb;
                    absmax_pairs(P, ma, mb);
                    emit_nvfp4<false>(P, ma, mb, gsc, rg_inv, row, row_ok, kb, half, p);
                }
            }
            q0 += static_cast<uint32_t>(nblk);
        }
        QPH(7);
    }
    if (p.phase == 1 && p.amax_bits != nullptr && warp == 0) {
        // lanes 0..15 hold the maxima of the CTA's rows r; one atomic per CTA (non-negative
        // floats order like their bit patterns)
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) cta_amax = fmaxf(cta_amax, __shfl_xor_sync(kFullMask, cta_amax, o));
        if (lane == 0) atomicMax(p.amax_bits, __float_as_uint(cta_amax));
    }
    QPH_FLUSH;
}

struct Choice {
    int csplit, max_nb;
};

// Cluster schedule: at most one 64-block per consumer warp where the cluster size allows (at
// most 16 CTAs per row tile); K = 16384 gives 16 blocks per CTA.
Choice choose(int K) {
    const int nblk = K / 64;
    int cs = (nblk + kConsumerWarps - 1) / kConsumerWarps;
    if (cs > 16) cs = 16;
    if (cs < 1) cs = 1;
    return Choice{cs, (nblk + cs - 1) / cs};
}

template <int R, bool kInt8>
cudaError_t launch_r(const CUtensorMap& tm, const QParams& qp, bool stream, int num_sms, cudaStream_t st) {
    static bool attr_set = false;
    if (!attr_set) {
        const Layout worst = make_layout(kMaxBlocks, R);
        cudaError_t e = cudaFuncSetAttribute(quantize_kernel<R, kInt8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(worst.total));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(quantize_kernel<R, kInt8>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        const SLayout sworst = make_stream_layout(16384, R);
        e = cudaFuncSetAttribute(quantize_stream_kernel<R, kInt8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(sworst.total));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    cudaLaunchConfig_t cfg{};
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    int na = 0;
    at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (stream) {
        const SLayout lay = make_stream_layout(qp.K, R);
        int per_sm = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quantize_stream_kernel<R, kInt8>, kThreads,
                                                                      lay.total);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) return cudaErrorInvalidConfiguration;
        // Every resident CTA is used even when the row tiles in flight outgrow the L2 and part of
        // the second pass comes from DRAM: the kernel is bound by its instructions with DRAM well
        // below its peak.  Two CTAs per SM of up to 112 registers (no spills at rank 0 or 16)
        // measured 323 us at K = 8960 against 332 us for three CTAs capped at 72 registers.
        // the WQ_QUANT_CTAS_PER_SM knob overrides the residency (tuning)
        const int v = tune(kTuneQuantCtasPerSm);
        if (v >= 1 && v <= per_sm + 8) per_sm = v;
        const int grid = qp.row_tiles < per_sm * num_sms ? qp.row_tiles : per_sm * num_sms;
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        cfg.dynamicSmemBytes = lay.total;
        cfg.attrs = at;
        cfg.numAttrs = na;
        return cudaLaunchKernelEx(&cfg, quantize_stream_kernel<R, kInt8>, tm, qp);
    }
    const Layout lay = make_layout(qp.max_nb, R);
    cfg.gridDim = dim3(static_cast<unsigned>(qp.row_tiles * qp.csplit));
    cfg.dynamicSmemBytes = lay.total;
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

bool quant_stream_schedule(int M, int num_sms) {
    // many row tiles: the persistent stream schedule; few: spread K over clusters
    bool stream = (M + kRows - 1) / kRows >= 2 * num_sms;
    // the WQ_QUANT_SCHEDULE knob pins the schedule (tuning and tests): 0 cluster, 1 stream,
    // 2 register-resident (where it applies; else stream)
    const int fm = tune(kTuneQuantSchedule);
    if (fm >= 0) stream = fm >= 1;
    return stream;
}

cudaError_t launch_quantize_act(const QuantArgs& a, cudaStream_t st) {
    if (a.M <= 0) return cudaSuccess;
    Choice ch = choose(a.K);
    const int row_tiles = (a.M + kRows - 1) / kRows;
    // batch-wide tensor scales run on the stream kernel: the maximum and the codes as two
    // launches (TENSOR) or the codes in one pass (STATIC)
    const bool stream = a.act_scale != WQ_ACT_SCALE_ROW || a.vt != nullptr || quant_stream_schedule(a.M, a.num_sms);
    // the WQ_QUANT_SPLIT knob pins the CTAs per row tile of the cluster schedule (tuning and tests)
    {
        const int v = tune(kTuneQuantSplit);
        const int nblk = a.K / 64;
        if (v >= 1 && v <= 16 && v <= nblk && (nblk + v - 1) / v <= kMaxBlocks) ch = Choice{v, (nblk + v - 1) / v};
    }
    if (ch.max_nb > kMaxBlocks) return cudaErrorInvalidValue;
    // many rows of a 4-bit layer with per-row scales and K <= 1536: the register-resident schedule
    // (knob value 1 pins the two-pass stream schedule instead)
    if (stream && tune(kTuneQuantSchedule) != 1 && quant_resident_eligible(a)) return launch_quantize_resident(a, st);
    QParams qp{};
    qp.M = a.M; qp.K = a.K; qp.nblk = a.K / 64; qp.csplit = ch.csplit; qp.max_nb = ch.max_nb;
    qp.row_tiles = row_tiles;
    qp.inv_s = a.inv_s; qp.rotate = a.rotate; qp.omega_blk = a.omega_blk; qp.n_out = a.n_out; qp.xo = a.xo;
    qp.xo_ld = a.xo_ld > a.n_out ? a.xo_ld : a.n_out;
    qp.phase = a.act_scale == WQ_ACT_SCALE_STATIC ? 3 : 0;
    qp.static_g = a.static_g;
    qp.amax_bits = a.amax_bits;
    qp.fp8 = a.fp8 ? 1 : 0;
    qp.fp8_bf16 = a.fp8_bf16 ? 1 : 0;
    qp.vt = a.vt;
    qp.r_real = a.r_real;
    qp.pfrag = a.pfrag; qp.u = a.u; qp.codes = a.codes; qp.sf = a.sf; qp.sf_layout = a.sf_layout; qp.g = a.g;
    qp.err = a.err;
    if (a.int8) {
        // 8-bit activations; the low-rank and kept-channel side outputs only for W4 layers at A8 steps
        if (qp.phase != 0 || ((a.r != 0 || a.n_out != 0) && !(a.fp8 && a.fp8_bf16))) return cudaErrorInvalidValue;
        switch (a.r) {
            case 0: return launch_r<0, true>(*a.tmX, qp, stream, a.num_sms, st);
            case 16: return launch_r<16, true>(*a.tmX, qp, stream, a.num_sms, st);
            case 32: return launch_r<32, true>(*a.tmX, qp, stream, a.num_sms, st);
            case 64: return launch_r<64, true>(*a.tmX, qp, stream, a.num_sms, st);
            default: return cudaErrorInvalidValue;
        }
    }
    auto launch = [&](const QParams& q) -> cudaError_t {
        switch (a.r) {
            case 0: return launch_r<0, false>(*a.tmX, q, stream, a.num_sms, st);
            case 16: return launch_r<16, false>(*a.tmX, q, stream, a.num_sms, st);
            case 32: return launch_r<32, false>(*a.tmX, q, stream, a.num_sms, st);
            case 64: return launch_r<64, false>(*a.tmX, q, stream, a.num_sms, st);
            default: return cudaErrorInvalidValue;
        }
    };
    if (a.vt != nullptr) {
        // Q-WAM projected complement: U first (phase 1 without the maximum), then both passes on
        // the projected values
        if (a.r == 0 || a.u == nullptr || a.act_scale != WQ_ACT_SCALE_ROW) return cudaErrorInvalidValue;
        QParams q1 = qp;
        q1.phase = 1;
        q1.amax_bits = nullptr;
        const cudaError_t e = launch(q1);
        if (e != cudaSuccess) return e;
        QParams q2 = qp;
        q2.phase = 6;
        return launch(q2);
    }
    if (a.act_scale == WQ_ACT_SCALE_TENSOR) {
        if (!a.amax_bits) return cudaErrorInvalidValue;
        QParams q1 = qp;
        q1.phase = 1;                   // maxima (and U, x_O), no codes
        const cudaError_t e = launch(q1);
        if (e != cudaSuccess) return e;
        QParams q2 = qp;
        q2.phase = 2;                   // codes with the batch's g
        return launch(q2);
    }
    return launch(qp);
}

}  // namespace wq
