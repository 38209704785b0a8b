// wq_peak.cu -- tensor-core issue-rate microbenchmark (no counterpart on the pages).
//
// One thread per CTA (or per CTA pair) issues `iters` dense tcgen05.mma instructions back to
// back on fixed shared-memory operands into one TMEM accumulator, optionally with tcgen05.cp
// copies of block-scale atoms in between, and the CTA times the run with %globaltimer and
// %clock64.  Nothing else competes for the tensor pipe, so the aggregate over all SMs is the
// rate the hardware retires that instruction form at: the measured dense peak that the GEMM's
// roofline fraction is read against, and the cost of the scale copies the block-scaled GEMM
// issues per K block.
//
// Forms: kind 0 = mxf4nvf4 block-scaled e2m1 x e2m1 (K = 64 per instruction, ue4m3 scales per
// 16), kind 1 = f16 with bf16 operands (K = 16), kind 2 = f8f6f4 with e4m3 operands (K = 32);
// N = 64..256; M = 128 on one CTA or 256 on a CTA pair (cta_group::2).  Copies: 0..3
// tcgen05.cp per MMA, shape 0 = 32x128b.warpx4 (one 512-byte scale atom), 1 = 128x256b (4 KiB).
#include <cuda_runtime.h>

#include <cstdint>
#include <string>
#include <vector>

#include "ptx.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int kPeakThreads = 128;
constexpr uint32_t kOffB = 16384;            // A: 128 rows x 128 B; B: 256 rows x 128 B
constexpr uint32_t kOffSf = 49152;           // scale region, 16 KiB (any copy shape stays inside)
constexpr uint32_t kOffBar = 65536;
constexpr uint32_t kPeakSmem = 200 * 1024;   // one CTA per SM (TMEM is taken whole)

struct PeakParams {
    int kind, n, copies, copy_shape, iters;
    int feeder;      // who issues the copies: 0 the MMA thread, 1 another warp (unordered),
                     // 2 warps 1-3 write TMEM with tcgen05.st from registers instead (unordered)
    int zero_data;   // 1: all-zero operands
    int accs;        // 1 or 2 accumulators, alternated MMA by MMA (2 needs n <= 128 for kind 0)
    unsigned long long* out;                 // per CTA: {ns, cycles}
    int* err;
};

__device__ __forceinline__ void cp_128x256b(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" :: "r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void cp_128x256b_pair(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::2.128x256b [%0], %1;" :: "r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void tmem_st_32x32b_x4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};"
                 :: "r"(taddr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ uint64_t clock64_now() {
    uint64_t c;
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(c));
    return c;
}

template <bool kPair>
__global__ void __launch_bounds__(kPeakThreads, 1) mma_peak_kernel(const PeakParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* bp = smem_raw + (base - raw);
    const uint32_t bar = base + kOffBar;
    uint32_t* holder = reinterpret_cast<uint32_t*>(bp + kOffBar + 16);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bp + kOffBar + 32);
    const uint32_t rank = kPair ? cluster_ctarank() : 0u;

    // operands: a fixed pseudo-random pattern that is finite in every input type
    for (uint32_t i = threadIdx.x; i < kOffSf / 4; i += kPeakThreads) {
        uint32_t v = (i * 2654435761u) ^ (i >> 3);
        if (p.kind == 1) v = (v & 0x007F007Fu) | 0x3F003F00u;      // bf16 in [0.5, 1)
        if (p.kind == 2) v &= 0x77777777u;                          // e4m3 without NaN
        if (p.zero_data) v = 0u;
        reinterpret_cast<uint32_t*>(bp)[i] = v;
    }
    for (uint32_t i = threadIdx.x; i < 16384u / 4; i += kPeakThreads)
        reinterpret_cast<uint32_t*>(bp + kOffSf)[i] = 0x38383838u;  // ue4m3 1.0
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    fence_proxy_async_smem();                // generic-proxy writes visible to the tensor core
    if (threadIdx.x < 32) {
        if (kPair) {
            tmem_alloc_pair(smem_u32(holder), 512);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(holder), 512);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (kPair) cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *holder;

    if (p.feeder == 1 && threadIdx.x == 32 && rank == 0) {
        // copies from another warp, alongside the MMAs (no ordering between the two)
        const uint64_t sd = smem_desc(base + kOffSf, 0, 128, 0);
        for (int i = 0; i < p.iters; ++i)
            for (int c = 0; c < p.copies; ++c) {
                const uint32_t slot = tmem + 320u + 48u * static_cast<uint32_t>(i & 3) + 4u * c;
                if (kPair) tmem_cp_pair_32x128b_x4(slot, sd);
                else tmem_cp_32x128b_x4(slot, sd);
            }
    }
    if (p.feeder == 2 && threadIdx.x >= 32) {
        // warps 1-3 write their lane quadrants of the slots from registers, alongside the MMAs
        const uint32_t q = static_cast<uint32_t>(threadIdx.x / 32);
        for (int i = 0; i < p.iters; ++i) {
            for (int c = 0; c < p.copies; ++c) {
                const uint32_t slot = tmem + ((32u * q) << 16) + 320u + 48u * static_cast<uint32_t>(i & 3) + 4u * c;
                tmem_st_32x32b_x4(slot, i, c, q, 7u);
            }
        }
        tmem_wait_st();
    }
    if (threadIdx.x == 0 && rank == 0) {
        const uint32_t M = kPair ? 256u : 128u;
        const uint32_t N = static_cast<uint32_t>(p.n);
        const uint32_t mn = ((N >> 3) << 17) | ((M >> 4) << 24);
        uint32_t idesc;
        if (p.kind == 0) idesc = (1u << 7) | (1u << 10) | mn;              // e2m1 x e2m1, f32 accumulate
        else if (p.kind == 1) idesc = (1u << 4) | (1u << 7) | (1u << 10) | mn;   // bf16 x bf16 -> f32
        else idesc = (1u << 4) | mn;                                       // e4m3 x e4m3 -> f32
        const uint64_t ad = smem_desc(base, 16, 1024, 2), bd = smem_desc(base + kOffB, 16, 1024, 2);
        const uint32_t sfa = tmem + 256u, sfb = tmem + 272u;
        const uint64_t sdesc = smem_desc(base + kOffSf, 0, 128, 0);
        const uint64_t sdesc_big = smem_desc(base + kOffSf, 128, 256, 0);
        // the scales the MMAs read, once
        if (kPair) {
            tmem_cp_pair_32x128b_x4(sfa, sdesc);
            tmem_cp_pair_32x128b_x4(sfb, sdesc);
            tmem_cp_pair_32x128b_x4(sfb + 4u, sdesc);
        } else {
            tmem_cp_32x128b_x4(sfa, sdesc);
            tmem_cp_32x128b_x4(sfb, sdesc);
            tmem_cp_32x128b_x4(sfb + 4u, sdesc);
        }
        const uint64_t t0 = global_timer_ns(), c0 = clock64_now();
        for (int i = 0; i < p.iters; ++i) {
            // copies go to four rotating 32-column slots past the MMAs' own scale columns
            const uint32_t slot = tmem + 320u + 48u * static_cast<uint32_t>(i & 3);
            for (int c = 0; p.feeder == 0 && c < p.copies; ++c) {
                if (p.copy_shape == 0) {
                    if (kPair) tmem_cp_pair_32x128b_x4(slot + 4u * c, sdesc);
                    else tmem_cp_32x128b_x4(slot + 4u * c, sdesc);
                } else {
                    if (kPair) cp_128x256b_pair(slot + 8u * c, sdesc_big);
                    else cp_128x256b(slot + 8u * c, sdesc_big);
                }
            }
            const uint32_t acc = i >= p.accs ? 1u : 0u;
            const uint32_t d = tmem + (p.accs == 2 && (i & 1) ? (p.kind == 0 ? 128u : 256u) : 0u);
            if (p.kind == 0) {
                if (kPair) mma_nvf4_pair(d, ad, bd, idesc, sfa, sfb, acc);
                else mma_nvf4(d, ad, bd, idesc, sfa, sfb, acc);
            } else if (p.kind == 1) {
                if (kPair) mma_f16_pair(d, ad, bd, idesc, acc);
                else mma_f16(d, ad, bd, idesc, acc);
            } else {
                if (kPair) mma_f8_pair(d, ad, bd, idesc, acc);
                else mma_f8(d, ad, bd, idesc, acc);
            }
        }
        if (kPair) tc_commit_pair_mc(bar, 0x3);
        else tc_commit(bar);
        mbar_wait(bar, 0, abort_flag, p.err, 95);
        const uint64_t t1 = global_timer_ns(), c1 = clock64_now();
        const int slot = kPair ? static_cast<int>(blockIdx.x) / 2 : static_cast<int>(blockIdx.x);
        p.out[2 * slot] = t1 - t0;
        p.out[2 * slot + 1] = c1 - c0;
    }
    if (kPair && threadIdx.x == 0 && rank == 1) mbar_wait(bar, 0, abort_flag, p.err, 96);   // the peer's MMAs are done
    tc_fence_before();
    __syncthreads();
    if (kPair) cluster_sync();
    if (threadIdx.x < 32) {
        tc_fence_after();
        if (kPair) tmem_dealloc_pair(tmem, 512);
        else tmem_dealloc(tmem, 512);
    }
}

}  // namespace
}  // namespace wq

extern "C" WQ_API wq_status wq_mma_peak(int kind, int n, int pair, int copies, int copy_shape, int iters,
                                        int feeder, int zero_data, int accs, double* tflops, double* ns_per_mma,
                                        double* sm_mhz) {
    using namespace wq;
    if (!tflops || !ns_per_mma || !sm_mhz || kind < 0 || kind > 2 || (n % 16) || n < 64 || n > 256 ||
        copies < 0 || copies > 3 || copy_shape < 0 || copy_shape > 1 || iters < 1 || iters > (1 << 22) ||
        feeder < 0 || feeder > 2 || (feeder == 2 && copy_shape != 0) || (feeder == 2 && pair) ||
        accs < 1 || accs > 2 || (accs == 2 && n > (kind == 0 ? 128 : 256))) {
        set_last_error("wq_mma_peak: bad argument");
        return WQ_ERR_INVALID;
    }
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int units = pair ? sms / 2 : sms;
    unsigned long long* d_out = nullptr;
    int* d_err = nullptr;
    auto cleanup = [&] { cudaFree(d_out); cudaFree(d_err); };
    if (cudaMalloc(&d_out, sizeof(unsigned long long) * 2 * units) != cudaSuccess ||
        cudaMalloc(&d_err, sizeof(int)) != cudaSuccess) {
        cleanup();
        set_last_error("wq_mma_peak: cudaMalloc failed");
        return WQ_ERR_OOM;
    }
    cudaMemset(d_err, 0, sizeof(int));
    PeakParams pp{kind, n, copies, copy_shape, iters, feeder, zero_data, accs, d_out, d_err};
    cudaError_t e;
    if (pair) {
        e = cudaFuncSetAttribute(mma_peak_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPeakSmem);
        if (e == cudaSuccess) {
            cudaLaunchConfig_t cfg{};
            cfg.gridDim = dim3(static_cast<unsigned>(2 * units));
            cfg.blockDim = dim3(kPeakThreads);
            cfg.dynamicSmemBytes = kPeakSmem;
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = 2;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            cfg.attrs = at;
            cfg.numAttrs = 1;
            e = cudaLaunchKernelEx(&cfg, mma_peak_kernel<true>, pp);
        }
    } else {
        e = cudaFuncSetAttribute(mma_peak_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPeakSmem);
        if (e == cudaSuccess) {
            mma_peak_kernel<false><<<units, kPeakThreads, kPeakSmem>>>(pp);
            e = cudaGetLastError();
        }
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    std::vector<unsigned long long> out(2 * units);
    int err = 0;
    if (e == cudaSuccess) e = cudaMemcpy(out.data(), d_out, out.size() * 8, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(&err, d_err, sizeof(int), cudaMemcpyDeviceToHost);
    cleanup();
    if (e != cudaSuccess) {
        set_last_error((std::string("wq_mma_peak: ") + cudaGetErrorString(e)).c_str());
        return WQ_ERR_CUDA;
    }
    if (err) {
        set_last_error("wq_mma_peak: a wait timed out");
        return WQ_ERR_TIMEOUT;
    }
    const double kdepth = kind == 0 ? 64.0 : (kind == 1 ? 16.0 : 32.0);
    const double flops_per_mma = 2.0 * (pair ? 256.0 : 128.0) * n * kdepth;
    double rate = 0.0, ns = 0.0, mhz = 0.0;
    for (int u = 0; u < units; ++u) {
        const double t = static_cast<double>(out[2 * u]);
        rate += flops_per_mma * iters / t;          // flop per ns = GFLOP/s
        ns += t / iters;
        mhz += static_cast<double>(out[2 * u + 1]) / t * 1e3;
    }
    *tflops = rate / 1e3;
    *ns_per_mma = ns / units;
    *sm_mhz = mhz / units;
    return WQ_OK;
}
