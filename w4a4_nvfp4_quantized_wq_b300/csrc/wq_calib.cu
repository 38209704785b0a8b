// wq_calib.cu -- on-device outlier calibration (QuantWAMs sec. 3.1, Eq. (1)-(3), one context):
// the pooled squared energy of every channel of the transformed activation,
//     z(c) = mean_t xt[t, c]^2,
// and the Top-K channels by z that stay in 16-bit.  xt is the activation quantiser's transform
// of each row (smoothing before or after the block-64 Walsh-Hadamard butterflies, the pages'
// order, one fp32 operation each); squares and sums are fp64.
//
//   energy_partial_kernel  CTA (64-channel block, 1024-row group): each thread transforms its
//                          rows' block in registers and accumulates the 64 squares; the CTA
//                          reduces them in a fixed order (shuffle tree, then warps in order).
//   energy_final_kernel    z(c) = sum over row groups in order / M.
//   topk_flag_kernel       channel c is selected when fewer than n channels rank above it
//                          (larger z, or equal z and a lower index).
//   topk_compact_kernel    the selected channels in ascending order (one CTA, block scan).
#include <cuda_bf16.h>

#include <string>

#include "ptx.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int kCalThreads = 128;
constexpr int kRowsPerGroup = 1024;
constexpr int kRankThreads = 256;
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kCalThreads) energy_partial_kernel(const uint16_t* __restrict__ x, int M, int K,
                                                                     const float* __restrict__ s, int rotate,
                                                                     double* __restrict__ partial) {
    const int kb = blockIdx.x, g = blockIdx.y;
    const int r0 = g * kRowsPerGroup, r1 = min(M, r0 + kRowsPerGroup);
    const bool after = (rotate & 3) == 3;
    float inv[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) inv[i] = s != nullptr ? __fdiv_rn(1.0f, __ldg(s + kb * 64 + i)) : 1.0f;
    double acc[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) acc[i] = 0.0;
    for (int r = r0 + static_cast<int>(threadIdx.x); r < r1; r += kCalThreads) {
        const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(r) * K + kb * 64);
        float v[64];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint4 q = __ldg(src + j);
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                v[8 * j + 2 * e] = __uint_as_float(w[e] << 16);
                v[8 * j + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
            }
        }
        if (s != nullptr && !after) {
#pragma unroll
            for (int i = 0; i < 64; ++i) v[i] = __fmul_rn(v[i], inv[i]);
        }
        if (rotate & 1) {
#pragma unroll
            for (int h = 1; h < 64; h <<= 1)
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    if ((i & h) == 0) {
                        const float a = v[i], b = v[i + h];
                        v[i] = __fadd_rn(a, b);
                        v[i + h] = __fsub_rn(a, b);
                    }
#pragma unroll
            for (int i = 0; i < 64; ++i) v[i] = __fmul_rn(v[i], 0.125f);
            if (s != nullptr && after) {
#pragma unroll
                for (int i = 0; i < 64; ++i) v[i] = __fmul_rn(v[i], inv[i]);
            }
        }
#pragma unroll
        for (int i = 0; i < 64; ++i) {
            const double d = static_cast<double>(v[i]);
            acc[i] = __dadd_rn(acc[i], __dmul_rn(d, d));    // the square of an fp32 value is exact in fp64
        }
    }
    __shared__ double red[kCalThreads / 32][64];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
#pragma unroll
    for (int i = 0; i < 64; ++i) {
        double t = acc[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t = __dadd_rn(t, __shfl_xor_sync(0xFFFFFFFFu, t, o));
        if (lane == 0) red[warp][i] = t;
    }
    __syncthreads();
    if (threadIdx.x < 64) {
        double t = 0.0;
#pragma unroll
        for (int w = 0; w < kCalThreads / 32; ++w) t = __dadd_rn(t, red[w][threadIdx.x]);
        partial[static_cast<size_t>(g) * K + kb * 64 + threadIdx.x] = t;
    }
}

__global__ void energy_final_kernel(const double* __restrict__ partial, int groups, int K, int M,
                                    double* __restrict__ z) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= K) return;
    double t = 0.0;
    for (int g = 0; g < groups; ++g) t = __dadd_rn(t, partial[static_cast<size_t>(g) * K + c]);
    z[c] = M > 0 ? __ddiv_rn(t, static_cast<double>(M)) : 0.0;
}

__global__ void __launch_bounds__(kRankThreads) topk_flag_kernel(const double* __restrict__ z, int K, int n,
                                                                 uint8_t* __restrict__ flag) {
    extern __shared__ double zs[];
    for (int i = threadIdx.x; i < K; i += kRankThreads) zs[i] = z[i];
    __syncthreads();
    const int c = blockIdx.x * kRankThreads + threadIdx.x;
    if (c >= K) return;
    const double zc = zs[c];
    int above = 0;
    for (int i = 0; i < K; ++i) {
        const double zi = zs[i];
        above += (zi > zc || (zi == zc && i < c)) ? 1 : 0;
    }
    flag[c] = above < n ? 1 : 0;
}

__global__ void __launch_bounds__(kScanThreads) topk_compact_kernel(const uint8_t* __restrict__ flag, int K,
                                                                    int32_t* __restrict__ omega) {
    __shared__ int counts[kScanThreads];
    const int per = (K + kScanThreads - 1) / kScanThreads;
    const int lo = threadIdx.x * per, hi = min(K, lo + per);
    int cnt = 0;
    for (int c = lo; c < hi; ++c) cnt += flag[c];
    counts[threadIdx.x] = cnt;
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int t = 0; t < kScanThreads; ++t) {
            const int c = counts[t];
            counts[t] = run;
            run += c;
        }
    }
    __syncthreads();
    int pos = counts[threadIdx.x];
    for (int c = lo; c < hi; ++c)
        if (flag[c]) omega[pos++] = c;
}

size_t calib_groups(int M) { return static_cast<size_t>((M + kRowsPerGroup - 1) / kRowsPerGroup); }

}  // namespace
}  // namespace wq

extern "C" WQ_API size_t wq_calibration_workspace_bytes(int M, int K) {
    if (M <= 0 || K <= 0) return 0;
    const size_t part = wq::calib_groups(M) * static_cast<size_t>(K) * 8;
    return (part + 1023) / 1024 * 1024 + (static_cast<size_t>(K) + 1023) / 1024 * 1024;
}

extern "C" WQ_API wq_status wq_calibrate_outliers(const void* x, int M, int K, const float* s, int rotate,
                                                  int transform_order, int n_top, double* z, int32_t* omega,
                                                  void* workspace, size_t workspace_bytes, void* stream) {
    using namespace wq;
    if (!x || !z || (n_top > 0 && !omega) || !workspace) {
        set_last_error("wq_calibrate_outliers: NULL buffer");
        return WQ_ERR_INVALID;
    }
    if (M <= 0 || K <= 0 || n_top < 0 || n_top > K || (rotate != 0 && rotate != 1) ||
        (transform_order != WQ_ORDER_SMOOTH_ROTATE && transform_order != WQ_ORDER_ROTATE_SMOOTH)) {
        set_last_error("wq_calibrate_outliers: bad size or option");
        return WQ_ERR_INVALID;
    }
    if (K % 64 || K > 16384) {
        set_last_error("wq_calibrate_outliers: K must be a multiple of 64 and <= 16384");
        return WQ_ERR_UNSUPPORTED;
    }
    if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(workspace) & 255) ||
        (reinterpret_cast<uintptr_t>(z) & 7) || (reinterpret_cast<uintptr_t>(s) & 3)) {
        set_last_error("wq_calibrate_outliers: x 16-byte, z 8-byte, s 4-byte and the workspace 256-byte aligned");
        return WQ_ERR_INVALID;
    }
    if (workspace_bytes < wq_calibration_workspace_bytes(M, K)) {
        set_last_error("wq_calibrate_outliers: workspace too small");
        return WQ_ERR_INVALID;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int groups = static_cast<int>(calib_groups(M));
    double* partial = static_cast<double*>(workspace);
    uint8_t* flag = static_cast<uint8_t*>(workspace) + (static_cast<size_t>(groups) * K * 8 + 1023) / 1024 * 1024;
    const int rot = rotate | (rotate && transform_order == WQ_ORDER_ROTATE_SMOOTH ? 2 : 0);
    energy_partial_kernel<<<dim3(K / 64, groups), kCalThreads, 0, st>>>(static_cast<const uint16_t*>(x), M, K, s, rot,
                                                                        partial);
    energy_final_kernel<<<(K + 255) / 256, 256, 0, st>>>(partial, groups, K, M, z);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess && n_top > 0) {
        static bool attr = false;
        if (!attr) {
            e = cudaFuncSetAttribute(topk_flag_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 16384 * 8);
            attr = e == cudaSuccess;
        }
        if (e == cudaSuccess) {
            topk_flag_kernel<<<(K + kRankThreads - 1) / kRankThreads, kRankThreads, static_cast<size_t>(K) * 8, st>>>(
                z, K, n_top, flag);
            topk_compact_kernel<<<1, kScanThreads, 0, st>>>(flag, K, omega);
            e = cudaGetLastError();
        }
    }
    if (e != cudaSuccess) {
        set_last_error((std::string("wq_calibrate_outliers: ") + cudaGetErrorString(e)).c_str());
        return WQ_ERR_CUDA;
    }
    return WQ_OK;
}
