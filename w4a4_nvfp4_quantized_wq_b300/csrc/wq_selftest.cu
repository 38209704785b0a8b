// wq_selftest.cu -- exercises the failure path that every kernel of the library relies on.
//
// Every barrier wait in the kernels is bounded: after WQ_WAIT_NS of global time it records a
// site code in the device error flag, raises the CTA's abort flag so that the CTA's other
// roles stop waiting too, and returns, so that a lost arrival ends as an error status on the
// host (wq_check_device_error -> WQ_ERR_TIMEOUT) with the context still usable.  This entry
// point makes such a wait run out on purpose -- an mbarrier that nothing arrives on -- without
// any fault, trap or endless loop.
#include <cuda_runtime.h>

#include <string>

#include "ptx.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int kSiteFirst = 91;     // the wait that runs out
constexpr int kSiteSecond = 92;    // the wait released by the abort flag (never recorded)
constexpr uint64_t kHeadStartNs = 500000000ull;   // the second wait starts 0.5 s later

__global__ void wait_timeout_kernel(int* err, int* released, unsigned long long* waited_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);            // one arrival expected; none is ever made
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    volatile int* af = &abort_flag;
    if (threadIdx.x == 0) {
        const uint64_t t0 = global_timer_ns();
        const bool ok = mbar_wait(b, 0, af, err, kSiteFirst);
        waited_ns[0] = global_timer_ns() - t0;
        if (!ok) atomicAdd(released, 1);
    } else if (threadIdx.x == 32) {
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < kHeadStartNs) {
        }
        // its own limit would end at 0.5 s + WQ_WAIT_NS; the first wait's abort comes earlier
        const bool ok = mbar_wait(b, 0, af, err, kSiteSecond);
        waited_ns[1] = global_timer_ns() - t0;
        if (!ok) atomicAdd(released, 1);
    }
    __syncthreads();
}

}  // namespace
}  // namespace wq

extern "C" WQ_API wq_status wq_selftest_wait_timeout(int* site, double* waited_ms, int* released) {
    if (!site || !waited_ms || !released) {
        wq::set_last_error("NULL output");
        return WQ_ERR_INVALID;
    }
    struct Buf {
        int err, released;
        unsigned long long waited[2];
    };
    Buf* d = nullptr;
    if (cudaMalloc(&d, sizeof(Buf)) != cudaSuccess) {
        wq::set_last_error("cudaMalloc failed");
        return WQ_ERR_OOM;
    }
    Buf hb{};
    cudaError_t e = cudaMemcpy(d, &hb, sizeof(Buf), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) {
        wq::wait_timeout_kernel<<<1, 64>>>(&d->err, &d->released, d->waited);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(&hb, d, sizeof(Buf), cudaMemcpyDeviceToHost);
    cudaFree(d);
    if (e != cudaSuccess) {
        wq::set_last_error((std::string("wait self-test: ") + cudaGetErrorString(e)).c_str());
        return WQ_ERR_CUDA;
    }
    *site = hb.err;
    *released = hb.released;
    waited_ms[0] = static_cast<double>(hb.waited[0]) * 1e-6;
    waited_ms[1] = static_cast<double>(hb.waited[1]) * 1e-6;
    if (hb.err == 0) return WQ_OK;   // the wait did not run out: the caller's check fails
    wq::set_last_error(("kernel barrier wait timed out (site " + std::to_string(hb.err) + ")").c_str());
    return WQ_ERR_TIMEOUT;
}
