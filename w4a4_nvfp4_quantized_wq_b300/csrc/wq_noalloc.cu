// wq_noalloc.cu -- wq_linear_forward_noalloc: the forward for callers that cannot allocate
// device memory (a plugin inside a host engine that owns all allocations, a real-time
// control loop that forbids allocation after start-up).  Its scratch is one static device
// array of WQ_NOALLOC_SCRATCH_BYTES; the library allocates nothing on this path.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "wq_internal.h"

namespace {

constexpr size_t kScratchBytes = WQ_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 256;

// Shared by every call on a device; it keeps the previous call's contents.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};   // device address of g_noalloc_scratch per device

}  // namespace

extern "C" WQ_API wq_status wq_linear_forward_noalloc(wq_weights_t h, const void* x, int M, void* y,
                                                      void* stream) {
    if (!h) {
        wq::set_last_error("NULL handle");
        return WQ_ERR_INVALID;
    }
    if (M < 0) {
        wq::set_last_error("M < 0");
        return WQ_ERR_INVALID;
    }
    const size_t need = wq_workspace_bytes(h, M);
    if (need > kScratchBytes) {
        const std::string msg = "wq_linear_forward_noalloc: M = " + std::to_string(M) + " needs " +
                                std::to_string(need) + " bytes of scratch, more than the static " +
                                std::to_string(kScratchBytes) + "-byte array; use wq_linear_forward";
        wq::set_last_error(msg.c_str());
        return WQ_ERR_UNSUPPORTED;
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        wq::set_last_error("wq_linear_forward_noalloc: cannot determine the current device");
        return WQ_ERR_CUDA;
    }
    // the scratch must be the copy on the handle's device, where the kernels run
    if (dev != wq::handle_device(h)) {
        wq::set_last_error("wq_linear_forward_noalloc: the current device is not the handle's device");
        return WQ_ERR_INVALID;
    }
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_scratch_addr[dev]) {
            // one-time set-up per device, with that device current
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess || !p) {
                const std::string msg = std::string("cudaGetSymbolAddress failed: ") + cudaGetErrorString(e);
                wq::set_last_error(msg.c_str());
                return WQ_ERR_CUDA;
            }
            g_scratch_addr[dev] = p;
        }
        scratch = g_scratch_addr[dev];
    }
    return wq_linear_forward(h, x, M, y, scratch, kScratchBytes, stream);
}
