// Allocation-free staged loopback all-reduce: the staged comparator with its
// workspace in a file-scope device array instead of caller memory.
//
// Who needs it: callers that cannot call cudaMalloc -- code running while a
// stream is captured into a CUDA graph, and runtimes whose device memory is
// owned by their own allocator or reserved up front. They still pass the
// arenas; the stack rows live in the array below.
#include <atomic>
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "detfold.h"

namespace detfold {
int record_cuda_status(cudaError_t e);
}

namespace {

// The scratch: DETFOLD_NOALLOC_SCRATCH_BYTES on every device that loads the
// library, held until the process exits. Shared by every call.
static __device__ __align__(256) unsigned char g_noalloc_scratch[DETFOLD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup;
std::atomic<void *> g_scratch_addr[kMaxDevices];

// Device address of the array on the current device, looked up once per
// device with that device current. In host code the array's name is only a
// host-side stand-in, so every device access goes through this address.
int scratch_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return detfold::record_cuda_status(e);
    if (dev < 0 || dev >= kMaxDevices) return detfold::record_cuda_status(cudaErrorInvalidDevice);
    void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        std::lock_guard<std::mutex> lock(g_setup);
        p = g_scratch_addr[dev].load(std::memory_order_acquire);
        if (!p) {
            e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess) return detfold::record_cuda_status(e);
            if (!p) return detfold::record_cuda_status(cudaErrorInvalidSymbol);
            g_scratch_addr[dev].store(p, std::memory_order_release);
        }
    }
    *out = p;
    return DETFOLD_OK;
}

}  // namespace

extern "C" int detfold_loopback_allreduce_staged_noalloc(float *const *arenas, int W, int64_t len,
                                                         float mean_scale, int flags, void *stream)
{
    const int64_t need = detfold_staged_workspace_bytes(len, W);
    if (need < 0) return (int)need;  // invalid W or len
    void *ws = nullptr;
    if (W > 1 && len > 0) {
        if (need > DETFOLD_NOALLOC_SCRATCH_BYTES) return DETFOLD_ERR_SCRATCH_LIMIT;
        if (int rc = scratch_address(&ws)) return rc;
    }
    return detfold_loopback_allreduce_staged_ex(arenas, W, len, mean_scale, flags, ws,
                                                DETFOLD_NOALLOC_SCRATCH_BYTES, stream);
}
