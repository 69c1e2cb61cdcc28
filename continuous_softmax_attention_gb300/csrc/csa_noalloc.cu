// Scratch memory of csa_decode_noalloc: a file-scope device array, so that
// the entry point allocates nothing.  It sits in a translation unit of its
// own, so that with lazy module loading only a process that calls
// csa_decode_noalloc loads it and holds its CSA_DECODE_NOALLOC_SCRATCH_BYTES
// on the device; csa_decode and the other entry points never touch it.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "csa.h"
#include "csa_internal.h"

static __device__ __align__(256) float g_noalloc_scratch[CSA_DECODE_NOALLOC_SCRATCH_BYTES / 4];

namespace {

constexpr int kMaxDevices = 64;

// The host-side name of the array is not a device address: the device copy's
// address is looked up with cudaGetSymbolAddress, with the device current.
// It is kept per device together with the CUDA context it was taken in; a
// device reset makes a new primary context, whose address is looked up
// again on the next call.
struct NoallocEntry {
    CUcontext ctx = nullptr;
    void *addr = nullptr;
};
std::mutex g_mutex;
NoallocEntry g_entry[kMaxDevices];

PFN_cuCtxGetCurrent_v4000 ctx_get_current_fn() {
    static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 4000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(ptr);
    });
    return fn;
}

}  // namespace

int csa_decode_noalloc_scratch(void **addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CSA_ERR_NO_DEVICE;
    if (dev < 0 || dev >= kMaxDevices) return CSA_ERR_UNSUPPORTED;
    auto get_ctx = ctx_get_current_fn();
    if (!get_ctx) return CSA_ERR_CUDA;
    CUcontext ctx = nullptr;
    if (get_ctx(&ctx) != CUDA_SUCCESS) return CSA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    NoallocEntry &e = g_entry[dev];
    if (ctx == nullptr || e.addr == nullptr || e.ctx != ctx) {
        void *p = nullptr;
        // dev is the current device here, so the address is that device's
        // copy (the runtime makes the device's primary context current first
        // if no context is)
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return CSA_ERR_CUDA;
        if (get_ctx(&ctx) != CUDA_SUCCESS || !ctx) return CSA_ERR_CUDA;
        e.addr = p;
        e.ctx = ctx;
    }
    *addr = e.addr;
    return CSA_OK;
}
