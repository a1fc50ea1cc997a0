// gemm_splitk_static.cu -- the library's own scratch for the split-K GEMM entry
// point that allocates nothing (mm_gemm_f32_splitk_noalloc).
//
// Some callers cannot call cudaMalloc, or pass a workspace, at the point where
// they multiply: their device memory is owned by another allocator (a
// framework's caching pool that has reserved the memory it manages), or they run
// on a path where cudaMalloc's implicit device-wide synchronisation is not
// acceptable.  For them the split-K partial tiles go to this file-scope array
// instead of a caller-provided workspace.  Every GPU that loads the library holds
// the array until the process exits.
//
// In host code `g_splitk_scratch` names a host-side stand-in, not a device
// address; its device address is looked up here with cudaGetSymbolAddress, once
// per device, with that device current, and cached.
#include "mm_internal.h"

#include <cuda_runtime.h>

#include <mutex>

namespace mm {

static __device__ __align__(256) float g_splitk_scratch[kSplitkStaticFloats];

cudaError_t splitk_static_scratch(float **ptr, int64_t *floats) {
    static std::mutex mu;
    static float *addr[64] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_splitk_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = static_cast<float *>(p);
    }
    *ptr = addr[dev];
    *floats = kSplitkStaticFloats;
    return cudaSuccess;
}

}  // namespace mm
