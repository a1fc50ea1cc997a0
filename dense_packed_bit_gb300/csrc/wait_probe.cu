// wait_probe.cu -- failure-detection probe for the bounded device waits (sm_103a).
//
// Every pipelined kernel of the library waits on mbarriers through
// mbar_wait_limit (mm_common.cuh) with a limit of kWaitLimitNs; a wait that runs
// out records a code in its translation unit's device error word, the kernel
// returns instead of trapping, and mm_check_device_error reports MM_ERR_TIMEOUT.
// This kernel exercises that path without breaking any computing kernel: one
// warp initialises an mbarrier that expects a single arrival and waits on its
// first phase through the same helper with a short caller-chosen limit.  When
// asked to arrive first, the phase completes and the wait returns at once; when
// not, nothing can complete the phase, the wait runs out after the limit, and
// the kernel records kDevErrProbe and returns.  The wait ends in both cases:
// it is bounded by %globaltimer, and the host accepts limits of at most 0.1 s.
#include "mm_common.cuh"
#include "mm_internal.h"

namespace mm {

__device__ unsigned int g_probe_err;

__global__ void __launch_bounds__(32) wait_probe_kernel(int arrive, unsigned long long limit_ns,
                                                        unsigned long long *out) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x != 0) return;
    if (arrive) mbar_arrive(&bar);
    const unsigned long long t0 = global_ns();
    const bool done = mbar_wait_limit(&bar, 0, limit_ns);
    const unsigned long long t1 = global_ns();
    if (!done) atomicExch(&g_probe_err, kDevErrProbe);
    if (out) {
        out[0] = done ? 1ull : 0ull;
        out[1] = t1 - t0;
    }
}

cudaError_t launch_wait_probe(int arrive, unsigned long long limit_ns, unsigned long long *out, cudaStream_t s) {
    wait_probe_kernel<<<1, 32, 0, s>>>(arrive, limit_ns, out);
    return cudaGetLastError();
}

unsigned int wait_probe_take_device_error(cudaError_t *err) {
    unsigned int v = 0;
    *err = cudaMemcpyFromSymbol(&v, g_probe_err, sizeof(v));
    if (*err == cudaSuccess && v != 0) {
        const unsigned int zero = 0;
        *err = cudaMemcpyToSymbol(g_probe_err, &zero, sizeof(zero));
    }
    return v;
}

}  // namespace mm
