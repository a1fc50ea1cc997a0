// mm_common.cuh -- device helpers shared by the libmm kernels (sm_103a).
//
// Inline PTX for mbarriers, TMA tile loads, programmatic dependent launch and
// streaming global loads.  Every wait here is bounded by wall-clock time read
// from %globaltimer; a wait that runs out records an error code in the calling
// translation unit's device error word and reports failure to its caller,
// which then returns without trapping.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace mm {

// Upper bound of any single device-side wait (nanoseconds).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

// Error codes written to a translation unit's device error word.
enum : unsigned int {
    kDevErrNone = 0,
    kDevErrWaitFull = 1,    // consumer wait for a filled pipeline stage ran out
    kDevErrWaitEmpty = 2,   // producer wait for a drained stage ran out
    kDevErrWaitMma = 3,     // wait for tensor-core completion ran out
    kDevErrDrain = 4,       // wait for in-flight copies after an error ran out
    kDevErrProbe = 5        // the failure-detection probe's wait ran out (as asked)
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// The dynamic shared-memory base rounded up to ALIGN bytes.  The result is formed
// by pointer arithmetic on the shared array itself (not by a round trip through an
// integer), so the compiler still knows every pointer derived from it addresses
// shared memory and emits shared loads and stores with 32-bit addresses.
template <int ALIGN>
__device__ __forceinline__ uint8_t *smem_aligned(uint8_t *raw) {
    const uint32_t a = smem_u32(raw);
    return raw + ((ALIGN - (a & (ALIGN - 1))) & (ALIGN - 1));
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait until the barrier phase with the given parity completes, for at most
// limit_ns.  Returns false when the limit ran out.
__device__ __forceinline__ bool mbar_wait_limit(uint64_t *bar, uint32_t parity, unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
}

// mbar_wait_limit with the kernels' limit, kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    return mbar_wait_limit(bar, parity, kWaitLimitNs);
}

// try_wait that lets the hardware suspend the thread for up to `suspend_ns` while the
// phase is incomplete (it resumes as soon as the phase completes), so waiting warps
// take no issue slots from the warps that compute.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t *bar, uint32_t parity, uint32_t suspend_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(suspend_ns)
        : "memory");
    return ok != 0;
}

// mbar_wait built on suspending tries: for waits that are long compared with the
// work of the other warps on the SM (whole tiles streaming in from HBM).
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait_suspend(bar, parity, 100000u)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait_suspend(bar, parity, 100000u))
        if (global_ns() - t0 > kWaitLimitNs) return false;
    return true;
}

// Named barrier over `nthreads` threads (a multiple of 32), id 1..15 (0 is __syncthreads).
__device__ __forceinline__ void bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- clusters

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every non-exited thread of every CTA in the cluster arrives, then waits.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The two halves of cluster_sync, for work between the arrival and the wait.
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Address of the same shared-memory location in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}

// Arrive on the mbarrier at a shared::cluster address (this CTA's or a peer's)
// with the instruction's default semantics.  Shared-memory operands written
// before it for a peer's tensor-core MMA are first made visible to the async
// proxy (fence.proxy.async); an explicit cluster-scope release here measured
// about twice as slow for the whole GEMM pipeline on GB300.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

__device__ __forceinline__ float4 ld_cluster_v4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// ---------------------------------------------------------------- TMA

// 2-D tiled bulk tensor load into this CTA's shared memory, completion
// reported as transaction bytes on `bar`.  c0 is the innermost coordinate.
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const void *tmap, uint64_t *bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(tmap), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

// 3-D form of tma_load_2d (c2: the outermost coordinate, e.g. the matrix of a batch).
__device__ __forceinline__ void tma_load_3d(void *smem_dst, const void *tmap, uint64_t *bar, int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(tmap), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// 2-D tiled bulk tensor store from this CTA's shared memory (the box in the tensor map's
// layout and swizzle) to global memory; parts of the box outside the tensor are not
// written.  Completion is tracked by the issuing thread's bulk async-groups.
__device__ __forceinline__ void tma_store_2d(const void *tmap, const void *smem_src, int c0, int c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(tmap),
                 "r"(smem_u32(smem_src)), "r"(c0), "r"(c1)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until this thread's committed bulk groups have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Wait until this thread's committed bulk groups have completed (writes performed).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// 1-D bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from
// global into this CTA's shared memory, completion reported on `bar`.
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gsrc, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(smem_dst)), "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from this
// CTA's shared memory to shared memory of a CTA of the cluster (shared::cluster
// addresses of the destination and of its mbarrier), completion reported there
// as transaction bytes.
__device__ __forceinline__ void bulk_copy_to_cluster(uint32_t dst_cluster, const void *src, uint32_t bytes,
                                                     uint32_t bar_cluster) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst_cluster), "r"(smem_u32(src)), "r"(bytes), "r"(bar_cluster)
                 : "memory");
}

// Wait until every bulk copy this thread committed has finished reading its source.
__device__ __forceinline__ void bulk_commit_and_wait_read() {
    asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// ---------------------------------------------------------------- PDL

// Block until every grid this one depends on has completed and its writes
// are visible.  A no-op when the grid was not launched as a dependent.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the next dependent grid in the stream to begin launching.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- loads

// 16-byte read-only load that bypasses L1 allocation (streamed weights).
__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// ---------------------------------------------------------------- packed fp32 pairs

// d = a * b + c on two fp32 lanes at once (sm_100+ packed f32x2 FMA), round to nearest.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    unsigned long long A, B, C, D;
    A = *reinterpret_cast<unsigned long long *>(&a);
    B = *reinterpret_cast<unsigned long long *>(&b);
    C = *reinterpret_cast<unsigned long long *>(&c);
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(D) : "l"(A), "l"(B), "l"(C));
    return *reinterpret_cast<float2 *>(&D);
}

// (d0, d1) += a * (b0, b1): two independent fp32 FMAs, each rounded once, in one packed
// f32x2 instruction (half the issue slots of two FFMAs; the same bits)
__device__ __forceinline__ void fma2_bcast(float &d0, float &d1, float a, float b0, float b1) {
    unsigned long long A, B, D;
    asm("mov.b64 %0, {%1, %1};" : "=l"(A) : "r"(__float_as_uint(a)));
    asm("mov.b64 %0, {%1, %2};" : "=l"(B) : "r"(__float_as_uint(b0)), "r"(__float_as_uint(b1)));
    asm("mov.b64 %0, {%1, %2};" : "=l"(D) : "r"(__float_as_uint(d0)), "r"(__float_as_uint(d1)));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(D) : "l"(A), "l"(B));
    unsigned lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(D));
    d0 = __uint_as_float(lo);
    d1 = __uint_as_float(hi);
}

}  // namespace mm
