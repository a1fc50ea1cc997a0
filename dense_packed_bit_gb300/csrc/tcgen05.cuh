// tcgen05.cuh -- 5th-generation tensor core helpers for sm_103a (inline PTX).
//
// Tensor memory (TMEM) allocation, the shared-memory matrix descriptors and
// instruction descriptors that tcgen05.mma reads, single-thread MMA issue with
// completion reported on an mbarrier (tcgen05.commit), and TMEM -> register
// loads for the epilogue.
//
// Operand layout used throughout: K-major tiles with the 128-byte swizzle --
// rows of 128 bytes along K, groups of 8 rows (1024 bytes) stacked along M/N,
// the 16-byte chunk j of row r stored at chunk j ^ (r % 8).  This is the layout
// a TMA tile load with CU_TENSOR_MAP_SWIZZLE_128B writes, and the one the
// kernels write themselves when they build an operand in shared memory.
#pragma once

#include "mm_common.cuh"

namespace mm {

// ---------------------------------------------------------------- TMEM

// Allocate `ncols` TMEM columns (power of two, >= 32); the whole warp executes
// this and the base address is written to *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Make generic-proxy shared-memory writes visible to the async proxy (MMA / TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- descriptors

// Shared-memory matrix descriptor for a K-major operand with the 128-byte
// swizzle: start address (>> 4) in bits 0-13, leading byte offset (unused for
// this layout, encoded as 1) in bits 16-29, stride byte offset (1024: the
// distance between 8-row groups) in bits 32-45, descriptor version 1 in bits
// 46-47, swizzle mode 2 (128-byte) in bits 61-63.  The operand base must be
// 1024-byte aligned; advancing the start address by 32 bytes steps K by 32
// bytes inside the swizzled rows.
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Swizzle-mode codes of the shared-memory descriptor (bits 61-63).
constexpr uint32_t kSdescSw128 = 2, kSdescSw64 = 4, kSdescSw32 = 6;

// General shared-memory matrix descriptor: start address, leading and stride
// byte offsets, swizzle mode.  For a K-major swizzled operand the stride byte
// offset is the distance between 8-row groups along M/N and the leading one is
// unused (encoded as 16 bytes).
__device__ __forceinline__ uint64_t sdesc_make(uint32_t smem_addr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                               uint32_t swizzle) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)swizzle << 61;
    return d;
}

// Instruction descriptor: D format in bits 4-5 (1 = f32), A and B formats in
// bits 7-9 and 10-12 (kind::f16: 0 = f16, 1 = bf16; kind::tf32: 2 = tf32),
// A / B major-ness in bits 15 / 16 (0 = K-major), N >> 3 in bits 17-22,
// M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t make_idesc(uint32_t a_fmt, uint32_t b_fmt, uint32_t N, uint32_t M) {
    return (1u << 4) | (a_fmt << 7) | (b_fmt << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

constexpr uint32_t kFmtF16 = 0, kFmtBF16 = 1, kFmtTF32 = 2;


// ---------------------------------------------------------------- MMA

// D[tmem] (+)= A[smem] * B[smem]^T, one CTA, kind::f16 (f16/bf16 operands).
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Same for kind::tf32 (fp32 containers, the MMA reads the top 19 bits).
__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// ---------------------------------------------------------------- CTA pairs (cta_group::2)
//
// A pair of CTAs in one cluster of 2 runs one M = 256 MMA: each CTA holds its
// 128 rows of A and half of the N columns of B at the same shared-memory
// offsets, and its own 128 lanes of the accumulator in its tensor memory.
// Allocation and release are done by one warp in each CTA of the pair; the
// MMAs are issued by one thread of the even CTA; completion is signalled on
// the mbarrier at the same offset in every CTA of `mask`.

__device__ __forceinline__ void tmem_alloc_pair(uint32_t *slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void umma_tf32_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit_pair(uint64_t *bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(mask)
        : "memory");
}

// ---------------------------------------------------------------- TMEM -> registers

// Each thread of the warp reads 32 consecutive fp32 columns of its TMEM lane
// (lane = the warp's 32-lane quarter + thread index).  The wait for the load
// is part of the same asm statement, so the registers are never read early.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace mm
