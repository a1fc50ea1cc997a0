// gemv_mma.cuh -- pieces shared by the tensor-core GEMV kernels: the
// m16n8k16 MMA, the exact fp16 encodings of 2-bit fields and the per-slot
// scales.  See gemv_packed2_mma.cu for the encoding.
#pragma once

#include "mm_common.cuh"

#include <cuda_fp16.h>

namespace mm {
namespace gemv_mma {

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t hmul2_bits(uint32_t x, uint32_t m) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(m));
    return r;
}

__host__ __device__ constexpr int slot_p(int s) { return s < 5 ? 2 * s : 2 * (s - 5); }
__host__ __device__ constexpr uint32_t slot_mask(int s) { return (3u << slot_p(s)) | (3u << (16 + slot_p(s))); }
// A operand of the "every field = 1" MMAs: fp16x2 of 2^(p-24) (subnormal) or 2^(p-10) (normal)
__host__ __device__ constexpr uint32_t slot_ones(int s, bool norm) {
    return norm ? (((uint32_t)(5 + slot_p(s)) << 10) | ((uint32_t)(5 + slot_p(s)) << 26))
                : ((1u << slot_p(s)) | (1u << (16 + slot_p(s))));
}

__device__ __forceinline__ uint32_t hsub2_one(uint32_t h) {  // h - (1, 1), exact here
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x3C003C00u));
    return r;
}

// A operand for one slot of a word: exact fp16x2 of (c_lo, c_hi) * 2^(p-24) (subnormal) or,
// with the 1.0 exponent or'ed in and 1 subtracted, (c_lo, c_hi) * 2^(p-10) (normal).
template <bool NORM>
__device__ __forceinline__ uint32_t slot_operand(uint32_t w, uint32_t m) {
    if (NORM) return hsub2_one((w & m) | 0x3C003C00u);
    return w & m;
}

__device__ __forceinline__ float h2f(uint16_t h) { return __half2float(__ushort_as_half(h)); }

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// 2^(24 - p) (subnormal encoding) or 2^(10 - p) (normal) for the slot held in output column n
template <bool NORM>
__device__ __forceinline__ float col_scale(int n) {
    const int p = n < 5 ? 2 * n : 2 * (n - 5);
    return __int_as_float((127 + (NORM ? 10 : 24) - p) << 23);
}

}  // namespace gemv_mma
}  // namespace mm
