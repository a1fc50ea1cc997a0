// tf32x3_split.cuh -- the operand split of the 3xTF32 tensor-core GEMMs (Ootomo and
// Yokota, IJHPCA 2022): a = a_hi + a_lo with a_hi the fp32 value with its 13 low
// mantissa bits cleared (what a kind::tf32 MMA reads from a raw fp32 container) and
// a_lo = a - a_hi, exact.  Operand tiles are K-major with the 64-byte swizzle: rows
// of 16 fp32 along K, 16-byte chunk c of row r at chunk c ^ ((r >> 1) & 3), 8-row
// groups 512 bytes apart.  Shared by gemm_tf32x3_ws.cu and gemm_skinny_tc.cu.
#pragma once

#include "mm_common.cuh"

namespace mm {
namespace tf32x3 {

constexpr int BK = 16;  // fp32 of K per staged slab: one 64-byte swizzled row

__device__ __forceinline__ float lo_part(float a) {
    return __fsub_rn(a, __uint_as_float(__float_as_uint(a) & 0xFFFFE000u));
}

__device__ __forceinline__ float4 lo_part4(float4 v) {
    return make_float4(lo_part(v.x), lo_part(v.y), lo_part(v.z), lo_part(v.w));
}

// K-contiguous operand (BYTES of raw tile in the operand layout, which is its hi tile):
// the lo tile at the same offsets.  NT threads, thread index ct.
template <int BYTES, int NT>
__device__ __forceinline__ void lo_in_place_layout(const uint8_t *raw, uint8_t *lo, int ct) {
    constexpr int N4 = BYTES / 16, R = (N4 + NT - 1) / NT;
    float4 v[R];
#pragma unroll
    for (int i = 0; i < R; ++i)
        if (N4 % NT == 0 || ct + i * NT < N4) v[i] = *reinterpret_cast<const float4 *>(raw + (ct + i * NT) * 16);
#pragma unroll
    for (int i = 0; i < R; ++i)
        if (N4 % NT == 0 || ct + i * NT < N4) *reinterpret_cast<float4 *>(lo + (ct + i * NT) * 16) = lo_part4(v[i]);
}

// K-contiguous operand copied out of its landing buffer: hi = raw and lo at the same
// offsets in other tiles, so that the raw buffer can be refilled at once.
template <int BYTES, int NT>
__device__ __forceinline__ void split_same_layout(const uint8_t *raw, uint8_t *hi, uint8_t *lo, int ct) {
    constexpr int N4 = BYTES / 16, R = (N4 + NT - 1) / NT;
    float4 v[R];
#pragma unroll
    for (int i = 0; i < R; ++i)
        if (N4 % NT == 0 || ct + i * NT < N4) v[i] = *reinterpret_cast<const float4 *>(raw + (ct + i * NT) * 16);
#pragma unroll
    for (int i = 0; i < R; ++i)
        if (N4 % NT == 0 || ct + i * NT < N4) {
            *reinterpret_cast<float4 *>(hi + (ct + i * NT) * 16) = v[i];
            *reinterpret_cast<float4 *>(lo + (ct + i * NT) * 16) = lo_part4(v[i]);
        }
}

// K-contiguous operand landed as unswizzled rows of PITCH fp32 (PITCH / 16 slabs side by
// side): slab j (fp32 16 j .. 16 j + 15 of every row) -> K-major swizzled hi and lo tiles.
// With PITCH = 16 an 8-lane phase of the 16-byte reads covers two consecutive 64-byte rows
// (conflict-free); wider rows put its two rows on the same banks (two-way conflicts).  The
// stores are conflict-free.  NT threads, thread index ct.
template <int ROWS, int PITCH, int NT>
__device__ __forceinline__ void split_rows(const uint8_t *raw, int j, uint8_t *hi, uint8_t *lo, int ct) {
    constexpr int TASKS = ROWS * (BK / 4), R = (TASKS + NT - 1) / NT;
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const int idx = ct + i * NT;
        if (TASKS % NT != 0 && idx >= TASKS) break;
        const int r = idx >> 2, c = idx & 3;
        const float4 v = *reinterpret_cast<const float4 *>(raw + r * PITCH * 4 + j * 64 + c * 16);
        const int off = r * 64 + ((c ^ ((r >> 1) & 3)) << 4);
        *reinterpret_cast<float4 *>(hi + off) = v;
        *reinterpret_cast<float4 *>(lo + off) = lo_part4(v);
    }
}

// M/N-contiguous operand: raw [k][r] (BK rows of ROWS fp32, unswizzled) -> K-major
// swizzled hi and lo tiles.  A warp covers 32 consecutive r: each column read is one
// 128-byte row segment and each 8-lane phase of the 16-byte stores hits 8 distinct
// bank groups.  NT threads, thread index ct.
template <int ROWS, int NT>
__device__ __forceinline__ void split_transpose(const uint8_t *raw, uint8_t *hi, uint8_t *lo, int ct) {
    const float *src = reinterpret_cast<const float *>(raw);
    constexpr int TASKS = ROWS * (BK / 4), R = (TASKS + NT - 1) / NT;
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const int idx = ct + i * NT;
        if (TASKS % NT != 0 && idx >= TASKS) break;
        const int r = idx % ROWS, c = idx / ROWS;
        const float4 v = make_float4(src[(4 * c + 0) * ROWS + r], src[(4 * c + 1) * ROWS + r],
                                     src[(4 * c + 2) * ROWS + r], src[(4 * c + 3) * ROWS + r]);
        const int off = r * 64 + ((c ^ ((r >> 1) & 3)) << 4);
        *reinterpret_cast<float4 *>(hi + off) = v;
        *reinterpret_cast<float4 *>(lo + off) = lo_part4(v);
    }
}

}  // namespace tf32x3
}  // namespace mm
