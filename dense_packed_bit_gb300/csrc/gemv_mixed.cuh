// gemv_mixed.cuh -- exact 2-bit field decode for the SIMT GEMV kernels, on the
// mixed-precision FMA (fp16 inputs, fp32 accumulator).
//
// A 32-bit code word holds 16 fields, field f at bits 2f.  One LOP3 keeps two
// of them, at bits q and 16 + q with q <= 8, and the two 16-bit halves of the
// result, read as fp16, are the subnormals c 2^(q-24) (fields 5-7 and 13-15 take
// the word shifted right by 10 first).  fma.rn.f32.f16 multiplies each half by
// its field's fp16 x into an fp32 accumulator of class q / 2: the product
// c x 2^(q-24) has at most 13 significant bits and is exact.  At the end the
// five classes are scaled by 2^(24-q) (exact) and added.  Scaling every field
// by a constant (all fields 1: sum x; all fields 2: 2 sum x) scales every
// product, every accumulator and the total exactly.
#pragma once

#include <cstdint>

namespace mm {

// acc += lo(m) x_lo + hi(m) x_hi: m holds two fields as fp16 subnormals; xl / xh are the fp16
// pairs holding the low and the high field's x, SL / SH name the half of each ("p0"/"p1" of xl,
// "r0"/"r1" of xh).
#define MIX2(acc, m, xl, xh, SL, SH)                  \
    asm("{\n\t.reg .b16 a0, a1, p0, p1, r0, r1;\n\t" \
        "mov.b32 {a0, a1}, %1;\n\t"                  \
        "mov.b32 {p0, p1}, %2;\n\t"                  \
        "mov.b32 {r0, r1}, %3;\n\t"                  \
        "fma.rn.f32.f16 %0, a0, " SL ", %0;\n\t"     \
        "fma.rn.f32.f16 %0, a1, " SH ", %0;\n\t}"    \
        : "+f"(acc)                                   \
        : "r"(m), "r"(xl), "r"(xh))

// 16 fields of word w (field f at bits 2f) against x[f] (X[j] = fp16 pair x[2j], x[2j+1]):
// pairs (f, f + 8); classes q = 0, 2, 4, 6, 8 -> acc[0..4]
__device__ __forceinline__ void word_mixed(uint32_t w, const uint32_t (&X)[8], float (&acc)[5]) {
    const uint32_t ws = w >> 10;
    MIX2(acc[0], w & 0x00030003u, X[0], X[4], "p0", "r0");   // f0 (q 0), f8
    MIX2(acc[1], w & 0x000C000Cu, X[0], X[4], "p1", "r1");   // f1 (q 2), f9
    MIX2(acc[2], w & 0x00300030u, X[1], X[5], "p0", "r0");   // f2 (q 4), f10
    MIX2(acc[3], w & 0x00C000C0u, X[1], X[5], "p1", "r1");   // f3 (q 6), f11
    MIX2(acc[4], w & 0x03000300u, X[2], X[6], "p0", "r0");   // f4 (q 8), f12
    MIX2(acc[0], ws & 0x00030003u, X[2], X[6], "p1", "r1");  // f5 (q 0), f13
    MIX2(acc[1], ws & 0x000C000Cu, X[3], X[7], "p0", "r0");  // f6 (q 2), f14
    MIX2(acc[2], ws & 0x00300030u, X[3], X[7], "p1", "r1");  // f7 (q 4), f15
}

__device__ __forceinline__ float mixed_total(const float (&acc)[5]) {
    return acc[0] * 16777216.0f + acc[1] * 4194304.0f + acc[2] * 1048576.0f + acc[3] * 262144.0f +
           acc[4] * 65536.0f;
}

}  // namespace mm
