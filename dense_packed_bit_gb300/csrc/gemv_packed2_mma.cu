// gemv_packed2_mma.cu -- 2-bit GEMV whose multiply-accumulate runs on the
// tensor cores (mma.sync m16n8k16, fp16 operands, fp32 accumulators).
//
// Why: the GEMV streams 4.5 MiB of codes ("Kernel 0112", "What is being
// measured"), but on the SIMT pipes it cannot keep up with HBM: every 2-bit
// field needs at least one integer instruction to become an fp32 operand, and
// the integer pipe issues 64 lanes/clk/SM against ~94 fields/clk/SM needed at
// the measured HBM bandwidth.  Here one LOP3 and one fp16x2 subtraction turn
// two fields into an exact half2, and the products and sums go to the tensor
// cores, which take their A operand straight from registers.
//
// Encoding.  In a 32-bit code word, field j sits at bits 2j..2j+1.  The mask
// (3 << p) | (3 << (16 + p)) keeps fields p/2 and 8 + p/2; or'ed with the fp16
// exponent of 1.0 in both halves this is the half2 (1 + c_lo 2^(p-10),
// 1 + c_hi 2^(p-10)) (p <= 8 keeps the field inside the 10-bit mantissa), and
// one fp16x2 subtraction of (1, 1) leaves (c_lo, c_hi) * 2^(p-10) exactly.
// Slots s = 0..4 use p = 2s on the word; slots 5..7 use p = 2(s-5) on the word
// shifted right by 10.  Slot s therefore carries fields s and s + 8.  (The
// masked word alone is the exact fp16 subnormal pair c * 2^(p-24), one
// instruction cheaper, but its products are not always accumulated exactly:
// all-zero-entry rows then failed to cancel to 0.)
//
// One MMA works on one slot: A = the slot's half2s of two words of rows g and
// g+8 per thread, B = the matching x values.  Each slot has its own power of
// two, so slot s writes only output column s: thread (g, t) supplies B column g
// and zeroes it (fp16 multiply by 0 or 1) unless g == s.  After the k loop the
// eight columns are scaled by 2^(10 - p_s) (exact) and summed across the quad.
//
// Affine codebooks (codebook[c] = c0 + c*d): the MMAs give S1 = sum c_k x_k;
// sum x_k comes from the same MMAs with every field equal to 1 (constant A),
// accumulated and reduced in exactly the same order, and
// y = scale * (c0 * sum x + d * S1).  When all fields of a row are the zero
// entry c_z in {0,1,2}, S1 is exactly c_z times sum x and the row returns 0.
//
// Layout: a warp owns RB blocks of 16 rows over a contiguous range of 256-field
// slabs; KW warps split a row's slabs and combine their partial sums through
// shared memory in a fixed order (no atomics, reproducible bit for bit).  Per
// slab, thread (g, t) loads the 16-byte chunk 4*slab + t of rows g and g + 8 of
// each row block: a quad reads 64 contiguous bytes of a row.  All of a warp's
// code loads (up to SB slabs) are issued before any arithmetic.
#include "gemv_mma.cuh"
#include "mm_common.cuh"
#include "mm_internal.h"

#include <cuda_fp16.h>

#include <mutex>

namespace mm {
namespace {

using namespace gemv_mma;

template <int RB, int KW, int SB, bool NORM>
__global__ void __launch_bounds__(RB == 1 ? 512 : 256) gemv2_mma_kernel(const PackedArgs a, const int prefetch) {
    extern __shared__ uint4 smem4[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int RW = nwarps / KW;
    const int rw = warp % RW, kw = warp / RW;
    const int g = lane >> 2, t = lane & 3;
    const int NS = (int)(a.cols >> 8);
    const int s_begin = (kw * NS) / KW, s_end = ((kw + 1) * NS) / KW;
    const int64_t rb0 = ((int64_t)blockIdx.x * RW + rw) * RB;
    const int64_t rowbytes = a.cols >> 2;

    uint4 *xw = smem4;                                                   // cols/2 half2
    float *red = reinterpret_cast<float *>(smem4 + (a.cols >> 3));      // [KW][RW][RB*16 + 1]

    uint4 q[SB][RB][2];
    auto load = [&](int j0) {
#pragma unroll
        for (int jj = 0; jj < SB; ++jj)
#pragma unroll
            for (int b = 0; b < RB; ++b)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int j = j0 + jj;
                    const int64_t row = (rb0 + b) * 16 + g + 8 * h;
                    if (j < s_end && row < a.rows)
                        q[jj][b][h] = ld_stream_v4(a.codes + row * rowbytes + (int64_t)(4 * j + t) * 16);
                    else
                        q[jj][b][h] = make_uint4(0u, 0u, 0u, 0u);
                }
    };

    if (prefetch >= 1) {
        load(s_begin);
        // chained calls: the next call may launch only once this one has passed its wait,
        // so at most one call runs ahead (its weight loads) instead of a queue of parked ones
        if (prefetch == 1) pdl_wait();
        pdl_launch_dependents();
    } else {
        pdl_wait();
        load(s_begin);
        pdl_launch_dependents();
    }

    // ---- x -> shared as xw[(chunk*8 + g)*4 + i] = (x[64c+16i+g], x[64c+16i+g+8]); every
    // load of a batch is issued before the first store
    {
        uint32_t *xw32 = reinterpret_cast<uint32_t *>(xw);
        const int ne = (int)(a.cols >> 1);
        constexpr int XB = 4;
        for (int e0 = threadIdx.x; e0 < ne; e0 += XB * blockDim.x) {
            uint16_t lo[XB], hi[XB];
#pragma unroll
            for (int u = 0; u < XB; ++u) {
                const int e = e0 + u * blockDim.x;
                if (e < ne) {
                    const int k = 64 * (e >> 5) + 16 * (e & 3) + ((e >> 2) & 7);
                    lo[u] = __ldg(a.x + k);
                    hi[u] = __ldg(a.x + k + 8);
                }
            }
#pragma unroll
            for (int u = 0; u < XB; ++u) {
                const int e = e0 + u * blockDim.x;
                if (e < ne) xw32[e] = (uint32_t)lo[u] | ((uint32_t)hi[u] << 16);
            }
        }
        __syncthreads();
    }

    // two accumulators per row block (slots of even / odd index) shorten the
    // MMA dependency chains; sum x uses the same split and order
    float d[RB][2][4];
#pragma unroll
    for (int b = 0; b < RB; ++b)
#pragma unroll
        for (int z = 0; z < 2; ++z) d[b][z][0] = d[b][z][1] = d[b][z][2] = d[b][z][3] = 0.f;
    float dx[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    uint32_t onehot[8];
#pragma unroll
    for (int s = 0; s < 8; ++s) onehot[s] = (g == s) ? 0x3C003C00u : 0u;  // fp16x2 (1, 1) or (0, 0)

    for (int j0 = s_begin; j0 < s_end; j0 += SB) {
        if (j0 > s_begin) load(j0);
#pragma unroll
        for (int jj = 0; jj < SB; ++jj) {
            const int j = j0 + jj;
            if (j >= s_end) break;
            const uint4 xv = xw[(4 * j + t) * 8 + g];
#pragma unroll
            for (int wp = 0; wp < 2; ++wp) {
                const uint32_t xa = word_of(xv, 2 * wp), xb = word_of(xv, 2 * wp + 1);
                uint32_t w[RB][4], ws[RB][4];  // words a (rows g, g+8), b (rows g, g+8); and shifted by 10
#pragma unroll
                for (int b = 0; b < RB; ++b) {
                    w[b][0] = word_of(q[jj][b][0], 2 * wp);
                    w[b][1] = word_of(q[jj][b][1], 2 * wp);
                    w[b][2] = word_of(q[jj][b][0], 2 * wp + 1);
                    w[b][3] = word_of(q[jj][b][1], 2 * wp + 1);
#pragma unroll
                    for (int u = 0; u < 4; ++u) ws[b][u] = w[b][u] >> 10;
                }
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint32_t b0 = hmul2_bits(xa, onehot[s]);
                    const uint32_t b1 = hmul2_bits(xb, onehot[s]);
                    const uint32_t one = slot_ones(s, NORM);
                    mma16816(dx[s & 1], one, one, one, one, b0, b1);
                    const uint32_t m = slot_mask(s);
#pragma unroll
                    for (int b = 0; b < RB; ++b) {
                        const uint32_t *src = s < 5 ? w[b] : ws[b];
                        mma16816(d[b][s & 1], slot_operand<NORM>(src[0], m), slot_operand<NORM>(src[1], m),
                                 slot_operand<NORM>(src[2], m), slot_operand<NORM>(src[3], m), b0, b1);
                    }
                }
            }
        }
    }

    // ---- columns -> row sums: scale each slot column, reduce over the quad
    const float sc0 = col_scale<NORM>(2 * t), sc1 = col_scale<NORM>(2 * t + 1);
    float sx = __fadd_rn(__fmul_rn(__fadd_rn(dx[0][0], dx[1][0]), sc0), __fmul_rn(__fadd_rn(dx[0][1], dx[1][1]), sc1));
    sx += __shfl_xor_sync(0xffffffffu, sx, 1);
    sx += __shfl_xor_sync(0xffffffffu, sx, 2);
    float v[RB][2];
#pragma unroll
    for (int b = 0; b < RB; ++b) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float s = __fadd_rn(__fmul_rn(__fadd_rn(d[b][0][2 * h], d[b][1][2 * h]), sc0),
                                __fmul_rn(__fadd_rn(d[b][0][2 * h + 1], d[b][1][2 * h + 1]), sc1));
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            v[b][h] = s;
        }
    }

    const float c0 = a.cb[0], dd = a.cb[1] - a.cb[0];
    if (KW == 1) {
        if (t == 0) {
#pragma unroll
            for (int b = 0; b < RB; ++b)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int64_t row = (rb0 + b) * 16 + g + 8 * h;
                    if (row < a.rows)
                        a.y[row] = h2f(a.scales[row]) * __fadd_rn(__fmul_rn(c0, sx), __fmul_rn(dd, v[b][h]));
                }
        }
        return;
    }
    // ---- combine the KW partial sums in a fixed order
    constexpr int PER = RB * 16 + 1;
    float *mine = red + (kw * RW + rw) * PER;
    if (t == 0) {
#pragma unroll
        for (int b = 0; b < RB; ++b) {
            mine[b * 16 + g] = v[b][0];
            mine[b * 16 + g + 8] = v[b][1];
        }
    }
    if (lane == 0) mine[RB * 16] = sx;
    __syncthreads();
    if (kw == 0) {
        for (int i = lane; i < RB * 16; i += 32) {
            const int64_t row = rb0 * 16 + i;
            float s1 = red[rw * PER + i], sxa = red[rw * PER + RB * 16];
#pragma unroll
            for (int k = 1; k < KW; ++k) {
                s1 += red[(k * RW + rw) * PER + i];
                sxa += red[(k * RW + rw) * PER + RB * 16];
            }
            if (row < a.rows) a.y[row] = h2f(a.scales[row]) * __fadd_rn(__fmul_rn(c0, sxa), __fmul_rn(dd, s1));
        }
    }
}

constexpr int kMaxMmaCols = 32768;

template <int RB, int KW, bool NORM>
cudaError_t launch_mma(const PackedArgs &a, const GemvConfig &cfg, cudaStream_t st) {
    constexpr int SB = RB >= 4 ? 1 : 2;
    auto kern = gemv2_mma_kernel<RB, KW, SB, NORM>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 2 * kMaxMmaCols + 16384);
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int RW = cfg.warps / KW;
    if (RW < 1 || RW * KW != cfg.warps) return cudaErrorInvalidValue;
    const int64_t rowblocks = (a.rows + 15) / 16;
    const int64_t per_cta = (int64_t)RW * RB;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)((rowblocks + per_cta - 1) / per_cta));
    lc.blockDim = dim3(32 * cfg.warps);
    lc.dynamicSmemBytes = (size_t)a.cols * 2 + (size_t)KW * RW * (RB * 16 + 1) * 4;
    lc.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = cfg.pdl ? 1 : 0;
    lc.attrs = attr;
    lc.numAttrs = 1;
    const int prefetch = !cfg.pdl ? 0 : cfg.independent ? 2 : cfg.weights_static ? 1 : 0;
    return cudaLaunchKernelEx(&lc, kern, a, prefetch);
}

template <int RB, bool NORM>
cudaError_t launch_mma_k(const PackedArgs &a, const GemvConfig &cfg, cudaStream_t st) {
    switch (cfg.split) {
        case 1: return launch_mma<RB, 1, NORM>(a, cfg, st);
        case 2: return launch_mma<RB, 2, NORM>(a, cfg, st);
        case 3: return launch_mma<RB, 3, NORM>(a, cfg, st);
        case 4: return launch_mma<RB, 4, NORM>(a, cfg, st);
        case 6: return launch_mma<RB, 6, NORM>(a, cfg, st);
        default: return cudaErrorInvalidValue;
    }
}



}  // namespace

bool gemv_mma_supported(const PackedArgs &a) {
    return a.cols % 256 == 0 && a.cols <= kMaxMmaCols && (reinterpret_cast<uintptr_t>(a.codes) % 16) == 0 &&
           (reinterpret_cast<uintptr_t>(a.x) % 16) == 0;
}

cudaError_t launch_gemv_mma(const PackedArgs &a, const GemvConfig &cfg, cudaStream_t st) {
    if (!gemv_mma_supported(a)) return cudaErrorNotSupported;
    switch (cfg.rows_per_lane) {
        case 1: return launch_mma_k<1, true>(a, cfg, st);
        case 2: return launch_mma_k<2, true>(a, cfg, st);
        case 4: return launch_mma_k<4, true>(a, cfg, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mm
