// gemv_packed2.cu -- y = diag(scale) . W . x for 2-bit packed W (sm_103a).
//
// "Kernel 0112", sections "What is being measured" and "The four variants":
// a 12,288 x 1,536 matrix of 2-bit weights times 1,536 inputs, where the
// run time is the time to stream the 4.5 MiB of weights, and where splitting
// each dot product across more threads (4 -> 16 -> 32 ways) is what made the
// kernel faster.  Here the split width S, the rows carried per lane R and the
// CTA size are template / launch knobs swept the same way.
//
// GB300 design (not the page's):
//  * 16-byte read-only streaming loads of the codes (64 fields per load), all
//    of a lane's loads issued before any arithmetic so the whole 4.5 MiB can be
//    in flight at once across the 152 SMs; S consecutive lanes read one row's
//    consecutive 16-byte chunks, so one warp instruction covers full 128-byte
//    lines of 32/S rows.
//  * x (fp16) is staged once per CTA in shared memory (fp32 for the select
//    decode, fp16 as it is for the affine one) in a layout XOR-swizzled by
//    chunk, so the S lanes of a row group read S different chunks without
//    bank conflicts.
//  * split-K partial sums reduced with __shfl_xor_sync in a fixed order (no
//    atomics): a given variant is bit-reproducible run to run.
//  * the per-row fp16 scale is applied once to the fp32 sum.
//
// Two decode variants:
//  * select: field -> codebook entry by two predicated selects, fp32 FMA.
//    Any codebook.
//  * affine: when codebook[c] == c0 + c*d exactly, sum_k cb[c_k] x_k is
//    evaluated as c0 * sum_k x_k + d * sum_k c_k x_k, the fields used in place
//    as fp16 subnormals against fp16 x with the mixed-precision FMA, one LOP3
//    per two fields (gemv_mixed.cuh; exact products).  Decoding stays exact:
//    one-hot x returns scale_r * cb[field] bit for bit.  sum_k x_k is
//    accumulated by every lane with the same FMAs (every field 1), classes,
//    order and shuffle tree as sum_k c_k x_k, so when every field of a row is
//    the codebook's zero entry c_z in {0, 1, 2}, d * sum c x is exactly
//    -c0 * sum x and the row returns 0.
#include "gemv_mixed.cuh"
#include "mm_common.cuh"
#include "mm_internal.h"

#include <cuda_fp16.h>

#include <mutex>

namespace mm {
namespace {

__device__ __forceinline__ float h2f(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// physical float4 slot of logical float4 index f of the staged x: a chunk of
// 64 fields is 16 float4s; its slots are XOR-permuted by (chunk & 7).
__device__ __forceinline__ int xs_slot(int f) { return f ^ ((f >> 4) & 7); }

// the same for the affine decode's fp16 x: a chunk of 64 fields is 8 slots of 16 bytes
__device__ __forceinline__ int xs16_slot(int g) { return g ^ ((g >> 3) & 7); }

__device__ __forceinline__ float cb_select(uint32_t c, float c0, float c1, float c2, float c3) {
    const float lo = (c & 1u) ? c1 : c0;
    const float hi = (c & 1u) ? c3 : c2;
    return (c & 2u) ? hi : lo;
}

__device__ __forceinline__ float2 select_word(uint32_t w, const float4 &x0, const float4 &x1, const float4 &x2,
                                              const float4 &x3, float2 acc, const PackedArgs &a) {
    const float xv[16] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w,
                          x2.x, x2.y, x2.z, x2.w, x3.x, x3.y, x3.z, x3.w};
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
        const float w0 = cb_select((w >> (2 * i)) & 3u, a.cb[0], a.cb[1], a.cb[2], a.cb[3]);
        const float w1 = cb_select((w >> (2 * i + 2)) & 3u, a.cb[0], a.cb[1], a.cb[2], a.cb[3]);
        acc.x = fmaf(w0, xv[i], acc.x);
        acc.y = fmaf(w1, xv[i + 1], acc.y);
    }
    return acc;
}

constexpr int kDeqSelect = 1;
constexpr int kDeqAffine = 2;

template <int S, int R, int CPL, int DQ>
__global__ void __launch_bounds__(512) gemv2_vec_kernel(const PackedArgs a, const int prefetch) {
    extern __shared__ float4 xs[];  // cols/4 float4, swizzled
    constexpr int GROUPS = 32 / S;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int kp = lane % S, rg = lane / S;
    const int64_t row0 = ((int64_t)blockIdx.x * nwarps + warp) * (GROUPS * R) + rg * R;
    const int nc = (int)(a.cols >> 6);
    const int64_t rowbytes = a.cols >> 2;

    uint4 q[R][CPL];
    auto load_batch = [&](int c0) {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int t = 0; t < CPL; ++t) {
                const int c = c0 + kp + S * t;
                const int64_t row = row0 + r;
                if (row < a.rows && c < nc)
                    q[r][t] = ld_stream_v4(a.codes + row * rowbytes + (int64_t)c * 16);
                else
                    q[r][t] = make_uint4(0u, 0u, 0u, 0u);
            }
    };

    // prefetch: 0 wait for earlier kernels first; 1 codes before the wait;
    // 2 no wait at all (the caller promised no dependence on queued work)
    if (prefetch >= 1) {
        load_batch(0);
        // chained calls: the next call may launch only once this one has passed its wait,
        // so at most one call runs ahead (its weight loads) instead of a queue of parked ones
        if (prefetch == 1) pdl_wait();
        pdl_launch_dependents();
    } else {
        pdl_wait();
        load_batch(0);
        pdl_launch_dependents();
    }

    // ---- stage x: the select decode takes fp32 values, the affine decode the fp16 values as they
    // are; every 16-byte load of a batch is issued before any of them is stored
    const int n8 = (int)(a.cols >> 3);
    constexpr int XU = 4;
    for (int base = threadIdx.x; base < n8; base += XU * blockDim.x) {
        uint4 hv[XU];
#pragma unroll
        for (int u = 0; u < XU; ++u) {
            const int g = base + u * blockDim.x;
            if (g < n8) hv[u] = __ldg(reinterpret_cast<const uint4 *>(a.x) + g);
        }
#pragma unroll
        for (int u = 0; u < XU; ++u) {
            const int g = base + u * blockDim.x;
            if (g < n8) {
                if (DQ == kDeqAffine) {
                    reinterpret_cast<uint4 *>(xs)[xs16_slot(g)] = hv[u];
                } else {
                    const uint32_t hw[4] = {hv[u].x, hv[u].y, hv[u].z, hv[u].w};
                    float v[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[i] = h2f((uint16_t)((hw[i >> 1] >> (16 * (i & 1))) & 0xFFFFu));
                    xs[xs_slot(2 * g)] = make_float4(v[0], v[1], v[2], v[3]);
                    xs[xs_slot(2 * g + 1)] = make_float4(v[4], v[5], v[6], v[7]);
                }
            }
        }
    }
    __syncthreads();

    // ---- multiply
    float2 acc[R];      // select decode
    float accm[R][5];   // affine decode: five classes per row (gemv_mixed.cuh)
    float accx[5];      // affine: this lane's sum of x, same classes and order as accm
#pragma unroll
    for (int r = 0; r < R; ++r) {
        acc[r] = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 5; ++k) accm[r][k] = 0.f;
    }
#pragma unroll
    for (int k = 0; k < 5; ++k) accx[k] = 0.f;
    const uint4 *xs16 = reinterpret_cast<const uint4 *>(xs);

    for (int c0 = 0; c0 < nc; c0 += S * CPL) {
        if (c0 > 0) load_batch(c0);
#pragma unroll
        for (int t = 0; t < CPL; ++t) {
            const int c = c0 + kp + S * t;
            if (c < nc) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (DQ == kDeqAffine) {
                        const uint4 xa = xs16[xs16_slot(8 * c + 2 * u)], xb = xs16[xs16_slot(8 * c + 2 * u + 1)];
                        const uint32_t X[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
                        word_mixed(0x55555555u, X, accx);
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            const uint32_t w = u == 0 ? q[r][t].x : u == 1 ? q[r][t].y : u == 2 ? q[r][t].z : q[r][t].w;
                            word_mixed(w, X, accm[r]);
                        }
                    } else {
                        const int f = 16 * c + 4 * u;
                        const float4 x0 = xs[xs_slot(f + 0)];
                        const float4 x1 = xs[xs_slot(f + 1)];
                        const float4 x2 = xs[xs_slot(f + 2)];
                        const float4 x3 = xs[xs_slot(f + 3)];
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            const uint32_t w = u == 0 ? q[r][t].x : u == 1 ? q[r][t].y : u == 2 ? q[r][t].z : q[r][t].w;
                            acc[r] = select_word(w, x0, x1, x2, x3, acc[r], a);
                        }
                    }
                }
            }
        }
    }

    // ---- reduce across the S lanes of a row, scale, store
    float s[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        s[r] = DQ == kDeqAffine ? mixed_total(accm[r]) : acc[r].x + acc[r].y;
#pragma unroll
        for (int off = S / 2; off > 0; off >>= 1) s[r] += __shfl_xor_sync(0xffffffffu, s[r], off);
    }
    float sx = 0.f;
    if (DQ == kDeqAffine) {
        sx = mixed_total(accx);
#pragma unroll
        for (int off = S / 2; off > 0; off >>= 1) sx += __shfl_xor_sync(0xffffffffu, sx, off);
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t row = row0 + r;
        if (kp == r && row < a.rows) {
            const float scale = h2f(a.scales[row]);
            float v;
            if (DQ == kDeqAffine) {
                // no contraction into an fma: a row of zero-entry fields gives exactly 0
                const float c0 = a.cb[0], d = a.cb[1] - a.cb[0];
                v = __fadd_rn(__fmul_rn(c0, sx), __fmul_rn(d, s[r]));
            } else {
                v = s[r];
            }
            a.y[row] = scale * v;
        }
    }
}

// Any cols, any alignment: one warp per row, lanes stride over the row's bytes.
__global__ void __launch_bounds__(256) gemv2_bytewise_kernel(const PackedArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    pdl_wait();
    if (row >= a.rows) return;
    const int64_t rowbytes = (a.cols + 3) >> 2;
    const uint8_t *rp = a.codes + row * rowbytes;
    float acc = 0.f;
    for (int64_t b = lane; b < rowbytes; b += 32) {
        const uint32_t byte = rp[b];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t k = 4 * b + i;
            if (k < a.cols)
                acc = fmaf(cb_select((byte >> (2 * i)) & 3u, a.cb[0], a.cb[1], a.cb[2], a.cb[3]), h2f(a.x[k]), acc);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) a.y[row] = h2f(a.scales[row]) * acc;
}

constexpr int kMaxStagedCols = 32768;  // x staged as fp32: 128 KiB of shared memory

template <int S, int R, int DQ>
cudaError_t launch_vec(const PackedArgs &a, const GemvConfig &cfg, cudaStream_t st) {
    constexpr int CPL = S == 4 ? 6 : S == 8 ? 3 : 2;
    auto kern = gemv2_vec_kernel<S, R, CPL, DQ>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxStagedCols * 4);
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int warps = cfg.warps;
    const int64_t rows_per_cta = (int64_t)warps * (32 / S) * R;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)((a.rows + rows_per_cta - 1) / rows_per_cta));
    lc.blockDim = dim3(32 * warps);
    lc.dynamicSmemBytes = (size_t)a.cols * 4;
    lc.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = cfg.pdl ? 1 : 0;
    lc.attrs = attr;
    lc.numAttrs = 1;
    const int prefetch = !cfg.pdl ? 0 : cfg.independent ? 2 : cfg.weights_static ? 1 : 0;
    return cudaLaunchKernelEx(&lc, kern, a, prefetch);
}

template <int S, int DQ>
cudaError_t launch_vec_r(const PackedArgs &a, const GemvConfig &cfg, cudaStream_t st) {
    switch (cfg.rows_per_lane) {
        case 1: return launch_vec<S, 1, DQ>(a, cfg, st);
        case 2: return launch_vec<S, 2, DQ>(a, cfg, st);
        case 4: return launch_vec<S, 4, DQ>(a, cfg, st);
        default: return cudaErrorInvalidValue;
    }
}

template <int DQ>
cudaError_t launch_vec_s(const PackedArgs &a, const GemvConfig &cfg, cudaStream_t st) {
    switch (cfg.split) {
        case 4: return launch_vec_r<4, DQ>(a, cfg, st);
        case 8: return launch_vec_r<8, DQ>(a, cfg, st);
        case 16: return launch_vec_r<16, DQ>(a, cfg, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool codebook_is_affine(const float cb[4]) {
    const float d = cb[1] - cb[0];
    // each entry must be reproduced exactly by c0 + c*d in fp32
    for (int c = 0; c < 4; ++c) {
        volatile float v = cb[0] + (float)c * d;
        if (v != cb[c]) return false;
    }
    // a zero entry at field 3 would not cancel exactly against c0 * sum x
    if (cb[3] == 0.0f && d != 0.0f) return false;
    return true;
}

bool gemv_vec_supported(const PackedArgs &a) {
    return a.cols % 64 == 0 && a.cols <= kMaxStagedCols && (reinterpret_cast<uintptr_t>(a.codes) % 16) == 0 &&
           (reinterpret_cast<uintptr_t>(a.x) % 16) == 0;
}

cudaError_t launch_gemv_packed2(const PackedArgs &a, const GemvConfig &cfg, cudaStream_t st) {
    if (cfg.dequant == 6) return launch_gemv_mxf4(a, cfg, st);
    if (cfg.dequant == 5) return launch_gemv_tc(a, cfg, st);
    if (cfg.dequant == kDeqAffine && cfg.staging) return launch_gemv_rows(a, cfg, st);
    if (cfg.dequant == 4) return launch_gemv_fp8(a, cfg, st);
    if (cfg.dequant == 3) return cfg.staging ? launch_gemv_tma(a, cfg, st) : launch_gemv_mma(a, cfg, st);
    if (!gemv_vec_supported(a)) {
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3((unsigned)((a.rows + 7) / 8));
        lc.blockDim = dim3(256);
        lc.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = cfg.pdl ? 1 : 0;
        lc.attrs = attr;
        lc.numAttrs = 1;
        return cudaLaunchKernelEx(&lc, gemv2_bytewise_kernel, a);
    }
    if (cfg.dequant == kDeqAffine) return launch_vec_s<kDeqAffine>(a, cfg, st);
    return launch_vec_s<kDeqSelect>(a, cfg, st);
}

}  // namespace mm
